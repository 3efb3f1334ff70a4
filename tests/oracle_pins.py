"""Pins of the float64 oracle against facts that do not come from the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError when the oracle disagrees with:

* torch's float64 CPU ``scaled_dot_product_attention`` (a library routine
  with the same definition: in the FFPA API reference, the signature of
  ``ffpa_attn_func`` follows torch's scaled_dot_product_attention),
* closed forms (softmax of known logits, Q = 0 gives a plain mean and
  LSE = ln(#visible keys), Nkv = 1 gives V_0 and LSE = scale*q.k_0),
* invariants of the definition (rows of softmax sum to one, GQA equals
  repeated-KV MHA, tail-aligned causal visibility, varlen equals
  per-sequence dense, shift and permutation invariances).

They live in a plain module so that ``test_oracle_pins.py`` runs them on the
real oracle and ``test_oracle_mutants.py`` runs them on copies of the oracle
with planted mistakes (each mutant must fail at least one pin).
"""
from __future__ import annotations

import math
import zlib

import torch
import torch.nn.functional as F

from exact_headdim_attention_gb300 import workloads as wl

ATOL = 1e-10


def _close(a, b, atol=ATOL, what=""):
    a = torch.as_tensor(a, dtype=torch.float64)
    b = torch.as_tensor(b, dtype=torch.float64)
    assert a.shape == b.shape, f"{what}: shape {tuple(a.shape)} vs {tuple(b.shape)}"
    fin = torch.isfinite(b)
    assert torch.equal(torch.isfinite(a), fin), f"{what}: finiteness differs"
    assert torch.equal(a[~fin], b[~fin]), f"{what}: infinities differ"
    err = (a[fin] - b[fin]).abs().max().item() if fin.any() else 0.0
    assert err <= atol, f"{what}: max |err| {err:.3e} > {atol:.1e}"


def tail_causal_keep(Nq, Nkv):
    """Tail-aligned causal visibility: row r keeps k <= r + (Nkv - Nq)."""
    return torch.ones(Nq, Nkv, dtype=torch.bool).tril(diagonal=Nkv - Nq)


def _sdpa_reference(q, k, v, mask, scale, causal):
    """torch float64 SDPA with the causal rule expressed as an explicit mask."""
    B, Hq, Nq, D = q.shape
    Nkv = k.shape[2]
    qd, kd, vd = q.double(), k.double(), v.double()
    m = None
    if mask is not None:
        m = mask.double() if mask.dtype != torch.bool else mask
    if causal:
        keep = tail_causal_keep(Nq, Nkv)
        if m is None:
            m = keep
        elif m.dtype == torch.bool:
            m = m & keep
        else:
            m = m.masked_fill(~keep, -math.inf)
    gqa = Hq != k.shape[1]
    o = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=m, scale=scale, enable_gqa=gqa)
    # LSE through library routines: matmul + logsumexp
    kr = kd.repeat_interleave(Hq // k.shape[1], dim=1)
    sc = (scale if scale is not None else 1 / math.sqrt(D)) * (qd @ kr.transpose(-1, -2))
    if m is not None:
        sc = sc.masked_fill(~m, -math.inf) if m.dtype == torch.bool else sc + m
    lse = torch.logsumexp(sc, dim=-1)
    return o, lse


def _bool_mask(g, shape, Nq, Nkv):
    m = torch.rand(*shape, generator=g) < 0.7
    m = m.expand(*shape[:-2], Nq, Nkv).clone() if shape[-2] == 1 else m
    # keep the tail diagonal so that no row is fully masked (causal or not)
    idx = torch.arange(Nq)
    m[..., idx, idx + (Nkv - Nq)] = True
    return m


SDPA_CASES = [
    # name, B, Hq, Hkv, Nq, Nkv, D, causal, mask, dtype, scale
    ("mha", 2, 2, 2, 5, 7, 64, False, None, torch.bfloat16, None),
    ("gqa", 1, 4, 2, 6, 6, 32, False, None, torch.bfloat16, None),
    ("mqa_causal_cross", 2, 3, 1, 3, 9, 16, True, None, torch.bfloat16, None),
    ("causal_self", 1, 2, 2, 8, 8, 16, True, None, torch.bfloat16, 0.3),
    ("bool_b1nk", 2, 2, 2, 4, 6, 16, False, ("bool", (2, 1, 4, 6)), torch.bfloat16, None),
    ("bool_nk_causal", 1, 4, 2, 5, 7, 16, True, ("bool", (5, 7)), torch.bfloat16, None),
    ("bool_h_bcast_q", 2, 2, 2, 3, 5, 16, False, ("bool", (1, 2, 1, 5)), torch.bfloat16, None),
    ("add_f32", 2, 2, 1, 4, 6, 16, False, ("f32", (2, 1, 4, 6)), torch.bfloat16, 0.7),
    ("add_qtype_causal", 1, 2, 2, 4, 6, 16, True, ("qtype", (1, 2, 4, 6)), torch.bfloat16, None),
    ("fp16", 1, 2, 2, 5, 5, 32, False, None, torch.float16, None),
    ("fp16_add_f32", 1, 2, 1, 3, 4, 16, True, ("f32", (3, 4)), torch.float16, 0.5),
    # additive masks in the input dtype holding -inf (FFPA API reference, `attn_mask`: a
    # floating mask is added to the scores; -inf removes the key)
    ("fp16_add_qtype_neg_inf", 2, 2, 2, 5, 7, 16, False, ("qtype_inf", (2, 1, 5, 7)), torch.float16, None),
    ("fp16_add_qtype_neg_inf_causal", 1, 4, 2, 4, 9, 32, True, ("qtype_inf", (1, 4, 4, 9)), torch.float16, 0.4),
    ("bf16_add_qtype_neg_inf", 1, 2, 1, 6, 6, 16, False, ("qtype_inf", (6, 6)), torch.bfloat16, None),
]


def _inf_mask(g, shape, Nq, Nkv, dtype):
    """Additive mask in `dtype`: N(0,1) with ~30 % of the entries -inf; the
    tail diagonal stays finite so that no row loses every key."""
    m = torch.randn(*shape, generator=g)
    m = m.masked_fill(torch.rand(*shape, generator=g) < 0.3, -math.inf)
    m = m.expand(*shape[:-2], Nq, Nkv).clone() if shape[-2] == 1 else m
    idx = torch.arange(Nq)
    m[..., idx, idx + (Nkv - Nq)] = 0.5
    return m.to(dtype)


def pin_sdpa_cases(orc, cases=SDPA_CASES):
    for (name, B, Hq, Hkv, Nq, Nkv, D, causal, mspec, dtype, scale) in cases:
        q, k, v, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed=zlib.crc32(name.encode()) % 100003, dtype=dtype)
        mask = None
        if mspec is not None:
            kind, shape = mspec
            if kind == "bool":
                mask = _bool_mask(g, shape, Nq, Nkv)
            elif kind == "f32":
                mask = torch.randn(*shape, generator=g)
            elif kind == "qtype_inf":
                mask = _inf_mask(g, shape, Nq, Nkv, dtype)
            else:
                mask = torch.randn(*shape, generator=g).to(dtype)
        o, lse = orc.attn_dense(q, k, v, attn_mask=mask, scale=scale, is_causal=causal)
        o_ref, lse_ref = _sdpa_reference(q, k, v, mask, scale, causal)
        _close(o, o_ref, what=f"{name}: O")
        _close(lse, lse_ref, what=f"{name}: LSE")


def pin_strided_inputs(orc):
    """Non-contiguous [B,N,H,D] views give the same result as contiguous copies."""
    g = torch.Generator().manual_seed(7)
    q = torch.randn(2, 6, 4, 32, generator=g).bfloat16().transpose(1, 2)   # [B,H,N,D] view
    k = torch.randn(2, 9, 2, 32, generator=g).bfloat16().transpose(1, 2)
    v = torch.randn(2, 9, 2, 32, generator=g).bfloat16().transpose(1, 2)
    o, lse = orc.attn_dense(q, k, v, is_causal=True)
    o_ref, lse_ref = _sdpa_reference(q.contiguous(), k.contiguous(), v.contiguous(), None, None, True)
    _close(o, o_ref, what="strided O")
    _close(lse, lse_ref, what="strided LSE")


def pin_closed_form_softmax(orc):
    """Logits (0, 1, 2) on one-hot values: O = softmax(0,1,2), LSE = ln(1+e+e^2)."""
    D = 64
    q = torch.zeros(1, 1, 1, D)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, 3, D)
    k[0, 0, :, 0] = torch.tensor([0.0, 1.0, 2.0])
    v = torch.zeros(1, 1, 3, D)
    for j in range(3):
        v[0, 0, j, j] = 1.0
    o, lse = orc.attn_dense(q.bfloat16(), k.bfloat16(), v.bfloat16(), scale=1.0)
    z = 1 + math.e + math.e ** 2
    want = torch.zeros(D, dtype=torch.float64)
    want[:3] = torch.tensor([1 / z, math.e / z, math.e ** 2 / z], dtype=torch.float64)
    _close(o[0, 0, 0], want, atol=1e-14, what="softmax(0,1,2)")
    _close(lse[0, 0, 0], torch.tensor(math.log(z), dtype=torch.float64), atol=1e-14, what="ln(1+e+e^2)")


def pin_zero_query(orc):
    """Q = 0: every visible key has weight 1, O is their mean and LSE = ln(count).

    With tail-aligned causal masking row r sees r + (Nkv - Nq) + 1 keys."""
    B, Hq, Hkv, Nq, Nkv, D = 1, 2, 1, 5, 8, 16
    _, k, v, _ = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed=11)
    q = torch.zeros(B, Hq, Nq, D, dtype=torch.bfloat16)
    for causal in (False, True):
        o, lse = orc.attn_dense(q, k, v, is_causal=causal)
        for r in range(Nq):
            n = r + (Nkv - Nq) + 1 if causal else Nkv
            want = v[0, 0, :n].double().mean(dim=0)
            for h in range(Hq):
                _close(o[0, h, r], want, atol=1e-14, what=f"Q=0 mean r={r}")
                _close(lse[0, h, r], torch.tensor(math.log(n), dtype=torch.float64), atol=1e-14,
                       what=f"Q=0 LSE r={r}")


def pin_single_key(orc):
    """Nkv = 1: O equals V_0 exactly and LSE equals scale * q.k_0."""
    q, k, v, _ = wl.draw_dense(2, 2, 2, 4, 1, 64, seed=12)
    o, lse = orc.attn_dense(q, k, v, scale=0.25)
    _close(o, v.double().expand(2, 2, 4, 64), atol=0.0, what="Nkv=1 O")
    want = 0.25 * torch.einsum("bhnd,bhd->bhn", q.double(), k[:, :, 0].double())
    _close(lse, want, atol=1e-12, what="Nkv=1 LSE")


def _same_values(a, b, what):
    """Element-wise identity of two float64 tensors, NaN matching NaN."""
    a = torch.as_tensor(a, dtype=torch.float64).reshape(-1)
    b = torch.as_tensor(b, dtype=torch.float64).reshape(-1)
    nan_a, nan_b = torch.isnan(a), torch.isnan(b)
    assert torch.equal(nan_a, nan_b), f"{what}: NaN positions differ ({int((nan_a != nan_b).sum())})"
    bad = (a[~nan_a] != b[~nan_b]).nonzero()
    assert bad.numel() == 0, f"{what}: {bad.numel()} values differ, first at {int(bad[0])}"


def pin_every_16bit_pattern(orc):
    """Nkv = 1 passes V through unchanged (weight exp(0) / 1), so every one of
    the 65 536 bit patterns of fp16 and of bf16 placed in V must come back as
    torch's own widening of that pattern: normals, both zeros, every
    subnormal, +-inf and NaN (IEEE binary16 and the top half of binary32)."""
    pat = torch.arange(65536, dtype=torch.int32).to(torch.int16).reshape(1, 1024, 1, 64)
    g = torch.Generator().manual_seed(16)
    for dtype in (torch.float16, torch.bfloat16):
        v = pat.view(dtype)
        q = torch.randn(1, 1024, 1, 64, generator=g).to(dtype)
        k = torch.randn(1, 1024, 1, 64, generator=g).to(dtype)
        o, _ = orc.attn_dense(q, k, v)
        _same_values(o, v.double(), f"{dtype} patterns")


def pin_rows_sum_to_one(orc):
    """V = 1 everywhere: each output element is sum_k softmax_k = 1."""
    B, Hq, Hkv, Nq, Nkv, D = 2, 4, 2, 6, 9, 32
    q, k, _, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed=13)
    v = torch.ones(B, Hkv, Nkv, D, dtype=torch.bfloat16)
    mask = torch.randn(B, 1, Nq, Nkv, generator=g)
    for causal in (False, True):
        o, _ = orc.attn_dense(q, k, v, attn_mask=mask, is_causal=causal)
        _close(o, torch.ones_like(o), atol=1e-13, what="rows sum to 1")


def pin_identical_values(orc):
    """All V rows equal to u: O = u for any logits."""
    q, k, _, g = wl.draw_dense(1, 2, 2, 5, 7, 32, seed=14)
    u = torch.randn(32, generator=g).bfloat16()
    v = u.expand(1, 2, 7, 32).contiguous()
    o, _ = orc.attn_dense(q, k, v, is_causal=True)
    _close(o, u.double().expand_as(o), atol=1e-13, what="identical V rows")


def pin_one_hot_logit(orc):
    """One key with a logit 60 above the rest selects its V row (to e^-60)."""
    D, Nkv, star = 64, 6, 3
    q = torch.zeros(1, 1, 1, D)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, Nkv, D)
    k[0, 0, star, 0] = 60.0
    g = torch.Generator().manual_seed(15)
    v = torch.randn(1, 1, Nkv, D, generator=g).bfloat16()
    o, lse = orc.attn_dense(q.bfloat16(), k.bfloat16(), v, scale=1.0)
    _close(o[0, 0, 0], v[0, 0, star].double(), atol=1e-20 + 1e-24, what="one-hot logit")
    _close(lse[0, 0, 0], torch.tensor(60.0 + math.log1p((Nkv - 1) * math.exp(-60.0)),
                                      dtype=torch.float64), atol=1e-14, what="one-hot LSE")


def pin_causal_visibility(orc):
    """Changing V at key t changes exactly the rows r with t <= r + (Nkv - Nq)."""
    B, H, Nq, Nkv, D = 1, 1, 6, 10, 16
    q, k, v, g = wl.draw_dense(B, H, H, Nq, Nkv, D, seed=16)
    o0, _ = orc.attn_dense(q, k, v, is_causal=True)
    for t in (Nkv - Nq, Nkv - Nq + 2, Nkv - 1):
        v2 = v.clone()
        v2[0, 0, t] = torch.randn(D, generator=g).bfloat16() * 4
        o1, _ = orc.attn_dense(q, k, v2, is_causal=True)
        for r in range(Nq):
            same = torch.equal(o0[0, 0, r], o1[0, 0, r])
            assert same == (t > r + (Nkv - Nq)), f"causal visibility broken at r={r}, t={t}"


def pin_gqa_is_repeated_mha(orc):
    """GQA equals MHA with K/V heads repeated group-wise (head hq reads hq // g)."""
    B, Hq, Hkv, Nq, Nkv, D = 2, 6, 2, 5, 7, 32
    q, k, v, _ = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed=17)
    o, lse = orc.attn_dense(q, k, v, is_causal=True)
    kr = k.repeat_interleave(Hq // Hkv, dim=1).contiguous()
    vr = v.repeat_interleave(Hq // Hkv, dim=1).contiguous()
    o2, lse2 = orc.attn_dense(q, kr, vr, is_causal=True)
    _close(o, o2, atol=0.0, what="GQA vs repeated MHA O")
    _close(lse, lse2, atol=0.0, what="GQA vs repeated MHA LSE")


def pin_shift_invariance(orc):
    """A constant additive mask c leaves O unchanged and adds c to LSE."""
    q, k, v, _ = wl.draw_dense(1, 2, 2, 4, 6, 32, seed=18)
    c = 1.75
    o0, l0 = orc.attn_dense(q, k, v, is_causal=True)
    o1, l1 = orc.attn_dense(q, k, v, attn_mask=torch.full((4, 6), c), is_causal=True)
    _close(o1, o0, atol=1e-13, what="shift O")
    _close(l1, l0 + c, atol=1e-13, what="shift LSE")


def pin_all_true_mask(orc):
    q, k, v, _ = wl.draw_dense(2, 2, 2, 4, 6, 32, seed=19)
    o0, l0 = orc.attn_dense(q, k, v)
    o1, l1 = orc.attn_dense(q, k, v, attn_mask=torch.ones(2, 1, 4, 6, dtype=torch.bool))
    _close(o1, o0, atol=0.0, what="all-true mask O")
    _close(l1, l0, atol=0.0, what="all-true mask LSE")


def pin_kv_permutation(orc):
    """Non-causal attention is invariant to permuting the key/value rows together."""
    q, k, v, g = wl.draw_dense(1, 2, 2, 4, 9, 32, seed=20)
    perm = torch.randperm(9, generator=g)
    o0, l0 = orc.attn_dense(q, k, v)
    o1, l1 = orc.attn_dense(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous())
    _close(o1, o0, atol=1e-13, what="KV permutation O")
    _close(l1, l0, atol=1e-13, what="KV permutation LSE")


def pin_scale_fold(orc):
    """Scaling Q by 2 (exact in bf16) with scale/2 leaves O and LSE unchanged."""
    q, k, v, _ = wl.draw_dense(1, 2, 2, 5, 6, 32, seed=21)
    o0, l0 = orc.attn_dense(q, k, v, scale=0.3)
    o1, l1 = orc.attn_dense(q * 2, k, v, scale=0.15)
    _close(o1, o0, atol=1e-13, what="scale fold O")
    _close(l1, l0, atol=1e-13, what="scale fold LSE")


def pin_fully_masked_row(orc):
    """A row with every key masked has O = 0 and LSE = -inf (adopted convention)."""
    q, k, v, _ = wl.draw_dense(1, 1, 1, 3, 4, 16, seed=22)
    mask = torch.ones(3, 4, dtype=torch.bool)
    mask[1] = False
    o, lse = orc.attn_dense(q, k, v, attn_mask=mask)
    assert torch.equal(o[0, 0, 1], torch.zeros(16, dtype=torch.float64))
    assert lse[0, 0, 1].item() == -math.inf
    assert torch.isfinite(lse[0, 0, [0, 2]]).all()


def pin_varlen_is_per_sequence_dense(orc):
    """Packed varlen equals the dense definition applied to each sequence,
    with lower-right causal alignment per sequence; also torch SDPA per sequence."""
    lq, lk = [3, 7, 1, 5], [5, 7, 4, 2]
    Hq, Hkv, D = 4, 2, 32
    q, k, v, cq, ck = wl.draw_varlen(lq, lk, Hq, Hkv, D, seed=23)
    for causal in (False, True):
        o, lse = orc.attn_varlen(q, k, v, cq, ck, causal=causal)
        for s in range(len(lq)):
            qs = q[cq[s]:cq[s + 1]].transpose(0, 1).unsqueeze(0).contiguous()
            ks = k[ck[s]:ck[s + 1]].transpose(0, 1).unsqueeze(0).contiguous()
            vs = v[ck[s]:ck[s + 1]].transpose(0, 1).unsqueeze(0).contiguous()
            od, ld = orc.attn_dense(qs, ks, vs, is_causal=causal)
            _close(o[cq[s]:cq[s + 1]], od[0].transpose(0, 1), atol=0.0, what=f"varlen seq {s} O")
            _close(lse[:, cq[s]:cq[s + 1]], ld[0], atol=0.0, what=f"varlen seq {s} LSE")
            if causal and lk[s] < lq[s]:
                continue   # rows with no visible key: SDPA gives NaN there
            o_ref, l_ref = _sdpa_reference(qs, ks, vs, None, None, causal)
            _close(od, o_ref, what=f"varlen seq {s} vs SDPA O")
            _close(ld, l_ref, what=f"varlen seq {s} vs SDPA LSE")
    # causal with a sequence shorter in keys than queries: early rows see nothing
    o, lse = orc.attn_varlen(q, k, v, cq, ck, causal=True)
    s = 3   # lq=5, lk=2: rows 0..2 see no key
    rows = slice(int(cq[s]), int(cq[s]) + 3)
    assert torch.equal(o[rows], torch.zeros_like(o[rows]))
    assert bool((lse[:, rows] == -math.inf).all())


def pin_varlen_default_cu_k(orc):
    """cu_seqlens_k = None means cu_seqlens_q (self-attention)."""
    lq = [4, 6]
    q, k, v, cq, _ = wl.draw_varlen(lq, lq, 2, 2, 16, seed=24)
    o0, l0 = orc.attn_varlen(q, k, v, cq, None, causal=True)
    o1, l1 = orc.attn_varlen(q, k, v, cq, cq, causal=True)
    _close(o0, o1, atol=0.0, what="cu_k default")
    _close(l0, l1, atol=0.0, what="cu_k default LSE")


def pin_sampled_rows(orc):
    """The row-sampling entry returns exactly the rows of the full computation."""
    q, k, v, g = wl.draw_dense(2, 4, 2, 7, 9, 32, seed=25)
    mask = torch.randn(2, 1, 7, 9, generator=g)
    o, lse = orc.attn_dense(q, k, v, attn_mask=mask, is_causal=True)
    rows = torch.tensor([0, 5, 13, 27, 55])
    o_r, l_r = orc.attn_dense(q, k, v, attn_mask=mask, is_causal=True, rows=rows)
    _close(o_r, o.reshape(-1, 32)[rows], atol=0.0, what="sampled rows O")
    _close(l_r, lse.reshape(-1)[rows], atol=0.0, what="sampled rows LSE")


# ------------------------------------------------------------------ backward
def _case_mask(g, mspec, Nq, Nkv, dtype):
    if mspec is None:
        return None
    kind, shape = mspec
    if kind == "bool":
        return _bool_mask(g, shape, Nq, Nkv)
    if kind == "f32":
        return torch.randn(*shape, generator=g)
    return torch.randn(*shape, generator=g).to(dtype)


def _sdpa_grads(q, k, v, dout, mask, scale, causal):
    """torch float64 autograd through SDPA (the causal rule as an explicit mask)."""
    Nq, Nkv = q.shape[2], k.shape[2]
    qd, kd, vd = (t.double().requires_grad_() for t in (q, k, v))
    m = None
    if mask is not None:
        m = mask.double() if mask.dtype != torch.bool else mask
    if causal:
        keep = tail_causal_keep(Nq, Nkv)
        if m is None:
            m = keep
        elif m.dtype == torch.bool:
            m = m & keep
        else:
            m = m.masked_fill(~keep, -math.inf)
    o = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=m, scale=scale,
                                       enable_gqa=q.shape[1] != k.shape[1])
    return torch.autograd.grad(o, (qd, kd, vd), dout.double())


def pin_bwd_sdpa_autograd(orc, cases=SDPA_CASES):
    """dQ, dK, dV equal torch's float64 autograd of SDPA on every forward case."""
    for (name, B, Hq, Hkv, Nq, Nkv, D, causal, mspec, dtype, scale) in cases:
        q, k, v, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed=zlib.crc32(name.encode()) % 100003,
                                   dtype=dtype)
        mask = _case_mask(g, mspec, Nq, Nkv, dtype)
        dout = torch.randn(B, Hq, Nq, D, generator=g).to(dtype)
        got = orc.attn_bwd_dense(q, k, v, dout, attn_mask=mask, scale=scale, is_causal=causal)
        ref = _sdpa_grads(q, k, v, dout, mask, scale, causal)
        for nm, a, b in zip(("dQ", "dK", "dV"), got, ref):
            _close(a, b, what=f"{name}: {nm}")


def pin_bwd_finite_differences(orc):
    """Central differences of sum(O * dO), O from an explicit float64 softmax
    formula (no autograd), at every entry of small Q, K and V."""
    g = torch.Generator().manual_seed(11)
    B, Hq, Hkv, Nq, Nkv, D = 1, 2, 1, 3, 5, 8
    q = torch.randn(B, Hq, Nq, D, generator=g).bfloat16()
    k = torch.randn(B, Hkv, Nkv, D, generator=g).bfloat16()
    v = torch.randn(B, Hkv, Nkv, D, generator=g).bfloat16()
    dout = torch.randn(B, Hq, Nq, D, generator=g).bfloat16()
    bias = torch.randn(Nq, Nkv, generator=g)
    scale = 0.45
    keep = tail_causal_keep(Nq, Nkv)

    def loss(qd, kd, vd):
        kr = kd.repeat_interleave(Hq // Hkv, dim=1)
        vr = vd.repeat_interleave(Hq // Hkv, dim=1)
        s = scale * (qd @ kr.transpose(-1, -2)) + bias.double()
        s = s.masked_fill(~keep, -math.inf)
        w = torch.exp(s - s.amax(-1, keepdim=True))
        o = (w / w.sum(-1, keepdim=True)) @ vr
        return (o * dout.double()).sum().item()

    dq, dk, dv = orc.attn_bwd_dense(q, k, v, dout, attn_mask=bias, scale=scale, is_causal=True)
    base = [q.double(), k.double(), v.double()]
    h = 1e-5
    for which, grad in enumerate((dq, dk, dv)):
        t = base[which]
        for idx in range(t.numel()):
            plus = [x.clone() for x in base]
            minus = [x.clone() for x in base]
            plus[which].view(-1)[idx] += h
            minus[which].view(-1)[idx] -= h
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            got = grad.reshape(-1)[idx].item()
            assert abs(fd - got) <= 1e-7, f"{'QKV'[which]}[{idx}]: {got} vs central difference {fd}"


def pin_bwd_invariants(orc):
    """Shifting every key by one vector leaves each row's softmax unchanged, so
    sum_j dK_j = 0 per key/value head; rows of P sum to one, so sum_j dV_j =
    sum of dO over the group's rows; constant V gives constant O, so dQ = dK = 0."""
    g = torch.Generator().manual_seed(5)
    B, Hq, Hkv, Nq, Nkv, D = 2, 4, 2, 7, 11, 16
    q = torch.randn(B, Hq, Nq, D, generator=g).bfloat16()
    k = torch.randn(B, Hkv, Nkv, D, generator=g).bfloat16()
    v = torch.randn(B, Hkv, Nkv, D, generator=g).bfloat16()
    dout = torch.randn(B, Hq, Nq, D, generator=g).bfloat16()
    for causal in (False, True):
        dq, dk, dv = orc.attn_bwd_dense(q, k, v, dout, is_causal=causal)
        _close(dk.sum(2), torch.zeros(B, Hkv, D), atol=1e-12, what=f"sum dK (causal={causal})")
        want = dout.double().view(B, Hkv, Hq // Hkv, Nq, D).sum((2, 3))
        _close(dv.sum(2), want, atol=1e-12, what=f"sum dV (causal={causal})")
    vc = torch.randn(B, Hkv, 1, D, generator=g).bfloat16().expand(B, Hkv, Nkv, D).contiguous()
    dq, dk, _ = orc.attn_bwd_dense(q, k, vc, dout, is_causal=True)
    _close(dq, torch.zeros_like(dq), atol=1e-12, what="dQ for constant V")
    _close(dk, torch.zeros_like(dk), atol=1e-12, what="dK for constant V")


def pin_bwd_sampled_rows(orc):
    """The sampled-row routine equals torch's float64 autograd on the rows it returns."""
    g = torch.Generator().manual_seed(9)
    B, Hq, Hkv, Nq, Nkv, D = 2, 4, 2, 6, 9, 16
    q = torch.randn(B, Hq, Nq, D, generator=g).bfloat16()
    k = torch.randn(B, Hkv, Nkv, D, generator=g).bfloat16()
    v = torch.randn(B, Hkv, Nkv, D, generator=g).bfloat16()
    dout = torch.randn(B, Hq, Nq, D, generator=g).bfloat16()
    qr = [0, 5, 13, B * Hq * Nq - 1]
    kr = [0, 4, 10, 17, B * Hkv * Nkv - 1]
    for causal in (False, True):
        dq, dk, dv = orc.attn_bwd_rows(q, k, v, dout, qr, kr, is_causal=causal)
        gq, gk, gv = _sdpa_grads(q, k, v, dout, None, None, causal)
        _close(dq, gq.reshape(-1, D)[qr], what=f"sampled dQ (causal={causal})")
        _close(dk, gk.reshape(-1, D)[kr], what=f"sampled dK (causal={causal})")
        _close(dv, gv.reshape(-1, D)[kr], what=f"sampled dV (causal={causal})")


def pin_bwd_varlen_equals_per_sequence(orc):
    """Packed varlen gradients equal each sequence's dense gradients (library
    autograd through SDPA on the unpacked sequence), causal and not, with GQA,
    an empty query sequence and unequal query/key lengths."""
    g = torch.Generator().manual_seed(13)
    Hq, Hkv, D = 4, 2, 16
    lq, lk = [5, 0, 9, 3], [7, 4, 9, 6]
    cu_q = torch.tensor([0] + list(torch.tensor(lq).cumsum(0)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(torch.tensor(lk).cumsum(0)), dtype=torch.int32)
    q = torch.randn(sum(lq), Hq, D, generator=g).bfloat16()
    k = torch.randn(sum(lk), Hkv, D, generator=g).bfloat16()
    v = torch.randn(sum(lk), Hkv, D, generator=g).bfloat16()
    dout = torch.randn(sum(lq), Hq, D, generator=g).bfloat16()
    for causal in (False, True):
        dq, dk, dv = orc.attn_bwd_varlen(q, k, v, dout, cu_q, cu_k, causal=causal)
        for s_ in range(len(lq)):
            a, b = int(cu_q[s_]), int(cu_q[s_ + 1])
            c, d = int(cu_k[s_]), int(cu_k[s_ + 1])
            if b - a == 0:
                _close(dk[c:d], torch.zeros(d - c, Hkv, D), what=f"seq {s_} dK (no queries)")
                continue
            if causal and d - c < b - a:
                continue
            gq, gk, gv = _sdpa_grads(q[a:b].transpose(0, 1)[None], k[c:d].transpose(0, 1)[None],
                                     v[c:d].transpose(0, 1)[None], dout[a:b].transpose(0, 1)[None],
                                     None, None, causal)
            _close(dq[a:b], gq[0].transpose(0, 1), what=f"seq {s_} dQ causal={causal}")
            _close(dk[c:d], gk[0].transpose(0, 1), what=f"seq {s_} dK causal={causal}")
            _close(dv[c:d], gv[0].transpose(0, 1), what=f"seq {s_} dV causal={causal}")




# ---------------------------------------------------------------- FP8 reference
# The FP8 forward's reference quantises Q, K and V per (batch, head, block of
# 128 rows) to e4m3 and attends exactly to the dequantised values (a reading
# of the FFPA README's FP8 kernels; the quantisation scheme is this build's).

def _e4m3_from_torch(x):
    """torch's own float8_e4m3fn conversion (nearest-even), after clamping to
    the finite range as a saturating conversion does."""
    return x.to(torch.float32).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)


def _e4m3_values():
    v = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    return v   # index = code; codes 0x7f and 0xff are NaN


def pin_e4m3_encoder_matches_torch(orc):
    """The oracle's e4m3 encoder (its own bit-level rounding) equals torch's
    float8_e4m3fn conversion bit for bit on every bf16 value in [-448, 448],
    on every midpoint between neighbouring e4m3 values (the ties), and on
    random float32 values over the normal and subnormal ranges."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float32)
    bits = bits[torch.isfinite(bits) & (bits.abs() <= 448)]
    vals = _e4m3_values()
    vals = vals[torch.isfinite(vals)].to(torch.float32).unique().sort().values
    mids = (vals[1:] + vals[:-1]) / 2
    g = torch.Generator().manual_seed(8)
    rnd = (torch.rand(200000, generator=g) * 2 - 1) * 448
    tiny = (torch.rand(50000, generator=g) * 2 - 1) * 2.0 ** -5
    x = torch.cat([bits, mids, rnd, tiny, torch.tensor([0.0, -0.0, 448.0, -448.0, 500.0, -1e9])])
    got = orc.e4m3_encode(x)
    want = _e4m3_from_torch(x)
    bad = (got != want).nonzero()
    assert bad.numel() == 0, f"e4m3 code of {x[bad[0, 0]].item()!r}: {int(got[bad[0, 0]])} vs {int(want[bad[0, 0]])}"


def pin_fp8_quantizer(orc):
    """Per 128-row block of each head: the block's largest |x| gets the code of
    +-448; every value dequantises within e4m3's rounding bound (2^-4 of |x|,
    or 2^-10 of the scale in the subnormal range); multiplying the input by a
    power of two multiplies only the scales; a change in one block leaves the
    others' codes alone; a zero block gives zero codes and scale 1; rows past
    N are zero."""
    g = torch.Generator().manual_seed(81)
    B, H, N, D = 2, 3, 300, 128
    mag = torch.exp(torch.randn(B, H, 3, 1, 1, generator=g) * 3)       # blocks of very different size
    x = (torch.randn(B, H, 384, D, generator=g).view(B, H, 3, 128, D) * mag).view(B, H, 384, D)[:, :, :N]
    x = x.bfloat16().contiguous()
    x[1, 2, 128:256] = 0                                                  # one zero block
    codes, s = orc.fp8_quantize(x)
    assert codes.shape == (B, H, 384, D) and s.shape == (B, H, 3)
    assert bool((codes[:, :, N:] == 0).all()), "rows past N must be zero"
    assert bool((codes[1, 2, 128:256] == 0).all()) and s[1, 2, 1].item() == 1.0
    xf = torch.zeros(B, H, 384, D, dtype=torch.float64)
    xf[:, :, :N] = x.double()
    blocks = xf.view(B, H, 3, 128 * D).abs()
    arg = blocks.argmax(dim=-1)
    cb = codes.view(B, H, 3, 128 * D)
    top = torch.gather(cb, -1, arg.unsqueeze(-1)).squeeze(-1)
    nonzero = blocks.amax(dim=-1) > 0
    assert bool(((top[nonzero] & 0x7f) == 0x7e).all()), "a block's largest |x| must map to +-448"
    deq = _e4m3_values()[codes.long()] * s.double().repeat_interleave(128, dim=2).unsqueeze(-1)
    bound = 2.0 ** -4 * xf.abs() + 2.0 ** -10 * s.double().repeat_interleave(128, dim=2).unsqueeze(-1)
    err = (deq - xf).abs()
    assert bool((err <= bound * (1 + 1e-6)).all()), f"dequantisation error {(err - bound).max().item():.3e} over the bound"
    c8, s8 = orc.fp8_quantize((x.float() * 8).bfloat16())
    assert torch.equal(c8, codes), "power-of-two scaling must leave the codes alone"
    assert torch.equal(s8[nonzero], (s * 8)[nonzero]) and bool((s8[~nonzero] == 1).all()), \
        "power-of-two scaling must multiply the scales (a zero block keeps scale 1)"
    x2 = x.clone()
    x2[0, 1, :128] *= 3
    c2, s2 = orc.fp8_quantize(x2)
    keep = torch.ones(B, H, 384, dtype=torch.bool)
    keep[0, 1, :128] = False
    assert torch.equal(c2[keep], codes[keep]), "blocks must be quantised independently"


def pin_fp8_attention_is_attention_of_the_dequantised_inputs(orc):
    """The FP8 reference equals torch's float64 SDPA applied to the
    dequantised Q, K, V (bool and additive masks, causal, GQA, cross)."""
    cases = [
        ("mha", 1, 2, 2, 70, 90, 128, False, None, None),
        ("gqa_causal_cross", 2, 4, 2, 130, 260, 128, True, None, 0.3),
        ("bool_mask", 1, 2, 1, 40, 140, 256, False, "bool", None),
        ("f32_mask_causal", 1, 2, 2, 60, 60, 128, True, "f32", None),
    ]
    vals = _e4m3_values()
    for name, B, Hq, Hkv, Nq, Nkv, D, causal, mk, scale in cases:
        q, k, v, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed=zlib.crc32(name.encode()) % 9973)
        mask = None
        if mk == "bool":
            mask = _bool_mask(g, (B, 1, Nq, Nkv), Nq, Nkv)
        elif mk == "f32":
            mask = torch.randn(B, Hq, Nq, Nkv, generator=g)
        deq = []
        for t in (q, k, v):
            c, s = orc.fp8_quantize(t)
            d = vals[c.long()] * s.double().repeat_interleave(128, dim=2).unsqueeze(-1)
            deq.append(d[:, :, :t.shape[2]])
        o, lse = orc.attn_fp8(q, k, v, attn_mask=mask, scale=scale, is_causal=causal)
        o_ref, lse_ref = _sdpa_reference(*deq, mask, scale, causal)
        _close(o, o_ref, what=f"fp8 {name}: O")
        _close(lse, lse_ref, what=f"fp8 {name}: LSE")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
