"""CUDA path (through the C ABI) against the float64 oracle, element by element.

Small problems are compared in full (sizes that still span several 128-row
and 128-key tiles plus a ragged tail); the full-size workloads are compared
on sampled rows, computed one by one by the oracle.
"""
import math

import pytest
import torch

import exact_headdim_attention_gb300 as pkg
import oracle
from exact_headdim_attention_gb300 import workloads as wl
from tests.gpu_util import check, device_ok, gather_rows, sample_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg.load_library()
    yield


def run_dense(q, k, v, mask=None, causal=False, scale=None, out=None, lse=None, kernel=None):
    gqa = q.shape[1] != k.shape[1]
    o, l = pkg.ffpa_fwd(q.to(DEV), k.to(DEV), v.to(DEV),
                        attn_mask=None if mask is None else mask.to(DEV), is_causal=causal,
                        scale=scale, enable_gqa=gqa, return_lse=True, out=out, lse=lse,
                        kernel=kernel)
    device_ok()
    return o, l


def dense_case(B, Hq, Hkv, Nq, Nkv, D, seed, causal=False, mask=None, scale=None,
               dtype=torch.bfloat16, std=1.0, kernel=None):
    q, k, v, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed, std=std, dtype=dtype)
    m = mask(g) if callable(mask) else mask
    o, l = run_dense(q, k, v, m, causal, scale, kernel=kernel)
    o_ref, l_ref = oracle.attn_dense(q, k, v, attn_mask=m, scale=scale, is_causal=causal)
    return check(o, l, o_ref, l_ref, what=f"B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nkv{Nkv} D{D}")


# ------------------------------------------------------------------ small, full
def test_tiny_d320_with_lse():
    w = wl.tiny_d320()
    x = wl.materialize(w)
    o, l = run_dense(x["q"], x["k"], x["v"])
    o_ref, l_ref = oracle.attn_dense(x["q"], x["k"], x["v"])
    check(o, l, o_ref, l_ref, "tiny_d320")


@pytest.mark.parametrize("D", [64, 128, 192, 256, 320, 384, 448, 512, 576, 640, 768, 896, 1024])
def test_headdims_ragged(D):
    dense_case(1, 2, 2, 300, 300, D, seed=D)


@pytest.mark.parametrize("D", [72, 120, 200, 264, 520, 1000])
def test_fine_headdims_ragged(D):
    """Head dims divisible by 8 but not by 64: zero-padded 64-column chunks."""
    dense_case(1, 2, 2, 300, 300, D, seed=5000 + D)


def test_fine_headdim_causal_gqa_cross():
    dense_case(2, 4, 2, 200, 333, 120, seed=5001, causal=True)


def test_fine_headdim_additive_mask_fp16():
    B, H, Nq, Nk = 1, 2, 190, 260
    dense_case(B, H, H, Nq, Nk, 200, seed=5002, dtype=torch.float16,
               mask=lambda g: torch.randn(B, 1, Nq, Nk, generator=g))


def test_fine_headdim_leaves_padding_untouched():
    """Only D columns are written: a strided O with room past D keeps its sentinel."""
    q, k, v, _ = wl.draw_dense(1, 2, 2, 150, 150, 72, seed=5003)
    big = torch.full((1, 2, 150, 80), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = big[..., :72]
    o, l = run_dense(q, k, v, out=out)
    o_ref, l_ref = oracle.attn_dense(q, k, v)
    check(out, l, o_ref, l_ref, "fine D=72 strided out")
    assert torch.isnan(big[..., 72:].float()).all()


@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (7, 7), (127, 129), (129, 127), (1, 300), (300, 1),
                                    (64, 513), (256, 256)])
@pytest.mark.parametrize("D", [128, 512])
def test_odd_lengths(Nq, Nkv, D):
    dense_case(2, 2, 2, Nq, Nkv, D, seed=Nq * 7 + Nkv)
    if Nkv >= Nq:
        dense_case(1, 2, 2, Nq, Nkv, D, seed=Nq + Nkv, causal=True)


@pytest.mark.parametrize("D", [256, 512, 1024])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 1), (3, 3)])
def test_causal_cross_gqa(D, Hq, Hkv):
    dense_case(2, Hq, Hkv, 200, 700, D, seed=D + Hq, causal=True)


def test_noncausal_cross_gqa_scale():
    dense_case(1, 6, 2, 333, 150, 384, seed=5, scale=0.11)


MASKS = {
    "bool_b1nk": lambda B, H, Nq, Nk: (lambda g: torch.rand(B, 1, Nq, Nk, generator=g) < 0.6),
    "bool_nk": lambda B, H, Nq, Nk: (lambda g: torch.rand(Nq, Nk, generator=g) < 0.3),
    "bool_h1k": lambda B, H, Nq, Nk: (lambda g: torch.rand(1, H, 1, Nk, generator=g) < 0.8),
    "f32_bhnk": lambda B, H, Nq, Nk: (lambda g: torch.randn(B, H, Nq, Nk, generator=g)),
    "f32_neg_inf": lambda B, H, Nq, Nk: (lambda g: wl.draw_additive_mask(g, B, Nq, Nk)),
    "qtype_b1nk": lambda B, H, Nq, Nk: (lambda g: torch.randn(B, 1, Nq, Nk, generator=g).bfloat16()),
}


@pytest.mark.parametrize("name", sorted(MASKS))
@pytest.mark.parametrize("causal", [False, True])
def test_masks(name, causal):
    B, H, Nq, Nk, D = 2, 2, 150, 300, 320
    dense_case(B, H, H, Nq, Nk, D, seed=len(name), causal=causal, mask=MASKS[name](B, H, Nq, Nk))


def test_fully_masked_rows_give_zero_and_neg_inf():
    B, H, Nq, Nk, D = 1, 2, 130, 200, 128
    q, k, v, g = wl.draw_dense(B, H, H, Nq, Nk, D, seed=77)
    m = torch.rand(B, H, Nq, Nk, generator=g) < 0.5
    m[0, 0, 5] = False
    m[0, 1, 129] = False
    o, l = run_dense(q, k, v, m)
    o_ref, l_ref = oracle.attn_dense(q, k, v, attn_mask=m)
    check(o, l, o_ref, l_ref, "fully masked rows")
    assert torch.equal(o[0, 0, 5].cpu(), torch.zeros(D, dtype=o.dtype))
    assert l[0, 0, 5].item() == -math.inf and l[0, 1, 129].item() == -math.inf


@pytest.mark.parametrize("D", [320, 768])
def test_fp16(D):
    dense_case(1, 2, 1, 200, 260, D, seed=D, causal=True, dtype=torch.float16)


def test_fp16_qtype_mask():
    B, H, Nq, Nk, D = 1, 2, 140, 140, 256
    dense_case(B, H, H, Nq, Nk, D, seed=3, dtype=torch.float16,
               mask=lambda g: torch.randn(B, 1, Nq, Nk, generator=g).half())


def _qtype_mask_with_neg_inf(g, shape, Nq, Nk, dtype):
    """Additive mask in the input dtype, ~25 % -inf, the diagonal kept finite."""
    m = torch.randn(*shape, generator=g)
    m = m.masked_fill(torch.rand(*shape, generator=g) < 0.25, -math.inf)
    m = m.expand(*shape[:-2], Nq, Nk).clone()
    i = torch.arange(Nq)
    m[..., i, i + (Nk - Nq)] = 0.0
    return m.to(dtype)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [128, 512, 1024])
def test_qtype_mask_with_neg_inf(dtype, D):
    """A 16-bit additive mask holding -inf (FFPA API reference, `attn_mask`:
    floating masks are added to the scores) removes those keys."""
    B, H, Nq, Nk = 2, 2, 190, 300
    for causal in (False, True):
        dense_case(B, H, H, Nq, Nk, D, seed=D + int(causal), dtype=dtype, causal=causal,
                   mask=lambda g: _qtype_mask_with_neg_inf(g, (B, 1, Nq, Nk), Nq, Nk, dtype))


def test_strided_views():
    """[B,N,H,D] tensors viewed as [B,H,N,D] (no copy), and K/V sliced from a wider buffer."""
    g = torch.Generator().manual_seed(9)
    B, H, Nq, Nk, D = 2, 4, 190, 260, 512
    qb = torch.randn(B, Nq, H, D, generator=g).bfloat16()
    kvb = torch.randn(B, Nk, H, 2 * D, generator=g).bfloat16()
    q = qb.transpose(1, 2)
    k = kvb[..., :D].transpose(1, 2)
    v = kvb[..., D:].transpose(1, 2)
    o, l = pkg.ffpa_fwd(qb.to(DEV).transpose(1, 2), kvb.to(DEV)[..., :D].transpose(1, 2),
                        kvb.to(DEV)[..., D:].transpose(1, 2), is_causal=True, return_lse=True)
    device_ok()
    o_ref, l_ref = oracle.attn_dense(q, k, v, is_causal=True)
    check(o, l, o_ref, l_ref, "strided")


def test_guard_bands_untouched():
    """O rows padded to a wider pitch and LSE inside a larger buffer: the
    padding keeps its sentinel (no write outside the output)."""
    B, H, Nq, Nk, D = 1, 3, 200, 333, 384
    q, k, v, _ = wl.draw_dense(B, H, H, Nq, Nk, D, seed=11)
    pitch = D + 64
    big = torch.full((B, H, Nq + 2, pitch), 7.0, dtype=torch.bfloat16, device=DEV)
    out = big[:, :, 1:Nq + 1, :D]
    lbig = torch.full((B * H * Nq + 64,), 5.0, dtype=torch.float32, device=DEV)
    lse = lbig[32:32 + B * H * Nq].view(B, H, Nq)
    o, l = run_dense(q, k, v, causal=True, out=out, lse=lse)
    o_ref, l_ref = oracle.attn_dense(q, k, v, is_causal=True)
    check(o, l, o_ref, l_ref, "guard")
    bigc = big.cpu()
    assert (bigc[:, :, 0] == 7).all() and (bigc[:, :, Nq + 1] == 7).all()
    assert (bigc[..., D:] == 7).all()
    lc = lbig.cpu()
    assert (lc[:32] == 5).all() and (lc[32 + B * H * Nq:] == 5).all()


def test_empty_keys_and_queries():
    B, H, D = 1, 2, 128
    q = torch.randn(B, H, 50, D).bfloat16()
    k = torch.empty(B, H, 0, D, dtype=torch.bfloat16)
    o, l = run_dense(q, k, k)
    assert torch.equal(o.cpu(), torch.zeros_like(q)) and bool((l == -math.inf).all())
    o, l = run_dense(q[:, :, :0], q, q)
    assert o.numel() == 0
    o, l = run_dense(q[:0], q[:0], q[:0])
    assert o.numel() == 0


# --------------------------------------------------------- kernel invariants
def test_invariant_rows_sum_to_one():
    q, k, _, g = wl.draw_dense(1, 4, 2, 260, 390, 512, seed=31)
    v = torch.ones(1, 2, 390, 512, dtype=torch.bfloat16)
    o, _ = run_dense(q, k, v, causal=True, mask=torch.randn(1, 1, 260, 390, generator=g))
    assert (o.float() - 1).abs().max().item() <= 1e-2


@pytest.mark.parametrize("D,kernel", [(640, "single"), (512, "split"), (128, "dual"), (640, "split")])
def test_invariant_single_key_returns_v(D, kernel):
    """One key: O = V and LSE = scale q.k.  Exact where the running maximum is
    the row's own fp32 maximum (P = 1); the clusters of 3 and 4 CTAs (D = 640
    runs on 3) exchange maxima rounded up to bf16, so P is the bf16 rounding
    of exp2(x - m) <= 1 and O equals V to within bf16 rounding."""
    q, k, v, _ = wl.draw_dense(2, 2, 2, 129, 1, D, seed=32)
    o, l = run_dense(q, k, v, scale=0.25, kernel=kernel)
    want_o = v.expand(2, 2, 129, D)
    if pkg.selected_kernel(D, kernel=kernel) == "split" and D > 512:
        err = (o.cpu().double() - want_o.double()).abs()
        assert bool((err <= 2.0 ** -7 * want_o.double().abs() + 1e-6).all())
    else:
        assert torch.equal(o.cpu(), want_o)
    want = 0.25 * torch.einsum("bhnd,bhd->bhn", q.double(), k[:, :, 0].double())
    assert (l.cpu().double() - want).abs().max().item() <= 1e-3


def test_invariant_zero_query_lse_counts_visible_keys():
    Nq, Nk = 150, 400
    _, k, v, _ = wl.draw_dense(1, 2, 2, Nq, Nk, 256, seed=33)
    q = torch.zeros(1, 2, Nq, 256, dtype=torch.bfloat16)
    _, l = run_dense(q, k, v, causal=True)
    want = torch.tensor([math.log(i + Nk - Nq + 1) for i in range(Nq)], dtype=torch.float64)
    assert (l.cpu().double() - want).abs().max().item() <= 1e-3


def test_invariant_gqa_equals_repeated_mha():
    q, k, v, _ = wl.draw_dense(1, 8, 2, 200, 300, 512, seed=34)
    o1, l1 = run_dense(q, k, v, causal=True)
    o2, l2 = run_dense(q, k.repeat_interleave(4, 1), v.repeat_interleave(4, 1), causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_invariant_causal_visibility():
    Nq, Nk, D = 200, 330, 320
    q, k, v, g = wl.draw_dense(1, 1, 1, Nq, Nk, D, seed=35)
    o1, _ = run_dense(q, k, v, causal=True)
    t = 250
    v2 = v.clone()
    v2[0, 0, t:] = torch.randn(Nk - t, D, generator=g).bfloat16() * 3
    o2, _ = run_dense(q, k, v2, causal=True)
    limit = torch.arange(Nq) + (Nk - Nq)
    unchanged = (o1 == o2).all(dim=-1).cpu()[0, 0]
    assert bool(unchanged[limit < t].all()), "a row changed although key t is beyond its limit"
    assert (~unchanged[limit >= t]).float().mean().item() > 0.9


# ------------------------------------------- each kernel forced, same bar
@pytest.fixture(params=["single", "pair", "split"])
def variant(request):
    return request.param


@pytest.mark.parametrize("D", [128, 256, 384, 512, 768, 1024])
def test_variant_dense(variant, D):
    dense_case(1, 2, 2, 300, 300, D, seed=D + 1, kernel=variant)
    dense_case(2, 4, 1, 200, 700, D, seed=D + 2, causal=True, kernel=variant)
    dense_case(1, 2, 2, 65, 129, D, seed=D + 3, causal=True, kernel=variant)


@pytest.mark.parametrize("D", [128, 512, 1024])
def test_variant_masks(variant, D):
    B, H, Nq, Nk = 2, 2, 270, 300
    dense_case(B, H, H, Nq, Nk, D, seed=D + 4, mask=MASKS["bool_b1nk"](B, H, Nq, Nk), kernel=variant)
    dense_case(B, H, H, Nq, Nk, D, seed=D + 5, causal=True, mask=MASKS["f32_neg_inf"](B, H, Nq, Nk),
               kernel=variant)


def test_variant_fp16(variant):
    dense_case(1, 2, 1, 260, 260, 256, seed=9, causal=True, dtype=torch.float16, kernel=variant)


@pytest.mark.parametrize("D", [128, 256, 512, 768, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_variant_varlen(variant, D, causal):
    lq = [3, 130, 1, 257, 0, 64, 200, 300]
    lk = [5, 130, 2, 300, 7, 64, 450, 300]
    q, k, v, cq, ck = wl.draw_varlen(lq, lk, 4, 2, D, seed=D + int(causal))
    o, l = pkg.ffpa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(lq),
                               max(lk), causal=causal, enable_gqa=True, return_lse=True,
                               kernel=variant)
    device_ok()
    o_ref, l_ref = oracle.attn_varlen(q, k, v, cq, ck, causal=causal)
    check(o, l, o_ref, l_ref, f"varlen {variant}")


def test_variant_full_d512_sampled(variant):
    _sampled_dense(wl.headdim_sweep(512), n_random=8, kernel=variant)


# -------------------- column split on head dims padded to its instantiated shapes
@pytest.mark.parametrize("D", [192, 320, 448, 576, 640, 704, 832, 896, 960])
def test_split_padded_headdims(D):
    """D/64 chunks rounded up to 4, 6, 8, 12 or 16: the padding chunks are read
    as zeros and their output columns are not stored (guard band checked)."""
    dense_case(1, 2, 2, 300, 300, D, seed=D + 21, kernel="split")
    dense_case(2, 4, 1, 200, 700, D, seed=D + 22, causal=True, kernel="split")
    q, k, v, _ = wl.draw_dense(1, 2, 2, 140, 260, D, seed=D + 23)
    big = torch.full((1, 2, 140, D + 64), 3.0, dtype=torch.bfloat16, device=DEV)
    out = big[..., :D]
    o, l = run_dense(q, k, v, out=out, kernel="split")
    o_ref, l_ref = oracle.attn_dense(q, k, v)
    check(o, l, o_ref, l_ref, f"split padded D{D}")
    assert bool((big[..., D:] == 3.0).all()), "columns past D were written"


@pytest.mark.parametrize("D", [320, 640])
def test_split_padded_varlen(D):
    lq = [3, 130, 1, 257, 0, 64, 200]
    lk = [5, 130, 2, 300, 7, 64, 450]
    q, k, v, cq, ck = wl.draw_varlen(lq, lk, 4, 2, D, seed=D + 24)
    for causal in (False, True):
        o, l = pkg.ffpa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(lq),
                                   max(lk), causal=causal, enable_gqa=True, return_lse=True,
                                   kernel="split")
        device_ok()
        o_ref, l_ref = oracle.attn_varlen(q, k, v, cq, ck, causal=causal)
        check(o, l, o_ref, l_ref, f"varlen split padded D{D}")


# ------------------------------------------- dual-tile kernel (dense, D = 64, 128)
@pytest.mark.parametrize("D", [64, 128])
def test_dual_dense(D):
    """Two 128-row query tiles per CTA: ragged blocks (tile B partly or wholly
    past Nq), GQA, causal with Nkv > Nq, exact blocks, fp16, a negative scale."""
    dense_case(1, 2, 2, 300, 300, D, seed=D + 11, kernel="dual")        # last block: 44 rows, B empty
    dense_case(2, 4, 1, 200, 700, D, seed=D + 12, causal=True, kernel="dual")
    dense_case(1, 2, 2, 65, 129, D, seed=D + 13, causal=True, kernel="dual")
    dense_case(1, 3, 3, 512, 512, D, seed=D + 14, kernel="dual")
    dense_case(1, 2, 2, 384, 1000, D, seed=D + 15, causal=True, kernel="dual")
    dense_case(1, 2, 1, 260, 131, D, seed=D + 16, dtype=torch.float16, kernel="dual")
    dense_case(1, 2, 2, 257, 1, D, seed=D + 17, kernel="dual")          # one key
    dense_case(1, 2, 2, 129, 300, D, seed=D + 18, scale=-0.2, kernel="dual")


def test_dual_with_mask_runs_single():
    """A caller's mask at D = 128 with the dual choice: the call runs the
    single-CTA kernel and is exact."""
    B, H, Nq, Nk = 2, 2, 270, 300
    dense_case(B, H, H, Nq, Nk, 128, seed=19, mask=MASKS["bool_b1nk"](B, H, Nq, Nk), kernel="dual")


def test_dual_full_d128_sampled():
    _sampled_dense(wl.headdim_sweep(128), n_random=8, kernel="dual")


# ----------------------------------------------------------------- varlen
@pytest.mark.parametrize("D", [128, 512])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_small(D, causal):
    lq = [3, 130, 1, 257, 0, 64, 200]
    lk = [5, 130, 2, 200, 7, 64, 450]
    Hq, Hkv = 4, 2
    q, k, v, cq, ck = wl.draw_varlen(lq, lk, Hq, Hkv, D, seed=D)
    Tq = q.shape[0]
    pad = 40
    big = torch.full((Tq + 2 * pad, Hq, D), 3.0, dtype=torch.bfloat16, device=DEV)
    out = big[pad:pad + Tq]
    o, l = pkg.ffpa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(lq),
                               max(lk), causal=causal, enable_gqa=True, return_lse=True, out=out)
    device_ok()
    o_ref, l_ref = oracle.attn_varlen(q, k, v, cq, ck, causal=causal)
    check(o, l, o_ref, l_ref, "varlen")
    bc = big.cpu()
    assert (bc[:pad] == 3).all() and (bc[pad + Tq:] == 3).all()


def test_varlen_self_default_cu_k():
    lq = [100, 300, 129]
    q, k, v, cq, _ = wl.draw_varlen(lq, lq, 2, 2, 256, seed=3)
    o, l = pkg.ffpa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), None, 300, 300,
                               causal=True, return_lse=True)
    device_ok()
    o_ref, l_ref = oracle.attn_varlen(q, k, v, cq, None, causal=True)
    check(o, l, o_ref, l_ref, "varlen self")


# -------------------------------------------------------------- timeout path
def _timeout_then_correct(q, k, v, kernel=None, **kw):
    """A call whose first copy is dropped reports FFPA_ERR_DEVICE_TIMEOUT in its
    own status word (not in the shared fallback word); a normal call on the
    same context right after is correct."""
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkg.ffpa_fwd(qd, kd, vd, kernel=kernel, status=status, wait_timeout_ns=200_000_000,
                 test_drop_first_copy=True, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == pkg.FFPA_ERR_DEVICE_TIMEOUT
    assert pkg.ffpa_last_device_error() == pkg.FFPA_OK      # the fallback word was not touched
    o, l = run_dense(q, k, v, kernel=kernel)
    o_ref, l_ref = oracle.attn_dense(q, k, v)
    check(o, l, o_ref, l_ref, f"{kernel} kernel after timeout")


def test_bounded_wait_reports_timeout_and_context_survives():
    x = wl.materialize(wl.tiny_d320())
    _timeout_then_correct(x["q"], x["k"], x["v"])


def test_bounded_wait_pair_kernel():
    """Through the CTA-pair kernel: both CTAs of the pair time out."""
    q, k, v, _ = wl.draw_dense(1, 2, 2, 256, 256, 512, seed=41)
    _timeout_then_correct(q, k, v, kernel="pair")


@pytest.mark.parametrize("D", [512, 768, 1024])
def test_bounded_wait_split_kernel(D):
    """Through the column-split kernel (clusters of 2, 3 and 4 CTAs): rank 0
    loses a copy, the others wait for its tile maxima; all time out."""
    q, k, v, _ = wl.draw_dense(1, 2, 2, 200, 400, D, seed=43)
    _timeout_then_correct(q, k, v, kernel="split")


def test_bounded_wait_dual_kernel():
    """Through the dual-tile kernel: the MMA thread's first K stage never lands."""
    q, k, v, _ = wl.draw_dense(1, 2, 2, 300, 400, 128, seed=47)
    _timeout_then_correct(q, k, v, kernel="dual")


def test_bounded_wait_fallback_word():
    """Without a status word the timeout lands in the device's fallback word,
    which ffpa_last_device_error reports once and clears."""
    x = wl.materialize(wl.tiny_d320())
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    pkg.ffpa_fwd(q, k, v, wait_timeout_ns=200_000_000, test_drop_first_copy=True)
    assert pkg.ffpa_last_device_error() == pkg.FFPA_ERR_DEVICE_TIMEOUT
    assert pkg.ffpa_last_device_error() == pkg.FFPA_OK


def test_timeout_is_reported_on_its_own_stream_only():
    """Two streams, each call with its own status word; the test hook is set
    on stream A's call only.  A's word reports the timeout, B's stays zero and
    B's result is correct; later calls on both streams are correct."""
    q, k, v, _ = wl.draw_dense(1, 4, 4, 384, 512, 512, seed=47)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    sa, sb = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    st_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    st_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    pkg.ffpa_fwd(qd, kd, vd, stream=sa, status=st_a, wait_timeout_ns=300_000_000,
                 test_drop_first_copy=True)
    ob = pkg.ffpa_fwd(qd, kd, vd, stream=sb, status=st_b, wait_timeout_ns=300_000_000)
    torch.cuda.synchronize()
    assert int(st_a.item()) == pkg.FFPA_ERR_DEVICE_TIMEOUT
    assert int(st_b.item()) == pkg.FFPA_OK
    assert pkg.ffpa_last_device_error() == pkg.FFPA_OK
    o_ref, l_ref = oracle.attn_dense(q, k, v)
    check(ob, None, o_ref, l_ref, "stream B beside a timeout")
    for s in (sa, sb):
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        o, l = pkg.ffpa_fwd(qd, kd, vd, stream=s, status=st, return_lse=True)
        torch.cuda.synchronize()
        assert int(st.item()) == pkg.FFPA_OK
        check(o, l, o_ref, l_ref, "after the two-stream timeout")


def test_pointers_on_another_device_are_rejected():
    """A key tensor in host memory (pinned or not) is not a device pointer of
    q's GPU: the call returns FFPA_ERR_INVALID before any launch."""
    q, k, v, _ = wl.draw_dense(1, 2, 2, 128, 128, 128, seed=49)
    qd = q.to(DEV)
    for kh in (k, k.pin_memory()):
        with pytest.raises(ValueError):
            pkg.ffpa_fwd(qd, kh, v.to(DEV))
    with pytest.raises(ValueError):
        pkg.ffpa_fwd(qd, k.to(DEV), v.to(DEV), out=torch.empty_like(q))   # out on the host


def test_calls_from_a_thread_without_a_current_context():
    """A fresh host thread (like a framework's backward worker) has no CUDA
    context bound; the library binds the device's context for the call (the
    tensor-map encoder needs one) and puts the thread back as it found it."""
    import threading
    q, k, v, g = wl.draw_dense(1, 4, 2, 260, 260, 512, seed=51)
    dout = torch.randn(q.shape, generator=g).bfloat16()
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    res = {}

    def work():
        try:
            o, l = pkg.ffpa_fwd(qd, kd, vd, is_causal=True, enable_gqa=True, return_lse=True)
            res["fwd"] = (o, l)
            res["bwd"] = pkg.ffpa_bwd(dod, qd, kd, vd, o, l, is_causal=True, enable_gqa=True)
            torch.cuda.synchronize()
        except Exception as e:  # reported to the main thread
            res["error"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "error" not in res, res.get("error")
    device_ok()
    o_ref, l_ref = oracle.attn_dense(q, k, v, is_causal=True)
    check(*res["fwd"], o_ref, l_ref, "forward from a fresh thread")
    refs = oracle.attn_bwd_dense(q, k, v, dout, is_causal=True)
    for got, ref in zip(res["bwd"], refs):
        err = (got.double().cpu() - ref).abs().max().item()
        assert err <= 2e-2 * ref.abs().max().item()


def test_call_leaves_current_device_unchanged():
    before = torch.cuda.current_device()
    run_dense(*wl.draw_dense(1, 1, 1, 64, 64, 64, seed=50)[:3])
    assert torch.cuda.current_device() == before


# ------------------------------------------------------- full-size workloads
def _sampled_dense(w, n_random=8, kernel=None):
    """Every (batch, query head) pair: the first and last row of each 128-row
    query tile plus `n_random` seeded rows; and every output finite."""
    x = wl.materialize(w)
    o, l = run_dense(x["q"], x["k"], x["v"], mask=x["mask"], causal=w.causal, kernel=kernel)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(l).all()), f"{w.name}: non-finite"
    rows = sample_rows(w.B, w.Hq, w.Nq, n_random=n_random, seed=w.seed)
    o_ref, l_ref = oracle.attn_dense(x["q"], x["k"], x["v"], attn_mask=x["mask"], is_causal=w.causal,
                                     rows=rows)
    check(gather_rows(o, rows, w.D), l.reshape(-1)[rows.to(DEV)], o_ref, l_ref, w.name)


@pytest.mark.parametrize("D", wl.HEADDIM_SWEEP)
def test_full_headdim_sweep_sampled(D):
    _sampled_dense(wl.headdim_sweep(D))


def test_full_gqa_causal_sampled():
    _sampled_dense(wl.gqa_causal(), n_random=4)


def test_full_cross_additive_mask_sampled():
    _sampled_dense(wl.cross_additive_mask())


def test_full_varlen_causal_sampled():
    w = wl.varlen_causal()
    x = wl.materialize(w)
    q, k, v, cq = x["q"], x["k"], x["v"], x["cu_q"]
    o, l = pkg.ffpa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), None, x["max_q"],
                               x["max_k"], causal=True, enable_gqa=True, return_lse=True)
    device_ok()
    oc, lc = o.cpu(), l.cpu()
    for s, L in enumerate(x["seqlens"]):
        a = int(cq[s])
        qs = q[a:a + L].transpose(0, 1).unsqueeze(0)
        ks = k[a:a + L].transpose(0, 1).unsqueeze(0)
        vs = v[a:a + L].transpose(0, 1).unsqueeze(0)
        rows = sample_rows(1, w.Hq, L, n_random=8, seed=s)
        o_ref, l_ref = oracle.attn_dense(qs, ks, vs, is_causal=True, rows=rows)
        ok = oc[a:a + L].transpose(0, 1).reshape(-1, w.D)[rows]
        lk = lc[:, a:a + L].reshape(-1)[rows]
        check(ok, lk, o_ref, l_ref, f"varlen seq {s} (L={L})")
