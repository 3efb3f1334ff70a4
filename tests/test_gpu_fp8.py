"""FP8 (e4m3) forward through the C ABI against the oracle's FP8 reference.

Two checks per case:

* the quantisation the kernels wrote into the workspace (e4m3 codes of Q, K
  and transposed V, and the fp32 block scales) equals the oracle's, bit for
  bit (integer results of float decisions taken in the same precision);
* O is within the error bound that e4m3 implies for the one quantity the
  oracle does not round, P.  P is stored as e4m3(p * c) with c = 256 s_v /
  G <= 256; a rounded value has relative error <= 2^-4 (3 fraction bits) or
  absolute error <= 2^-10 (subnormals), so, with w the softmax weights of the
  dequantised scores, each output element obeys
      |O - O_ref| <= sum_j (2^-4 w_j + 2^-10 / c_j) |v_j| + 2^-8 |O_ref| + 1e-5
  (the last terms: O rounded to bf16, fp32 accumulation), and the mean error
  is compared with the root-sum-square of the same per-key terms.  LSE (from
  the unrounded p) must match within 1e-3.
"""
import math

import pytest
import torch

import exact_headdim_attention_gb300 as pkg
import oracle
from exact_headdim_attention_gb300 import workloads as wl
from tests.gpu_util import device_ok, sample_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
LSE_MAX = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg.load_library()
    yield


def _e4m3_values():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double()


def _dequant(codes, scales, N):
    d = _e4m3_values()[codes.long()] * scales.double().repeat_interleave(128, dim=2).unsqueeze(-1)
    return d[:, :, :N]


def run_fp8(q, k, v, mask=None, causal=False, scale=None, kernel=None):
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    ws = torch.full((pkg.fp8_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D),), 0x55, dtype=torch.uint8,
                    device=DEV)
    o, lse = pkg.ffpa_fwd_fp8(q.to(DEV), k.to(DEV), v.to(DEV),
                              attn_mask=None if mask is None else mask.to(DEV), is_causal=causal,
                              scale=scale, enable_gqa=Hq != Hkv, return_lse=True, workspace=ws,
                              kernel=kernel)
    device_ok()
    return o, lse, pkg.fp8_workspace_views(ws, B, Hq, Hkv, Nq, Nkv, D)


def check_codes(q, k, v, views, what):
    """The workspace's codes and scales equal the oracle's quantisation."""
    orc = oracle.default()
    q8, k8, v8t, sq, sk, sv = (t.cpu() for t in views)
    for name, x, codes, scales, transposed in (("Q", q, q8, sq, False), ("K", k, k8, sk, False),
                                               ("V", v, v8t, sv, True)):
        c_ref, s_ref = orc.fp8_quantize(x)
        got = codes.transpose(-1, -2) if transposed else codes
        assert torch.equal(scales, s_ref), f"{what}: {name} block scales differ"
        bad = (got != c_ref).nonzero()
        assert bad.numel() == 0, f"{what}: {name} codes differ at {bad[0].tolist()} ({bad.shape[0]} bytes)"


def fp8_bound(q, k, v, mask, causal, scale, rows=None):
    """Per-element bound (see the module docstring) on the requested rows
    (flat ids (b*Hq+h)*Nq+i; all rows when None), head by head."""
    orc = oracle.default()
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    qd, kd, vd = (_dequant(*orc.fp8_quantize(t), t.shape[2]) for t in (q, k, v))
    _, sv = orc.fp8_quantize(v)
    c = (256.0 * sv.double() / sv.double().amax(dim=-1, keepdim=True)).repeat_interleave(128, dim=2)
    c = c[:, :, :Nkv]                                               # [B, Hkv, Nkv]
    sc = scale if scale is not None else 1.0 / math.sqrt(D)
    m4 = None
    if mask is not None:
        m4 = mask
        while m4.dim() < 4:
            m4 = m4.unsqueeze(0)
        m4 = m4.expand(B, Hq, Nq, Nkv)
    rows = torch.arange(B * Hq * Nq) if rows is None else torch.as_tensor(rows)
    worst = torch.empty(rows.numel(), D, dtype=torch.float64)
    rss = torch.empty(rows.numel(), D, dtype=torch.float64)
    head = rows // Nq
    for bh in head.unique().tolist():
        sel = (head == bh).nonzero().squeeze(1)
        i = rows[sel] % Nq
        b, hq = divmod(bh, Hq)
        hk = hq // (Hq // Hkv)
        s = sc * qd[b, hq, i] @ kd[b, hk].transpose(0, 1)           # [n, Nkv]
        if m4 is not None:
            mr = m4[b, hq, i]
            s = s.masked_fill(~mr, -math.inf) if mr.dtype == torch.bool else s + mr.double()
        if causal:
            keep = torch.arange(Nkv).unsqueeze(0) <= (i + Nkv - Nq).unsqueeze(1)
            s = s.masked_fill(~keep, -math.inf)
        w = torch.softmax(s, dim=-1).nan_to_num(0.0)
        h = 2.0 ** -4 * w + (2.0 ** -10 / c[b, hk]).unsqueeze(0) * torch.isfinite(s)
        worst[sel] = h @ vd[b, hk].abs()
        rss[sel] = torch.sqrt((h * h) @ (vd[b, hk] * vd[b, hk]))
    return worst, rss


def check_fp8(o, lse, q, k, v, mask=None, causal=False, scale=None, rows=None, what=""):
    orc = oracle.default()
    D = q.shape[-1]
    o_ref, l_ref = orc.attn_fp8(q, k, v, attn_mask=mask, is_causal=causal, scale=scale, rows=rows)
    o_ref, l_ref = o_ref.reshape(-1, D), l_ref.reshape(-1)
    got = o.detach().double().cpu().reshape(-1, D)
    lgot = lse.detach().double().cpu().reshape(-1)
    if rows is not None:
        got, lgot = got[rows], lgot[rows]
    assert torch.isfinite(got).all(), f"{what}: non-finite output"
    worst, rss = fp8_bound(q, k, v, mask, causal, scale, rows)
    err = (got - o_ref).abs()
    limit = worst + 2.0 ** -8 * o_ref.abs() + 1e-5
    over = err > limit
    assert not bool(over.any()), (f"{what}: |err| {err[over][0].item():.3e} over the e4m3 bound "
                                  f"{limit[over][0].item():.3e} ({int(over.sum())} elements)")
    assert err.mean().item() <= 2.0 * rss.mean().item() + 2.0 ** -8 * o_ref.abs().mean().item(), \
        f"{what}: mean |err| {err.mean().item():.3e} vs rss bound {rss.mean().item():.3e}"
    inf = torch.isinf(l_ref)
    assert torch.equal(torch.isinf(lgot), inf), f"{what}: LSE -inf pattern differs"
    if (~inf).any():
        lerr = (lgot[~inf] - l_ref[~inf]).abs().max().item()
        assert lerr <= LSE_MAX, f"{what}: LSE max|err| {lerr:.3e}"
    return err.max().item(), err.mean().item(), worst.mean().item()


def fp8_case(B, Hq, Hkv, Nq, Nkv, D, seed, causal=False, mask=None, scale=None, dtype=torch.bfloat16,
             std=1.0, kernel=None):
    q, k, v, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed, std=std, dtype=dtype)
    m = mask(g) if callable(mask) else mask
    o, lse, views = run_fp8(q, k, v, m, causal, scale, kernel=kernel)
    what = f"fp8 {kernel or 'auto'} B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nkv{Nkv} D{D}"
    check_codes(q, k, v, views, what)
    return check_fp8(o, lse, q, k, v, m, causal, scale, what=what)


@pytest.mark.parametrize("D", [128, 256, 384, 512, 640, 768, 1024])
def test_fp8_headdims_ragged(D):
    fp8_case(1, 2, 2, 300, 300, D, seed=700 + D)


@pytest.mark.parametrize("D", [256, 512, 1024])
def test_fp8_causal_gqa_cross(D):
    fp8_case(2, 4, 2, 200, 460, D, seed=710 + D, causal=True)


@pytest.mark.parametrize("D", [256, 384, 512])
@pytest.mark.parametrize("kernel", ["single", "split"])
def test_fp8_both_kernels(D, kernel):
    """The column split (the default at these head dims) and the single-CTA
    FP8 kernel, forced: dense ragged, causal GQA cross attention, a mask."""
    fp8_case(1, 2, 2, 300, 300, D, seed=760 + D, kernel=kernel)
    fp8_case(2, 4, 2, 200, 460, D, seed=761 + D, causal=True, kernel=kernel)
    fp8_case(1, 2, 2, 129, 257, D, seed=762 + D, kernel=kernel,
             mask=lambda g: torch.rand(1, 1, 129, 257, generator=g) < 0.6)


@pytest.mark.parametrize("kind", ["bool", "f32_neg_inf", "qtype"])
def test_fp8_masks(kind):
    B, H, Nq, Nk, D = 2, 2, 150, 300, 512
    if kind == "bool":
        mask = lambda g: torch.rand(B, 1, Nq, Nk, generator=g) < 0.7  # noqa: E731
    elif kind == "f32_neg_inf":
        mask = lambda g: wl.draw_additive_mask(g, B, Nq, Nk)  # noqa: E731
    else:
        mask = lambda g: torch.randn(B, 1, Nq, Nk, generator=g).bfloat16()  # noqa: E731
    fp8_case(B, H, H, Nq, Nk, D, seed=720 + len(kind), mask=mask, causal=kind == "bool")


def test_fp8_fp16_inputs_and_scale():
    fp8_case(1, 2, 1, 200, 260, 256, seed=731, dtype=torch.float16, scale=0.07)


def test_fp8_blocks_of_very_different_size():
    """Per-block scales: Q and V rows whose magnitudes differ by 2^8 between
    blocks (logits up to ~16x larger in one query block; the LSE tolerance
    is absolute, so the logits stay moderate)."""
    q, k, v, g = wl.draw_dense(1, 2, 2, 384, 384, 256, seed=741)
    f = torch.tensor([1.0, 16.0, 1.0 / 16]).repeat_interleave(128).view(1, 1, 384, 1)
    q, v = (q.float() * f).bfloat16(), (v.float() * f).bfloat16()
    o, lse, views = run_fp8(q, k, v)
    check_codes(q, k, v, views, "mixed blocks")
    check_fp8(o, lse, q, k, v, what="mixed blocks")


def test_fp8_edges():
    # no keys: O = 0, LSE = -inf; a fully masked row likewise
    q, k, v, _ = wl.draw_dense(1, 2, 2, 50, 0, 128, seed=751)
    o, lse, _ = run_fp8(q, k, v)
    assert torch.equal(o.cpu(), torch.zeros_like(q)) and bool((lse == -math.inf).all())
    q, k, v, g = wl.draw_dense(1, 2, 2, 130, 200, 128, seed=752)
    m = torch.rand(1, 2, 130, 200, generator=g) < 0.5
    m[0, 1, 129] = False
    o, lse, _ = run_fp8(q, k, v, m)
    assert torch.equal(o[0, 1, 129].cpu(), torch.zeros(128, dtype=o.dtype)) and lse[0, 1, 129].item() == -math.inf
    # unsupported head dims and a short workspace are refused before any launch
    qd = torch.zeros(1, 2, 64, 192, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(NotImplementedError):
        pkg.ffpa_fwd_fp8(qd, qd, qd)
    qd = torch.zeros(1, 2, 64, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd_fp8(qd, qd, qd, workspace=torch.empty(1024, dtype=torch.uint8, device=DEV))


@pytest.mark.parametrize("kernel", ["single", "split"])
def test_fp8_bounded_wait_reports_timeout(kernel):
    q, k, v, _ = wl.draw_dense(1, 2, 2, 200, 300, 512, seed=761)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkg.ffpa_fwd_fp8(qd, kd, vd, status=status, wait_timeout_ns=200_000_000, test_drop_first_copy=True,
                     kernel=kernel)
    torch.cuda.synchronize()
    assert int(status.item()) == pkg.FFPA_ERR_DEVICE_TIMEOUT
    o, lse, views = run_fp8(q, k, v, kernel=kernel)
    check_fp8(o, lse, q, k, v, what=f"{kernel} after timeout")


def test_fp8_full_d512_sampled():
    """The bench workload (B1 H16 N4096 D512): every code and scale, and
    sampled rows of every head within the bound."""
    w = wl.headdim_sweep(512)
    x = wl.materialize(w)
    q, k, v = x["q"], x["k"], x["v"]
    o, lse, views = run_fp8(q, k, v)
    check_codes(q, k, v, views, w.name)
    rows = sample_rows(w.B, w.Hq, w.Nq, n_random=4, seed=w.seed)
    check_fp8(o, lse, q, k, v, rows=rows, what=w.name)
