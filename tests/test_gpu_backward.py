"""Backward kernels (through the C ABI ``ffpa_bwd``) against the float64 oracle.

The gradients are those of sum(O * dO) for a seeded upstream gradient dO;
the CUDA path starts from its own forward's O and LSE, the oracle from the
definition.  Small problems are compared in full (several 128-row and
128-key tiles plus a ragged tail); large ones on sampled rows that the
oracle computes one by one.

Tolerance, from the arithmetic of the path: P and dS are rounded to 16 bits
before the tensor-core products (relative error <= u = 2^-9 for bf16), the
products accumulate in fp32, and dQ, dK, dV are rounded to 16 bits once
more.  An output element is a sum of many terms with independent rounding
errors of relative size ~u, so its error is a few u of the typical output
magnitude: max |err| <= 2e-2 * max |ref| and mean |err| <= 1e-2 * mean |ref|
(about 10 u and 5 u).  Exactly zero gradients (a single key) have their own
bound in test_bwd_single_key.  delta = rowsum(dO * O) is an fp32 dot product
of the 16-bit inputs: relative 1e-4 of sum |dO * O|.
"""
import pytest
import torch

import exact_headdim_attention_gb300 as pkg
import oracle
from exact_headdim_attention_gb300 import workloads as wl
from tests.gpu_util import device_ok

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
G_MAX, G_MEAN = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg.load_library()
    yield


def check_grad(got, ref, what, g_max=G_MAX, g_mean=G_MEAN):
    got = got.detach().double().cpu().reshape(ref.shape)
    assert torch.isfinite(got).all(), f"{what}: non-finite values"
    if ref.numel() == 0:
        return 0.0, 0.0
    err = (got - ref).abs()
    rmax, rmean = ref.abs().max().item(), ref.abs().mean().item()
    emax, emean = err.max().item(), err.mean().item()
    print(f"{what}: max|err|/max|ref| {emax / max(rmax, 1e-300):.2e}  "
          f"mean|err|/mean|ref| {emean / max(rmean, 1e-300):.2e}")
    assert emax <= g_max * rmax, f"{what}: max|err| {emax:.3e} > {g_max} * {rmax:.3e}"
    assert emean <= g_mean * rmean, f"{what}: mean|err| {emean:.3e} > {g_mean} * {rmean:.3e}"
    return emax, emean


def draw(B, Hq, Hkv, Nq, Nkv, D, seed, dtype=torch.bfloat16):
    q, k, v, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed, dtype=dtype)
    dout = torch.randn(B, Hq, Nq, D, generator=g).to(dtype)
    return q, k, v, dout


def gpu_backward(q, k, v, dout, causal=False, scale=None, mask=None, workspace="auto"):
    """Forward then backward on the GPU, as a training step would run them.
    workspace="auto" takes the stored-tile path where it applies (D = 128,
    256, 384, 512), None the slice kernels."""
    gqa = q.shape[1] != k.shape[1]
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    md = None if mask is None else mask.to(DEV)
    o, lse = pkg.ffpa_fwd(qd, kd, vd, attn_mask=md, is_causal=causal, scale=scale, enable_gqa=gqa,
                          return_lse=True)
    dq, dk, dv, delta = pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, is_causal=causal, scale=scale,
                                     enable_gqa=gqa, attn_mask=md, return_delta=True,
                                     workspace=workspace)
    device_ok()
    return dq, dk, dv, delta, o


def bwd_case(B, Hq, Hkv, Nq, Nkv, D, seed, causal=False, scale=None, dtype=torch.bfloat16,
             mask=None, workspace="auto"):
    q, k, v, dout = draw(B, Hq, Hkv, Nq, Nkv, D, seed, dtype)
    m = mask(torch.Generator().manual_seed(seed + 7)) if callable(mask) else mask
    dq, dk, dv, delta, o = gpu_backward(q, k, v, dout, causal, scale, m, workspace)
    rq, rk, rv = oracle.attn_bwd_dense(q, k, v, dout, attn_mask=m, scale=scale, is_causal=causal)
    tag = f"B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nkv{Nkv} D{D} causal={causal} {dtype}"
    check_grad(dq, rq, f"{tag} dQ")
    check_grad(dk, rk, f"{tag} dK")
    check_grad(dv, rv, f"{tag} dV")
    # delta is rowsum(dO * O) over the CUDA path's own O
    want = (dout.double() * o.double().cpu()).sum(-1)
    scale_d = (dout.double() * o.double().cpu()).abs().sum(-1)
    assert ((delta.double().cpu() - want).abs() <= 1e-4 * scale_d + 1e-6).all(), f"{tag} delta"


# ------------------------------------------------------------------ small, full
@pytest.mark.parametrize("D", [64, 128, 192, 256, 320, 448, 512, 640, 768, 1024])
def test_bwd_headdims_ragged(D):
    bwd_case(1, 2, 2, 300, 300, D, seed=100 + D)


@pytest.mark.parametrize("D", [64, 128, 384, 512])
def test_bwd_causal(D):
    bwd_case(1, 2, 2, 300, 300, D, seed=200 + D, causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_gqa_cross(causal):
    bwd_case(2, 4, 2, 200, 333, 128, seed=31, causal=causal)


def test_bwd_mqa_causal_d512():
    bwd_case(1, 4, 1, 256, 256, 512, seed=32, causal=True)


def test_bwd_fp16_causal():
    bwd_case(1, 2, 2, 200, 200, 256, seed=33, causal=True, dtype=torch.float16)


def test_bwd_explicit_scale():
    bwd_case(1, 2, 1, 150, 260, 192, seed=34, scale=0.11, causal=True)


@pytest.mark.parametrize("Nq,Nkv,causal", [(7, 7, True), (1, 300, True), (2, 300, False),
                                           (129, 127, False), (127, 129, True), (128, 128, True)])
def test_bwd_lengths(Nq, Nkv, causal):
    bwd_case(1, 2, 2, Nq, Nkv, 128, seed=Nq * 1000 + Nkv, causal=causal)


@pytest.mark.parametrize("Nq,D", [(1, 128), (300, 128), (300, 256)])
def test_bwd_single_key(Nq, D):
    """Nkv = 1: the softmax is the constant 1, so dV_0 = sum_i dO_i and dQ = dK = 0.
    The kernel reaches the zeros up to rounding: the recomputed P = exp2(s - lse)
    is 1 within fp32 rounding (|P - 1| <= 2^-21), and dP_i = dO_i . V_0 (tensor
    core) and delta_i = dO_i . O_i (O = V_0 exactly) are the same D products
    summed in fp32 in different orders, so they differ by at most
    D * 2^-24 * sum_d |dO_id V_0d| (a factor 2 above that is taken: D 2^-23).
    Hence |dS_i| <= e_i = 2^-21 |dP_i| + D 2^-23 sum_d |dO_id V_0d|, |dQ_i| <=
    scale e_i max|K_0| and |dK_0| <= scale sum_i e_i max|Q_i|; a factor 2 covers
    the 16-bit roundings of dS (stored tiles at D = 256) and of the outputs."""
    q, k, v, dout = draw(1, 2, 2, Nq, 1, D, seed=38 + Nq + D)
    dq, dk, dv, _, _ = gpu_backward(q, k, v, dout)
    scale = D ** -0.5
    prod = dout.double() * v.double()                                    # [1,2,Nq,D]
    e = 2.0 ** -21 * prod.sum(-1).abs() + D * 2.0 ** -23 * prod.abs().sum(-1)   # [1,2,Nq]
    bq = 2 * scale * e.unsqueeze(-1) * k.double().abs().amax(-1, keepdim=True)
    assert (dq.double().cpu().abs() <= bq).all(), "dQ not zero within the rounding bound"
    bk = 2 * scale * (e * q.double().abs().amax(-1)).sum(-1)               # [1,2]
    assert (dk.double().cpu().abs().amax(-1).squeeze(-1) <= bk).all(), "dK not zero within the bound"
    check_grad(dv, dout.double().sum(2, keepdim=True), f"Nq{Nq} Nkv1 dV")


# ------------------------------------------------------------------ stored tiles vs slices
# D = 128, 256, 384, 512 take the stored-tile path by default; the same cases on
# the slice kernels (workspace=None) keep both paths checked.
@pytest.mark.parametrize("D,causal", [(256, False), (384, True), (512, False), (512, True)])
def test_bwd_sliced_path(D, causal):
    bwd_case(1, 2, 2, 300, 300, D, seed=300 + D + causal, causal=causal, workspace=None)


@pytest.mark.parametrize("Nq,Nkv,causal", [(200, 333, False), (130, 390, True), (1, 129, True),
                                           (129, 3, False), (256, 256, True)])
def test_bwd_tiles_lengths_gqa(Nq, Nkv, causal):
    """Cross lengths, ragged tails on both sides, lower-right causal with more
    keys than queries, GQA groups of 4 summed into one dK/dV tile."""
    bwd_case(2, 4, 1, Nq, Nkv, 256, seed=Nq + 7 * Nkv, causal=causal)


def test_bwd_tiles_masks():
    B, H, Nq, Nkv = 1, 2, 190, 260
    bwd_case(B, H, H, Nq, Nkv, 384, seed=57, mask=_bool_mask_with_dead_rows(B, H, Nq, Nkv))
    bwd_case(2, 4, 2, 150, 270, 256, seed=58, causal=True,
             mask=lambda g: torch.randn(1, 1, 150, 270, generator=g).bfloat16())


def _sentinel_workspace(q, k, D):
    B, Hq, Nq, _ = q.shape
    need = pkg.bwd_workspace_bytes(B, Hq, k.shape[1], Nq, k.shape[2], D, False)
    assert need == (2 * B * Hq * (-(-Nq // 128)) * (-(-k.shape[2] // 128)) + 1) * 32768
    return need


def _stored_p(ws, BH, n_qt, n_kt):
    """The stored P of the workspace as [BH, n_qt 128, n_kt 128]: blocks of
    32 KB per (bh, query tile, key tile) after the 32 KB zero block, 16-byte
    unit u (keys 8u..8u+7) of row r at byte 2048 u + 16 r."""
    blocks = ws[32768: 32768 + BH * n_qt * n_kt * 32768].view(torch.bfloat16).float().cpu()
    t = blocks.reshape(BH, n_qt, n_kt, 16, 128, 8).permute(0, 1, 4, 2, 3, 5)
    return t.reshape(BH, n_qt * 128, n_kt * 128)


def test_bwd_tiles_workspace_use():
    """A large-enough caller workspace is written (the stored-tile path ran:
    every stored P value is a probability, the rows of P sum to 1 over the
    keys); one byte too small leaves it untouched (the slice kernels ran).
    Both give the oracle's gradients."""
    B, H, N, D = 1, 2, 200, 256
    q, k, v, dout = draw(B, H, H, N, N, D, seed=59)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    o, lse = pkg.ffpa_fwd(qd, kd, vd, return_lse=True)
    need = _sentinel_workspace(q, k, D)
    rq, rk, rv = oracle.attn_bwd_dense(q, k, v, dout)
    for extra, used in ((64, True), (-1, False)):
        ws = torch.full((need + extra,), 0xFF, dtype=torch.uint8, device=DEV)
        dq, dk, dv = pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, workspace=ws)
        device_ok()
        check_grad(dq, rq, f"workspace {need + extra} dQ")
        check_grad(dk, rk, f"workspace {need + extra} dK")
        check_grad(dv, rv, f"workspace {need + extra} dV")
        if not used:
            assert bool((ws == 0xFF).all()), "a too-small workspace was written"
            continue
        assert bool((ws[:32768] == 0).all()), "the zero block"
        p = _stored_p(ws, B * H, 2, 2)
        assert torch.isfinite(p).all() and (p >= 0).all() and (p <= 1.0001).all()
        assert (p[:, N:, :] == 0).all() and (p[:, :, N:] == 0).all(), "padding of the stored P"
        rowsum = p[:, :N, :N].double().sum(-1)
        assert ((rowsum - 1).abs() < 2e-2).all(), "stored P rows do not sum to 1"


# ------------------------------------------------------------------ masks
def _bool_mask_with_dead_rows(B, H, Nq, Nkv):
    def make(g):
        m = torch.rand(B, H, Nq, Nkv, generator=g) < 0.6
        m[:, :, 3] = False                    # fully masked rows: LSE = -inf, no contribution
        m[0, -1, Nq - 1] = False
        return m
    return make


def test_bwd_bool_mask_with_dead_rows():
    bwd_case(2, 2, 2, 200, 300, 128, seed=51, mask=_bool_mask_with_dead_rows(2, 2, 200, 300))


def test_bwd_additive_f32_mask_d512():
    B, H, Nq, Nkv = 1, 2, 190, 260
    bwd_case(B, H, H, Nq, Nkv, 512, seed=52,
             mask=lambda g: torch.randn(B, H, Nq, Nkv, generator=g))


def test_bwd_qtype_mask_broadcast_causal():
    Nq, Nkv = 150, 270
    bwd_case(2, 4, 2, Nq, Nkv, 128, seed=53, causal=True,
             mask=lambda g: torch.randn(1, 1, Nq, Nkv, generator=g).bfloat16())


def test_bwd_bool_mask_fp16_gqa():
    B, Hq, Nq, Nkv = 1, 4, 140, 140
    bwd_case(B, Hq, 2, Nq, Nkv, 256, seed=54, dtype=torch.float16,
             mask=lambda g: (torch.rand(B, 1, Nq, Nkv, generator=g) < 0.7) | torch.eye(Nq, Nkv, dtype=torch.bool))


def test_bwd_strided_views():
    """[B, N, H, D] storage viewed as [B, H, N, D] (non-contiguous strides)."""
    g = torch.Generator().manual_seed(35)
    B, H, Hkv, N, D = 2, 4, 2, 190, 256
    q = torch.randn(B, N, H, D, generator=g).bfloat16().transpose(1, 2)
    k = torch.randn(B, N, Hkv, D, generator=g).bfloat16().transpose(1, 2)
    v = torch.randn(B, N, Hkv, D, generator=g).bfloat16().transpose(1, 2)
    dout = torch.randn(B, N, H, D, generator=g).bfloat16().transpose(1, 2)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    o, lse = pkg.ffpa_fwd(qd, kd, vd, is_causal=True, enable_gqa=True, return_lse=True)
    dq, dk, dv = pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, is_causal=True, enable_gqa=True)
    device_ok()
    rq, rk, rv = oracle.attn_bwd_dense(q, k, v, dout, is_causal=True)
    check_grad(dq, rq, "strided dQ")
    check_grad(dk, rk, "strided dK")
    check_grad(dv, rv, "strided dV")


def test_bwd_empty_sides():
    """No query rows: dK = dV = 0.  No keys: dQ = 0."""
    q, k, v, dout = draw(1, 2, 2, 0, 200, 128, seed=36)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    o = torch.empty_like(qd)
    lse = torch.empty(1, 2, 0, device=DEV)
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, dk=dk, dv=dv)
    device_ok()
    assert torch.equal(dk.float().cpu(), torch.zeros(dk.shape)) and torch.equal(dv.float().cpu(), torch.zeros(dv.shape))
    q, k, v, dout = draw(1, 2, 2, 130, 0, 128, seed=37)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    o, lse = pkg.ffpa_fwd(qd, kd, vd, return_lse=True)
    dq = torch.full_like(qd, float("nan"))
    pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, dq=dq)
    device_ok()
    assert torch.equal(dq.float().cpu(), torch.zeros(dq.shape))


# ------------------------------------------------------------------ large, sampled
def _sampled(B, Hq, Hkv, N, D, seed, causal, q_heads, kv_heads, n_rows=48, workspace="auto"):
    q, k, v, dout = draw(B, Hq, Hkv, N, N, D, seed)
    dq, dk, dv, _, _ = gpu_backward(q, k, v, dout, causal, workspace=workspace)
    g = torch.Generator().manual_seed(seed)
    edge = [0, 1, 127, 128, N - 129, N - 1]
    qr = [h * N + i for h in q_heads for i in edge + torch.randint(0, N, (n_rows,), generator=g).tolist()]
    kr = [h * N + j for h in kv_heads for j in edge + torch.randint(0, N, (n_rows // 2,), generator=g).tolist()]
    rq, rk, rv = oracle.attn_bwd_rows(q, k, v, dout, qr, kr, is_causal=causal)
    tag = f"B{B} Hq{Hq} Hkv{Hkv} N{N} D{D} causal={causal}"
    check_grad(dq.reshape(-1, D)[torch.tensor(qr, device=DEV)], rq, f"{tag} sampled dQ")
    check_grad(dk.reshape(-1, D)[torch.tensor(kr, device=DEV)], rk, f"{tag} sampled dK")
    check_grad(dv.reshape(-1, D)[torch.tensor(kr, device=DEV)], rv, f"{tag} sampled dV")


@pytest.mark.parametrize("workspace", ["auto", None])
def test_bwd_full_size_d512_sampled(workspace):
    """The self-attention workload B1 H16 N4096 D512 on sampled rows (stored
    tiles, as the benchmark runs it, and the slice kernels): dQ rows of every
    head, dK/dV rows of the first, a middle and the last head."""
    _sampled(1, 16, 16, 4096, 512, seed=41, causal=False, q_heads=list(range(16)), kv_heads=[0, 7, 15],
             workspace=workspace)


@pytest.mark.parametrize("D", [128, 256, 384])
def test_bwd_full_size_tiles_sampled(D):
    """B1 H16 N4096 at the other stored-tile head dims (one workspace block
    per tile, D/64 chunks per operand) on sampled rows."""
    _sampled(1, 16, 16, 4096, D, seed=44 + D, causal=False, q_heads=list(range(16)), kv_heads=[0, 15])


def test_bwd_gqa_causal_d512_sampled():
    _sampled(1, 8, 2, 2048, 512, seed=42, causal=True, q_heads=list(range(8)), kv_heads=[0, 1])


# ------------------------------------------------------------------ autograd
def test_autograd_through_custom_op():
    q, k, v, dout = draw(1, 4, 2, 260, 260, 512, seed=43)
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    o = pkg.ffpa_attn_func(qd, kd, vd, is_causal=True, enable_gqa=True)
    o.backward(dout.to(DEV))
    device_ok()
    rq, rk, rv = oracle.attn_bwd_dense(q, k, v, dout, is_causal=True)
    check_grad(qd.grad, rq, "autograd dQ")
    check_grad(kd.grad, rk, "autograd dK")
    check_grad(vd.grad, rv, "autograd dV")


def test_autograd_with_bool_mask():
    q, k, v, dout = draw(1, 2, 2, 160, 200, 128, seed=44)
    mask = torch.rand(160, 200, generator=torch.Generator().manual_seed(45)) < 0.8
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    o = pkg.ffpa_attn_func(qd, kd, vd, attn_mask=mask.to(DEV))
    o.backward(dout.to(DEV))
    device_ok()
    rq, rk, rv = oracle.attn_bwd_dense(q, k, v, dout, attn_mask=mask)
    check_grad(qd.grad, rq, "autograd masked dQ")
    check_grad(kd.grad, rk, "autograd masked dK")
    check_grad(vd.grad, rv, "autograd masked dV")


def test_autograd_lse_output_unused_or_used():
    """An LSE that is returned but not used by the loss needs no gradient (the
    backward receives none and reads nothing from the device); a loss that
    uses it raises, since no LSE gradient is formed."""
    q, k, v, dout = draw(1, 2, 2, 150, 150, 128, seed=48)
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    o, lse = pkg.ffpa_attn_func(qd, kd, vd, is_causal=True, return_lse=True)
    o.backward(dout.to(DEV))
    device_ok()
    rq, rk, rv = oracle.attn_bwd_dense(q, k, v, dout, is_causal=True)
    check_grad(qd.grad, rq, "dQ with LSE returned")
    o, lse = pkg.ffpa_attn_func(qd, kd, vd, return_lse=True)
    with pytest.raises(NotImplementedError):
        (o.sum() + lse.sum()).backward()


def test_autograd_mask_gradient_raises():
    q, k, v, _ = draw(1, 2, 2, 64, 64, 128, seed=46)
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    bias = torch.zeros(64, 64, device=DEV, requires_grad=True)
    o = pkg.ffpa_attn_func(qd, kd, vd, attn_mask=bias)
    with pytest.raises(NotImplementedError):
        o.sum().backward()


# ------------------------------------------------------------------ bounded waits
@pytest.mark.parametrize("workspace", ["auto", None])
def test_bwd_bounded_wait_reports_timeout_and_context_survives(workspace):
    """The first ring stage of every backward CTA is dropped (test hook): the MMA
    thread's wait on it runs out, the kernels drain, free TMEM and report
    FFPA_ERR_DEVICE_TIMEOUT; the next call on the same context is correct.
    Both the stored-tile kernels and the slice kernels."""
    q, k, v, dout = draw(1, 2, 2, 200, 200, 256, seed=61)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    o, lse = pkg.ffpa_fwd(qd, kd, vd, return_lse=True)
    device_ok()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, status=status, wait_timeout_ns=200_000_000,
                 test_drop_first_copy=True, workspace=workspace)
    torch.cuda.synchronize()
    assert int(status.item()) == pkg.FFPA_ERR_DEVICE_TIMEOUT
    assert pkg.ffpa_last_device_error() == pkg.FFPA_OK
    dq, dk, dv = pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, workspace=workspace)
    device_ok()
    rq, rk, rv = oracle.attn_bwd_dense(q, k, v, dout)
    check_grad(dq, rq, "dQ after timeout")
    check_grad(dk, rk, "dK after timeout")
    check_grad(dv, rv, "dV after timeout")


# ------------------------------------------------------------------ varlen
def varlen_bwd_case(lq, lk, Hq, Hkv, D, seed, causal, workspace="auto"):
    g = torch.Generator().manual_seed(seed)
    cu_q = torch.tensor([0] + torch.tensor(lq).cumsum(0).tolist(), dtype=torch.int32)
    cu_k = torch.tensor([0] + torch.tensor(lk).cumsum(0).tolist(), dtype=torch.int32)
    Tq, Tk = sum(lq), sum(lk)
    q = torch.randn(Tq, Hq, D, generator=g).bfloat16()
    k = torch.randn(Tk, Hkv, D, generator=g).bfloat16()
    v = torch.randn(Tk, Hkv, D, generator=g).bfloat16()
    dout = torch.randn(Tq, Hq, D, generator=g).bfloat16()
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    cqd, ckd = cu_q.to(DEV), cu_k.to(DEV)
    gqa = Hq != Hkv
    o, lse = pkg.ffpa_fwd_varlen(qd, kd, vd, cqd, ckd, max(lq), max(lk), causal=causal,
                                 enable_gqa=gqa, return_lse=True)
    dq, dk, dv, delta = pkg.ffpa_bwd_varlen(dod, qd, kd, vd, o, lse, cqd, ckd, max(lq), max(lk),
                                            causal=causal, enable_gqa=gqa, return_delta=True,
                                            workspace=workspace)
    device_ok()
    rq, rk, rv = oracle.attn_bwd_varlen(q, k, v, dout, cu_q, cu_k, causal=causal)
    tag = f"varlen lq={lq} lk={lk} Hq{Hq} Hkv{Hkv} D{D} causal={causal}"
    check_grad(dq, rq, f"{tag} dQ")
    check_grad(dk, rk, f"{tag} dK")
    check_grad(dv, rv, f"{tag} dV")
    prod = dout.double() * o.double().cpu()
    assert ((delta.double().cpu() - prod.sum(-1).T).abs() <= 1e-4 * prod.abs().sum(-1).T + 1e-6).all()


def test_bwd_varlen_causal_gqa():
    varlen_bwd_case([300, 128, 1, 450], [300, 128, 1, 450], 4, 2, 128, seed=71, causal=True)


def test_bwd_varlen_cross_d512():
    varlen_bwd_case([100, 200, 0, 64], [150, 200, 30, 300], 2, 2, 512, seed=72, causal=False)


def test_bwd_varlen_causal_fewer_keys():
    """Rows that see no key (lower-right alignment with Lk < Lq) get zero gradients."""
    varlen_bwd_case([50, 10, 257], [20, 10, 260], 2, 1, 256, seed=73, causal=True)


@pytest.mark.parametrize("workspace", ["auto", None])
@pytest.mark.parametrize("D,causal", [(512, True), (384, False), (256, True)])
def test_bwd_varlen_tiles(D, causal, workspace):
    """Stored tiles (workspace="auto") and slice kernels on ragged packed
    sequences: an empty sequence, one shorter than a tile, GQA groups of 2."""
    varlen_bwd_case([300, 0, 77, 450, 129], [300, 0, 77, 450, 129], 4, 2, D, seed=80 + D, causal=causal,
                    workspace=workspace)


def test_bwd_varlen_tiles_cross_fewer_keys():
    """Cross lengths per sequence, some with fewer keys than queries (lower-right
    causal: the first rows see no key and get zero gradients)."""
    varlen_bwd_case([200, 33, 300], [150, 40, 500], 2, 1, 512, seed=91, causal=True)
    varlen_bwd_case([200, 33, 300], [150, 40, 500], 2, 2, 256, seed=92, causal=False)


@pytest.mark.parametrize("workspace", ["auto", None])
def test_bwd_varlen_full_size_sampled(workspace):
    """The packed causal workload (8 sequences of 512..4096 rows, Hq16 Hkv4,
    D512) at full size: dQ rows of every query head of every sequence, dK/dV
    rows of every KV head in the shortest sequence and of the last KV head in
    the longest (the oracle's cost per KV head grows with the group's rows
    times the sequence length).  Each sequence is its own dense causal
    problem for the oracle."""
    w = wl.varlen_causal()
    m = wl.materialize(w)
    q, k, v, cu, lens = m["q"], m["k"], m["v"], m["cu_q"], m["seqlens"]
    g = torch.Generator().manual_seed(w.seed + 2)
    dout = torch.randn(q.shape, generator=g).to(q.dtype)
    qd, kd, vd, dod, cud = (t.to(DEV) for t in (q, k, v, dout, cu))
    o, lse = pkg.ffpa_fwd_varlen(qd, kd, vd, cud, None, max(lens), max(lens), causal=True,
                                 enable_gqa=True, return_lse=True)
    dq, dk, dv = pkg.ffpa_bwd_varlen(dod, qd, kd, vd, o, lse, cud, None, max(lens), max(lens),
                                     causal=True, enable_gqa=True, workspace=workspace)
    device_ok()
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    by_len = sorted(range(len(lens)), key=lambda s: lens[s])
    kv_heads = {by_len[0]: list(range(w.Hkv)), by_len[-1]: [w.Hkv - 1]}
    for s, L in enumerate(lens):
        a = int(cu[s])
        dense = lambda t: t[a:a + L].permute(1, 0, 2).unsqueeze(0)   # [1, H, L, D] view
        edge = [0, 1, 127, 128, L - 129, L - 1]
        q_rows = edge + torch.randint(0, L, (8,), generator=g).tolist()
        qr = [h * L + i for h in range(w.Hq) for i in q_rows]
        hks = kv_heads.get(s, [])
        k_rows = edge + torch.randint(0, L, (16,), generator=g).tolist() if hks else []
        kr = [hk * L + j for hk in hks for j in k_rows]
        rq, rk, rv = oracle.attn_bwd_rows(dense(q), dense(k), dense(v), dense(dout), qr, kr,
                                          is_causal=True)
        tag = f"varlen full size seq {s} (L={L})"
        check_grad(torch.stack([dq[a + i, h] for h in range(w.Hq) for i in q_rows]), rq, f"{tag} dQ")
        if kr:
            check_grad(torch.stack([dk[a + j, hk] for hk in hks for j in k_rows]), rk, f"{tag} dK heads {hks}")
            check_grad(torch.stack([dv[a + j, hk] for hk in hks for j in k_rows]), rv, f"{tag} dV heads {hks}")


def test_bwd_varlen_small_workspace_reports_invalid():
    """A workspace that holds the header and three blocks but fewer than the
    sequences need: the kernels skip the blocks past its end (no access
    outside it) and record FFPA_ERR_INVALID in the call's status word; the
    next call with a workspace of the full size is correct."""
    lq = [300, 450]
    g = torch.Generator().manual_seed(95)
    cu = torch.tensor([0, 300, 750], dtype=torch.int32)
    T, H, D = 750, 2, 512
    q, k, v, dout = (torch.randn(T, H, D, generator=g).bfloat16() for _ in range(4))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    cud = cu.to(DEV)
    o, lse = pkg.ffpa_fwd_varlen(qd, kd, vd, cud, None, 450, 450, causal=True, return_lse=True)
    device_ok()
    need = pkg.varlen_bwd_workspace_bytes(cu.tolist(), cu.tolist(), H, H, D, True)
    small = torch.zeros(1024 + 3 * 32768, dtype=torch.uint8, device=DEV)
    assert small.numel() < need
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkg.ffpa_bwd_varlen(dod, qd, kd, vd, o, lse, cud, None, 450, 450, causal=True, workspace=small,
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == pkg.FFPA_ERR_INVALID
    assert pkg.ffpa_last_device_error() == pkg.FFPA_OK
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    dq, dk, dv = pkg.ffpa_bwd_varlen(dod, qd, kd, vd, o, lse, cud, None, 450, 450, causal=True, workspace=ws)
    device_ok()
    rq, rk, rv = oracle.attn_bwd_varlen(q, k, v, dout, cu, cu, causal=True)
    check_grad(dq, rq, "varlen dQ after a small workspace")
    check_grad(dk, rk, "varlen dK after a small workspace")
    check_grad(dv, rv, "varlen dV after a small workspace")


def test_autograd_varlen():
    lq = [130, 70, 260]
    g = torch.Generator().manual_seed(74)
    cu = torch.tensor([0] + torch.tensor(lq).cumsum(0).tolist(), dtype=torch.int32)
    T, H, D = sum(lq), 2, 192
    q, k, v, dout = (torch.randn(T, H, D, generator=g).bfloat16() for _ in range(4))
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    o = pkg.ffpa_attn_varlen_func(qd, kd, vd, cu.to(DEV), None, max(lq), max(lq), causal=True)
    o.backward(dout.to(DEV))
    device_ok()
    rq, rk, rv = oracle.attn_bwd_varlen(q, k, v, dout, cu, causal=True)
    check_grad(qd.grad, rq, "autograd varlen dQ")
    check_grad(kd.grad, rk, "autograd varlen dK")
    check_grad(vd.grad, rv, "autograd varlen dV")
