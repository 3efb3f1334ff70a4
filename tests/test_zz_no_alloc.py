"""ffpa_bwd_noalloc, the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: plugins that receive only their tensors'
pointers from a host framework, runtimes that reserve every byte of device
memory up front, and latency-bound paths that cannot afford an allocation
(which may synchronise the device or fail when memory runs out).  For them
the backward keeps its per-row scratch in a fixed array inside the library.
These tests call that entry point through the C ABI and compare its
gradients with those of ffpa_bwd (which takes the scratch from the caller).

The file name makes pytest collect it last, so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import exact_headdim_attention_gb300 as pkg
from exact_headdim_attention_gb300 import workloads as wl

DEV = torch.device("cuda:0")
G_MAX, G_MEAN = 2e-2, 1e-2      # the backward tests' bound, relative to the reference's magnitude


def _strides(t):
    return (ctypes.c_int64 * 4)(*t.stride())


def _close(got, ref, what):
    got, ref = got.double().cpu(), ref.double().cpu()
    assert torch.isfinite(got).all(), f"{what}: non-finite values"
    err = (got - ref).abs()
    rmax, rmean = ref.abs().max().item(), ref.abs().mean().item()
    assert err.max().item() <= G_MAX * rmax, f"{what}: max|err| {err.max().item():.3e}"
    assert err.mean().item() <= G_MEAN * rmean, f"{what}: mean|err| {err.mean().item():.3e}"


def _prepare(B, Hq, Hkv, Nq, Nkv, D, seed, causal):
    """Device inputs, the forward's O and LSE, and ffpa_bwd's gradients."""
    q, k, v, g = wl.draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed)
    dout = torch.randn(q.shape, generator=g).to(q.dtype)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    gqa = Hq != Hkv
    o, lse = pkg.ffpa_fwd(qd, kd, vd, is_causal=causal, enable_gqa=gqa, return_lse=True)
    ref = pkg.ffpa_bwd(dod, qd, kd, vd, o, lse, is_causal=causal, enable_gqa=gqa)
    torch.cuda.synchronize()
    return (qd, kd, vd, dod, o, lse, causal, gqa), ref


def _noalloc(lib, qd, kd, vd, dod, o, lse, causal, gqa):
    """One ffpa_bwd_noalloc call through the C ABI into caller-owned outputs."""
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    B, Hq, Nq, D = qd.shape
    Hkv, Nkv = kd.shape[1], kd.shape[2]
    stream = torch.cuda.current_stream(DEV).cuda_stream or None
    st = lib.ffpa_bwd_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                              dod.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), pkg.FFPA_BF16, B, Hq, Hkv, Nq, Nkv, D, _strides(qd),
                              _strides(kd), _strides(vd), _strides(o), _strides(dod),
                              _strides(dq), _strides(dk), _strides(dv), None, pkg.FFPA_MASK_NONE,
                              None, None, int(causal), int(gqa), stream)
    assert st == pkg.FFPA_OK, pkg.ffpa_status_string(st)
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_backward_matches_ffpa_bwd_on_calls_in_a_row():
    """Consecutive calls share the library's scratch array: a larger causal
    grouped-query problem, then a smaller one (which finds the first call's
    values in the array), then the first again; each matches ffpa_bwd."""
    lib = pkg.load_library()
    first = _prepare(1, 4, 2, 300, 300, 256, seed=71, causal=True)     # 1200 scratch rows
    second = _prepare(2, 2, 2, 200, 333, 512, seed=72, causal=False)   # 800 scratch rows
    for n, (args, ref) in enumerate((first, second, first)):
        got = _noalloc(lib, *args)
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            _close(a, b, f"call {n}: {name}")
    assert pkg.ffpa_last_device_error() == pkg.FFPA_OK


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    """B*Hq*Nq above the fixed array is refused before anything is enqueued
    (checked first, so the pointers are never looked at)."""
    lib = pkg.load_library()
    fake = 0x7F0000000000
    s = (ctypes.c_int64 * 4)(0, 0, 64, 1)
    rows = pkg.BWD_NOALLOC_MAX_ROWS
    for B, Hq, Nq in ((1, 1, rows + 1), (2, 16, rows // 32 + 1)):
        st = lib.ffpa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  pkg.FFPA_BF16, B, Hq, Hq, Nq, 128, 64, s, s, s, s, s, s, s, s,
                                  None, 0, None, None, 0, 0, None)
        assert st == pkg.FFPA_ERR_INVALID
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    big = q.expand(1, rows // 8 + 1, 8, 64)
    lse = torch.zeros(1, rows // 8 + 1, 8)
    with pytest.raises(ValueError, match="scratch"):
        pkg.ffpa_bwd_noalloc(big, big, big, big, big, lse, big, big, big)
