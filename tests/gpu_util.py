"""Helpers shared by the GPU parity tests (no attention arithmetic here)."""
from __future__ import annotations

import math

import torch

import exact_headdim_attention_gb300 as pkg

# Tolerances for bf16/fp16 O and fp32 LSE against the float64 oracle on the
# same inputs: max |err| <= 2e-2, mean |err| <= 2e-3, LSE within 1e-3.
O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def check(o, lse, o_ref, lse_ref, what="", o_max=O_MAX, o_mean=O_MEAN, lse_max=LSE_MAX):
    o = o.detach().double().cpu().reshape(o_ref.shape)
    assert torch.isfinite(o).all(), f"{what}: non-finite output"
    err = (o - o_ref).abs()
    mx, mean = err.max().item() if err.numel() else 0.0, err.mean().item() if err.numel() else 0.0
    assert mx <= o_max and mean <= o_mean, f"{what}: O max|err| {mx:.3e} mean {mean:.3e}"
    if lse is not None:
        lse = lse.detach().double().cpu().reshape(lse_ref.shape)
        inf_ref = torch.isinf(lse_ref)
        assert torch.equal(torch.isinf(lse), inf_ref), f"{what}: LSE -inf pattern differs"
        if (~inf_ref).any():
            lerr = (lse[~inf_ref] - lse_ref[~inf_ref]).abs().max().item()
            assert lerr <= lse_max, f"{what}: LSE max|err| {lerr:.3e}"
    return mx, mean


def device_ok():
    torch.cuda.synchronize()
    st = pkg.ffpa_last_device_error()
    assert st == pkg.FFPA_OK, pkg.ffpa_status_string(st)


def sample_rows(B, Hq, Nq, n_random=8, tile=128, heads=None, seed=0):
    """Flat row ids (b*Hq+h)*Nq+i of every (batch, head) pair (or of `heads`):
    the first and last row of every `tile`-row query tile plus `n_random`
    seeded random rows per head, so that every head, every grouped KV head
    and every query tile kind (first, interior, ragged last) is compared."""
    g = torch.Generator().manual_seed(seed)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    rows = []
    for b, h in heads:
        base = (b * Hq + h) * Nq
        idx = {i for t0 in range(0, Nq, tile) for i in (t0, min(Nq, t0 + tile) - 1)}
        idx |= set(torch.randint(0, Nq, (n_random,), generator=g).tolist())
        rows += [base + i for i in sorted(idx)]
    return torch.tensor(rows, dtype=torch.int64)


def gather_rows(t, rows, D):
    return t.reshape(-1, D)[rows.to(t.device)]


def nan_sentinel_(t):
    return t.fill_(float("nan"))


def ln(x):
    return math.log(x)
