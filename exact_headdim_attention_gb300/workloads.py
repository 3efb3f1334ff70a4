"""Seeded synthetic inputs shaped like the FFPA pages' workloads.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic, so both the CUDA path's tests and the float64
oracle can take their inputs from it.

Recipe (every tensor is drawn on the CPU from ``torch.Generator(seed)``):

* Q, K, V are drawn in that order as float32 ``randn * std`` and rounded
  to bf16 (or fp16) on the CPU; the same bytes are copied to the GPU, so the
  oracle and the kernel read identical values.
* An additive mask is drawn after V: float32 ``U(-2, 0)``, then each entry is
  set to ``-inf`` with probability 0.1 (Bernoulli); a row that would be
  fully ``-inf`` gets its first key redrawn from ``U(-2, 0)``.
* Varlen lengths are drawn first (before Q), uniformly from
  ``[lo, hi]`` inclusive; ``cu_seqlens = [0, cumsum(lengths)]`` (int32).

The named workloads follow the pages' problem statement (FFPA API
reference, ``ffpa_attn_func`` and ``ffpa_attn_varlen_func``) and the self
attention example of the README's "Quick Start" ([B, H, N, D] with large D).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEADDIM_SWEEP = (64, 128, 256, 320, 512, 768, 1024)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    D: int
    seed: int
    causal: bool = False
    std: float = 1.0
    additive_mask: bool = False
    varlen: bool = False
    nseq: int = 0
    len_lo: int = 0
    len_hi: int = 0
    return_lse: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def enable_gqa(self) -> bool:
        return self.Hq != self.Hkv


def tiny_d320() -> Workload:
    """B=1, Hq=Hkv=1, Nq=Nkv=128, D=320, N(0,1), LSE returned."""
    return Workload("tiny_d320", 1, 1, 1, 128, 128, 320, seed=1001, return_lse=True)


def headdim_sweep(D: int) -> Workload:
    """B=1, Hq=Hkv=16, Nq=Nkv=4096, N(0,1), non-causal, no mask."""
    assert D in HEADDIM_SWEEP
    return Workload(f"selfattn_b1_h16_n4096_d{D}", 1, 16, 16, 4096, 4096, D, seed=1002 + D)


def gqa_causal() -> Workload:
    """B=2, Hq=32, Hkv=8, Nq=Nkv=8192, D=512, causal (tail aligned)."""
    return Workload("gqa_causal_b2_hq32_hkv8_n8192_d512", 2, 32, 8, 8192, 8192, 512, seed=1003,
                    causal=True)


def cross_additive_mask() -> Workload:
    """B=4, H=8, Nq=1024, Nkv=4096, D=1024, N(0, 0.5^2), fp32 mask [B,1,Nq,Nkv]."""
    return Workload("cross_mask_b4_h8_nq1024_nkv4096_d1024", 4, 8, 8, 1024, 4096, 1024, seed=1004,
                    std=0.5, additive_mask=True)


def varlen_causal() -> Workload:
    """8 packed sequences, lengths U[512, 4096], Hq=16, Hkv=4, D=512, causal, LSE."""
    return Workload("varlen_causal_8seq_hq16_hkv4_d512", 1, 16, 4, 0, 0, 512, seed=1005,
                    causal=True, varlen=True, nseq=8, len_lo=512, len_hi=4096, return_lse=True)


def all_workloads() -> list[Workload]:
    return [tiny_d320()] + [headdim_sweep(d) for d in HEADDIM_SWEEP] + [
        gqa_causal(), cross_additive_mask(), varlen_causal()]


def useful_flops(w: Workload, seqlens: list[int] | None = None) -> float:
    """The pages' TFLOPS convention: 4*B*Hq*Nq*Nkv*D, halved for causal.

    For varlen each sequence contributes 4*Hq*L^2*D (halved when causal)."""
    if w.varlen:
        assert seqlens is not None
        f = sum(4.0 * w.Hq * L * L * w.D for L in seqlens)
    else:
        f = 4.0 * w.B * w.Hq * w.Nq * w.Nkv * w.D
    return f / 2 if w.causal else f


def _randn(g: torch.Generator, shape, std: float, dtype) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def draw_dense(B, Hq, Hkv, Nq, Nkv, D, seed, std=1.0, dtype=torch.bfloat16):
    """Q [B,Hq,Nq,D], K and V [B,Hkv,Nkv,D], contiguous CPU tensors."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (B, Hq, Nq, D), std, dtype)
    k = _randn(g, (B, Hkv, Nkv, D), std, dtype)
    v = _randn(g, (B, Hkv, Nkv, D), std, dtype)
    return q, k, v, g


def draw_additive_mask(g: torch.Generator, B, Nq, Nkv, p_neg_inf=0.1) -> torch.Tensor:
    """float32 [B,1,Nq,Nkv] ~ U(-2,0) with a fraction p_neg_inf set to -inf."""
    m = torch.rand(B, 1, Nq, Nkv, generator=g, dtype=torch.float32).mul_(-2.0)
    drop = torch.rand(B, 1, Nq, Nkv, generator=g, dtype=torch.float32) < p_neg_inf
    m.masked_fill_(drop, -math.inf)
    full = torch.isinf(m).all(dim=-1)
    if bool(full.any()):
        redraw = torch.rand(int(full.sum()), generator=g, dtype=torch.float32).mul_(-2.0)
        m[..., 0][full] = redraw
    return m


def draw_seqlens(seed, nseq, lo, hi) -> list[int]:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (nseq,), generator=g)]


def cu_seqlens(lengths: list[int]) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    return torch.tensor(cu, dtype=torch.int32)


def draw_varlen(lengths_q, lengths_k, Hq, Hkv, D, seed, std=1.0, dtype=torch.bfloat16):
    """Packed q [Tq,Hq,D], k and v [Tk,Hkv,D] plus int32 cu_seqlens."""
    g = torch.Generator().manual_seed(seed)
    Tq, Tk = sum(lengths_q), sum(lengths_k)
    q = _randn(g, (Tq, Hq, D), std, dtype)
    k = _randn(g, (Tk, Hkv, D), std, dtype)
    v = _randn(g, (Tk, Hkv, D), std, dtype)
    return q, k, v, cu_seqlens(lengths_q), cu_seqlens(lengths_k)


def materialize(w: Workload, dtype=torch.bfloat16) -> dict:
    """All inputs of a named workload as CPU tensors (dict)."""
    if w.varlen:
        lens = draw_seqlens(w.seed, w.nseq, w.len_lo, w.len_hi)
        q, k, v, cq, ck = draw_varlen(lens, lens, w.Hq, w.Hkv, w.D, w.seed + 1, w.std, dtype)
        return dict(q=q, k=k, v=v, cu_q=cq, cu_k=ck, seqlens=lens, max_q=max(lens), max_k=max(lens))
    q, k, v, g = draw_dense(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.seed, w.std, dtype)
    out = dict(q=q, k=k, v=v, mask=None)
    if w.additive_mask:
        out["mask"] = draw_additive_mask(g, w.B, w.Nq, w.Nkv)
    return out
