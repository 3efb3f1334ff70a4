"""Float64 CPU oracle for exact attention (forward and backward) -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or executes anything here.

The arithmetic lives in ``ffpa_oracle.c`` (plain C, double precision,
OpenMP over rows); this file compiles it with gcc and marshals torch CPU
tensors through ctypes.  The definition it follows is the FFPA API
reference ("ffpa_attn.ffpa_attn_func" and "ffpa_attn.ffpa_attn_varlen_func"):
O = softmax(scale * Q K^T + mask) V, scale defaulting to 1/sqrt(D), grouped
query heads, tail-aligned causal masking, and a natural-log LSE.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from pathlib import Path

import torch

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "ffpa_oracle.c"
_LIB_PATH = _HERE / "_build" / "libffpa_oracle.so"

BF16, FP16 = 0, 1
MASK_NONE, MASK_BOOL, MASK_F32, MASK_QTYPE = 0, 1, 2, 3


def compile_oracle(src: Path = _SRC, out: Path = _LIB_PATH, defines=()) -> Path:
    """gcc -O2 -fopenmp -shared; returns the path of the shared object."""
    out.parent.mkdir(parents=True, exist_ok=True)
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", str(src), "-o", str(out), "-lm"]
    cmd += [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    return out


def build() -> Path:
    return compile_oracle()


class Oracle:
    """ctypes view of one compiled oracle shared object."""

    def __init__(self, path: Path | str | None = None):
        path = Path(path) if path else _LIB_PATH
        if path == _LIB_PATH and (not path.exists() or path.stat().st_mtime < _SRC.stat().st_mtime):
            compile_oracle()
        self.lib = ctypes.CDLL(str(path))
        P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        self.lib.oracle_attn_dense.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P, P, I, P, D, I, P, L,
                                               P, P, I]
        self.lib.oracle_attn_dense.restype = I
        self.lib.oracle_attn_varlen.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, I, D, I, P, P, I]
        self.lib.oracle_attn_varlen.restype = I
        self.lib.oracle_attn_bwd_dense.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P, I, P,
                                                   D, I, P, P, P, I]
        self.lib.oracle_attn_bwd_dense.restype = I
        self.lib.oracle_attn_bwd_rows.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, D, I,
                                                  P, L, P, L, P, P, P, I]
        self.lib.oracle_attn_bwd_rows.restype = I
        self.lib.oracle_attn_bwd_varlen.argtypes = [P, P, P, P, I, I, I, I, P, P, P, P, P, P, I, D, I,
                                                    P, P, P, I]
        self.lib.oracle_attn_bwd_varlen.restype = I
        self.lib.oracle_e4m3_encode.argtypes = [P, L, P]
        self.lib.oracle_e4m3_encode.restype = I
        self.lib.oracle_fp8_quantize.argtypes = [P, I, I, I, I, I, P, P, P]
        self.lib.oracle_fp8_quantize.restype = I
        self.lib.oracle_attn_fp8.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P, P, I, P, D, I, P, L,
                                             P, P, I]
        self.lib.oracle_attn_fp8.restype = I

    # ------------------------------------------------------------------ dense
    def attn_dense(self, q, k, v, attn_mask=None, scale=None, is_causal=False, rows=None,
                   nthreads: int = 0):
        """q [B,Hq,Nq,D], k/v [B,Hkv,Nkv,D] (bf16/fp16 CPU tensors, D stride 1).

        attn_mask: None, bool (True keeps), float32 or q-dtype additive,
        broadcastable to [B,Hq,Nq,Nkv].  rows: optional int64 tensor of flat
        row ids (b*Hq+hq)*Nq+i.  Returns (O float64, LSE float64)."""
        return self._attn_dense_like(self.lib.oracle_attn_dense, q, k, v, attn_mask, scale,
                                     is_causal, rows, nthreads)

    def _attn_dense_like(self, fn, q, k, v, attn_mask, scale, is_causal, rows, nthreads):
        dtype = _dtype_code(q)
        assert k.dtype == q.dtype and v.dtype == q.dtype
        B, Hq, Nq, D = q.shape
        _, Hkv, Nkv, _ = k.shape
        for t in (q, k, v):
            assert t.device.type == "cpu" and t.stride(-1) == 1
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        mk, mptr, mstr, keep = MASK_NONE, None, (ctypes.c_int64 * 4)(0, 0, 0, 0), None
        if attn_mask is not None:
            m = attn_mask
            while m.dim() < 4:
                m = m.unsqueeze(0)
            m = m.expand(B, Hq, Nq, Nkv)
            if m.dtype == torch.bool:
                mk = MASK_BOOL
            elif m.dtype == torch.float32:
                mk = MASK_F32
            elif m.dtype == q.dtype:
                mk = MASK_QTYPE
            else:
                raise TypeError(f"mask dtype {m.dtype} not supported")
            keep = m
            mptr = m.data_ptr()
            mstr = (ctypes.c_int64 * 4)(*m.stride())
        if rows is None:
            nrows = B * Hq * Nq
            rows_t = None
        else:
            rows_t = torch.as_tensor(rows, dtype=torch.int64).contiguous()
            nrows = rows_t.numel()
        o = torch.empty(nrows, D, dtype=torch.float64)
        lse = torch.empty(nrows, dtype=torch.float64)
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), dtype, B, Hq, Hkv, Nq, Nkv, D,
                _strides(q), _strides(k), _strides(v), mptr, mk, mstr, float(scale),
                int(bool(is_causal)), None if rows_t is None else rows_t.data_ptr(), nrows,
                o.data_ptr(), lse.data_ptr(), nthreads)
        del keep
        if rc != 0:
            raise ValueError("the oracle rejected its arguments")
        if rows is None:
            return o.view(B, Hq, Nq, D), lse.view(B, Hq, Nq)
        return o, lse

    def attn_varlen(self, q, k, v, cu_q, cu_k=None, scale=None, causal=False, nthreads: int = 0):
        """Packed q [Tq,Hq,D], k/v [Tk,Hkv,D]; cu_* int32 [nseq+1].

        Returns (O float64 [Tq,Hq,D], LSE float64 [Hq,Tq])."""
        dtype = _dtype_code(q)
        Tq, Hq, D = q.shape
        _, Hkv, _ = k.shape
        cu_q = cu_q.to(torch.int32).contiguous()
        cu_k = cu_q if cu_k is None else cu_k.to(torch.int32).contiguous()
        nseq = cu_q.numel() - 1
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        o = torch.empty(Tq, Hq, D, dtype=torch.float64)
        lse = torch.empty(Hq, Tq, dtype=torch.float64)
        rc = self.lib.oracle_attn_varlen(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), dtype, Hq, Hkv, D,
            _strides(q), _strides(k), _strides(v), cu_q.data_ptr(), cu_k.data_ptr(), nseq,
            float(scale), int(bool(causal)), o.data_ptr(), lse.data_ptr(), nthreads)
        if rc != 0:
            raise ValueError("oracle_attn_varlen rejected its arguments")
        return o, lse


    # --------------------------------------------------------------- backward
    def attn_bwd_dense(self, q, k, v, dout, attn_mask=None, scale=None, is_causal=False,
                       nthreads: int = 0):
        """Gradients (dQ, dK, dV) in float64 of sum(O * dout) for the dense forward.

        q, dout [B,Hq,Nq,D]; k, v [B,Hkv,Nkv,D]; same dtypes and mask rules as
        attn_dense.  Returns dq [B,Hq,Nq,D], dk and dv [B,Hkv,Nkv,D]."""
        dtype = _dtype_code(q)
        assert k.dtype == q.dtype and v.dtype == q.dtype and dout.dtype == q.dtype
        B, Hq, Nq, D = q.shape
        _, Hkv, Nkv, _ = k.shape
        assert dout.shape == q.shape
        for t in (q, k, v, dout):
            assert t.device.type == "cpu" and t.stride(-1) == 1
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        mk, mptr, mstr, keep = _mask_args(attn_mask, q, B, Hq, Nq, Nkv)
        dq = torch.empty(B, Hq, Nq, D, dtype=torch.float64)
        dk = torch.empty(B, Hkv, Nkv, D, dtype=torch.float64)
        dv = torch.empty(B, Hkv, Nkv, D, dtype=torch.float64)
        rc = self.lib.oracle_attn_bwd_dense(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), dtype, B, Hq, Hkv, Nq, Nkv, D,
            _strides(q), _strides(k), _strides(v), _strides(dout), mptr, mk, mstr, float(scale),
            int(bool(is_causal)), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), nthreads)
        del keep
        if rc != 0:
            raise ValueError("oracle_attn_bwd_dense rejected its arguments")
        return dq, dk, dv

    def attn_bwd_rows(self, q, k, v, dout, q_rows, k_rows, scale=None, is_causal=False,
                      nthreads: int = 0):
        """Selected gradient rows (no mask): q_rows are flat ids (b*Hq+hq)*Nq+i of
        dQ rows, k_rows flat ids (b*Hkv+hk)*Nkv+j of dK/dV rows.  Returns
        (dq [len(q_rows),D], dk [len(k_rows),D], dv [len(k_rows),D]) in float64."""
        dtype = _dtype_code(q)
        B, Hq, Nq, D = q.shape
        _, Hkv, Nkv, _ = k.shape
        for t in (q, k, v, dout):
            assert t.device.type == "cpu" and t.stride(-1) == 1
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        qr = torch.as_tensor(q_rows, dtype=torch.int64).contiguous()
        kr = torch.as_tensor(k_rows, dtype=torch.int64).contiguous()
        dq = torch.empty(qr.numel(), D, dtype=torch.float64)
        dk = torch.empty(kr.numel(), D, dtype=torch.float64)
        dv = torch.empty(kr.numel(), D, dtype=torch.float64)
        rc = self.lib.oracle_attn_bwd_rows(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), dtype, B, Hq, Hkv, Nq, Nkv, D,
            _strides(q), _strides(k), _strides(v), _strides(dout), float(scale), int(bool(is_causal)),
            qr.data_ptr(), qr.numel(), kr.data_ptr(), kr.numel(), dq.data_ptr(), dk.data_ptr(),
            dv.data_ptr(), nthreads)
        if rc != 0:
            raise ValueError("oracle_attn_bwd_rows rejected its arguments")
        return dq, dk, dv

    def attn_bwd_varlen(self, q, k, v, dout, cu_q, cu_k=None, scale=None, causal=False,
                        nthreads: int = 0):
        """Gradients (dQ [Tq,Hq,D], dK, dV [Tk,Hkv,D], float64) of sum(O * dout) for
        the packed variable-length forward."""
        dtype = _dtype_code(q)
        Tq, Hq, D = q.shape
        Tk, Hkv, _ = k.shape
        for t in (q, k, v, dout):
            assert t.device.type == "cpu" and t.stride(-1) == 1
        cu_q = cu_q.to(torch.int32).contiguous()
        cu_k = cu_q if cu_k is None else cu_k.to(torch.int32).contiguous()
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        dq = torch.empty(Tq, Hq, D, dtype=torch.float64)
        dk = torch.empty(Tk, Hkv, D, dtype=torch.float64)
        dv = torch.empty(Tk, Hkv, D, dtype=torch.float64)
        rc = self.lib.oracle_attn_bwd_varlen(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), dtype, Hq, Hkv, D,
            _strides(q), _strides(k), _strides(v), _strides(dout), cu_q.data_ptr(), cu_k.data_ptr(),
            cu_q.numel() - 1, float(scale), int(bool(causal)), dq.data_ptr(), dk.data_ptr(),
            dv.data_ptr(), nthreads)
        if rc != 0:
            raise ValueError("oracle_attn_bwd_varlen rejected its arguments")
        return dq, dk, dv


def _fp8_methods():
    """FP8 forward reference (see the FP8 section of ffpa_oracle.c)."""

    def e4m3_encode(self, x: torch.Tensor) -> torch.Tensor:
        """uint8 e4m3 codes of float32 values (clamped to [-448, 448]), nearest-even."""
        x = x.detach().to(torch.float32).contiguous().reshape(-1)
        out = torch.empty(x.numel(), dtype=torch.uint8)
        if self.lib.oracle_e4m3_encode(x.data_ptr(), x.numel(), out.data_ptr()) != 0:
            raise ValueError("NaN given to the e4m3 encoder")
        return out

    def fp8_quantize(self, x: torch.Tensor):
        """codes uint8 [B,H,Npad,D] and scales float32 [B,H,Npad/128] of a bf16/fp16 [B,H,N,D]."""
        B, H, N, D = x.shape
        nblk = (N + 127) // 128
        codes = torch.empty(B, H, nblk * 128, D, dtype=torch.uint8)
        scales = torch.empty(B, H, nblk, dtype=torch.float32)
        rc = self.lib.oracle_fp8_quantize(x.data_ptr(), _dtype_code(x), B, H, N, D, _strides(x),
                                          codes.data_ptr(), scales.data_ptr())
        if rc != 0:
            raise ValueError("oracle_fp8_quantize rejected its arguments")
        return codes, scales

    def attn_fp8(self, q, k, v, attn_mask=None, scale=None, is_causal=False, rows=None,
                 nthreads: int = 0):
        """Exact attention (float64) on the per-block e4m3 quantised Q, K, V; arguments
        and results as attn_dense."""
        return self._attn_dense_like(self.lib.oracle_attn_fp8, q, k, v, attn_mask, scale,
                                     is_causal, rows, nthreads)

    return e4m3_encode, fp8_quantize, attn_fp8


Oracle.e4m3_encode, Oracle.fp8_quantize, Oracle.attn_fp8 = _fp8_methods()


def _mask_args(attn_mask, q, B, Hq, Nq, Nkv):
    """(kind, pointer, strides, keep-alive) of a mask broadcast to [B,Hq,Nq,Nkv]."""
    if attn_mask is None:
        return MASK_NONE, None, (ctypes.c_int64 * 4)(0, 0, 0, 0), None
    m = attn_mask
    while m.dim() < 4:
        m = m.unsqueeze(0)
    m = m.expand(B, Hq, Nq, Nkv)
    if m.dtype == torch.bool:
        mk = MASK_BOOL
    elif m.dtype == torch.float32:
        mk = MASK_F32
    elif m.dtype == q.dtype:
        mk = MASK_QTYPE
    else:
        raise TypeError(f"mask dtype {m.dtype} not supported")
    return mk, m.data_ptr(), (ctypes.c_int64 * 4)(*m.stride()), m


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    raise TypeError(f"oracle takes bf16/fp16 inputs, got {t.dtype}")


def _strides(t: torch.Tensor):
    return (ctypes.c_int64 * t.dim())(*t.stride())


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def attn_dense(*a, **kw):
    return default().attn_dense(*a, **kw)


def attn_varlen(*a, **kw):
    return default().attn_varlen(*a, **kw)


def attn_bwd_dense(*a, **kw):
    return default().attn_bwd_dense(*a, **kw)


def attn_bwd_rows(*a, **kw):
    return default().attn_bwd_rows(*a, **kw)


def attn_bwd_varlen(*a, **kw):
    return default().attn_bwd_varlen(*a, **kw)


def host_threads() -> int:
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)
