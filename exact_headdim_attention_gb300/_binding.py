"""ctypes binding of libffpa (include/ffpa.h): argument marshalling only.

Every step of the attention computation runs in the CUDA kernels behind
the C ABI.  This module turns torch tensors into device pointers, element
strides and sizes, allocates outputs with torch when the caller gives none,
and maps status codes to the exception classes of the FFPA API reference
("Raises": TypeError / ValueError / NotImplementedError).  There is no
fallback: a missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path

import torch

from . import build as _build

FFPA_OK, FFPA_ERR_DTYPE, FFPA_ERR_INVALID, FFPA_ERR_UNSUPPORTED, FFPA_ERR_CUDA, \
    FFPA_ERR_DEVICE_TIMEOUT = range(6)
FFPA_BF16, FFPA_FP16 = 0, 1
FFPA_MASK_NONE, FFPA_MASK_BOOL, FFPA_MASK_ADD_F32, FFPA_MASK_ADD_QTYPE = range(4)

EXPORTED = ("ffpa_fwd", "ffpa_fwd_ex", "ffpa_fwd_varlen", "ffpa_fwd_varlen_ex", "ffpa_bwd",
            "ffpa_bwd_ex", "ffpa_bwd_varlen", "ffpa_bwd_varlen_ex", "ffpa_status_string",
            "ffpa_last_device_error", "ffpa_selected_kernel", "ffpa_bwd_noalloc",
            "ffpa_fwd_fp8", "ffpa_fwd_fp8_ex", "ffpa_fwd_fp8_workspace_bytes", "ffpa_bwd_ws",
            "ffpa_bwd_ws_ex", "ffpa_bwd_workspace_bytes", "ffpa_bwd_varlen_ws", "ffpa_bwd_varlen_ws_ex",
            "ffpa_bwd_varlen_workspace_bytes")

KERNEL_VARIANTS = {"auto": 0, "single": 1, "pair": 2, "split": 3, "dual": 4}

_lib = None


class Options(ctypes.Structure):
    """ffpa_options of include/ffpa.h (one call's status word, wait limit, kernel, test hook)."""
    _fields_ = [("status", ctypes.c_void_p), ("wait_timeout_ns", ctypes.c_uint64),
                ("kernel", ctypes.c_int), ("test_drop_first_copy", ctypes.c_int)]


class FFPAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class FFPATypeError(TypeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class FFPAValueError(ValueError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class FFPANotImplementedError(NotImplementedError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def lib_path() -> Path:
    return _build.OUT


def load_library(path: str | Path | None = None) -> ctypes.CDLL:
    """Load libffpa.so; raises RuntimeError when it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else lib_path()
    if not p.exists():
        raise RuntimeError(
            f"libffpa.so not found at {p}: build it with "
            "`python -m exact_headdim_attention_gb300.build` (no fallback path exists)")
    lib = ctypes.CDLL(str(p))
    P, I = ctypes.c_void_p, ctypes.c_int
    O = ctypes.POINTER(Options)
    sigs = {
        "ffpa_fwd": [P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P, I, P, P, I, I, P],
        "ffpa_fwd_varlen": [P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, I, I, I, P, I, I, P],
        "ffpa_bwd": [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, I,
                     P, P, I, I, P],
        "ffpa_bwd_varlen": [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P,
                            P, I, I, I, P, I, I, P],
    }
    for name, args in sigs.items():
        getattr(lib, name).argtypes = args
        getattr(lib, name).restype = I
        getattr(lib, name + "_ex").argtypes = args + [O]
        getattr(lib, name + "_ex").restype = I
    fp8 = sigs["ffpa_fwd"][:-1] + [P, ctypes.c_size_t, P]   # + workspace, bytes, stream
    lib.ffpa_fwd_fp8.argtypes = fp8
    lib.ffpa_fwd_fp8.restype = I
    lib.ffpa_fwd_fp8_ex.argtypes = fp8 + [O]
    lib.ffpa_fwd_fp8_ex.restype = I
    lib.ffpa_fwd_fp8_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.ffpa_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
    bws = sigs["ffpa_bwd"][:-1] + [P, ctypes.c_size_t, P]   # + workspace, bytes, stream
    lib.ffpa_bwd_ws.argtypes = bws
    lib.ffpa_bwd_ws.restype = I
    lib.ffpa_bwd_ws_ex.argtypes = bws + [O]
    lib.ffpa_bwd_ws_ex.restype = I
    lib.ffpa_bwd_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.ffpa_bwd_workspace_bytes.restype = ctypes.c_size_t
    bvws = sigs["ffpa_bwd_varlen"][:-1] + [P, ctypes.c_size_t, P]   # + workspace, bytes, stream
    lib.ffpa_bwd_varlen_ws.argtypes = bvws
    lib.ffpa_bwd_varlen_ws.restype = I
    lib.ffpa_bwd_varlen_ws_ex.argtypes = bvws + [O]
    lib.ffpa_bwd_varlen_ws_ex.restype = I
    lib.ffpa_bwd_varlen_workspace_bytes.argtypes = [P, P, I, I, I, I, I]
    lib.ffpa_bwd_varlen_workspace_bytes.restype = ctypes.c_size_t
    # ffpa_bwd without the delta argument
    lib.ffpa_bwd_noalloc.argtypes = sigs["ffpa_bwd"][:9] + sigs["ffpa_bwd"][10:]
    lib.ffpa_bwd_noalloc.restype = I
    lib.ffpa_status_string.argtypes = [I]
    lib.ffpa_status_string.restype = ctypes.c_char_p
    lib.ffpa_last_device_error.argtypes = [P]
    lib.ffpa_last_device_error.restype = I
    lib.ffpa_selected_kernel.argtypes = [I, I, I]
    lib.ffpa_selected_kernel.restype = I
    if path is None:
        _lib = lib
    return lib


def ffpa_status_string(status: int) -> str:
    return load_library().ffpa_status_string(status).decode()


def _raise(status: int, what: str):
    msg = f"{what}: {ffpa_status_string(status)}"
    if status == FFPA_ERR_DTYPE:
        raise FFPATypeError(status, msg)
    if status == FFPA_ERR_INVALID:
        raise FFPAValueError(status, msg)
    if status == FFPA_ERR_UNSUPPORTED:
        raise FFPANotImplementedError(status, msg)
    raise FFPAError(status, msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FFPA_BF16
    if t.dtype == torch.float16:
        return FFPA_FP16
    return -1


def _strides(t: torch.Tensor):
    return (ctypes.c_int64 * t.dim())(*t.stride())


def _stream_handle(stream, t: torch.Tensor | None = None) -> int | None:
    """cudaStream_t of `stream`, else of torch's current stream on t's device."""
    if stream is None:
        if t is not None and not t.is_cuda:
            return None          # host tensors never reach a launch (the ABI rejects them)
        stream = torch.cuda.current_stream(None if t is None else t.device)
    return stream.cuda_stream or None


def _options(q: torch.Tensor, kernel, status, wait_timeout_ns, test_drop_first_copy):
    """ctypes ffpa_options for one call, or None when every field is the default."""
    if kernel is None and status is None and not wait_timeout_ns and not test_drop_first_copy:
        return None
    if kernel is not None and kernel not in KERNEL_VARIANTS:
        raise ValueError(f"kernel must be one of {sorted(KERNEL_VARIANTS)}, got {kernel!r}")
    if status is not None:
        if (status.dtype != torch.int32 or status.numel() != 1 or status.device != q.device):
            raise ValueError("status must be a one-element int32 tensor on q's device")
    return ctypes.byref(Options(None if status is None else status.data_ptr(),
                                int(wait_timeout_ns or 0), KERNEL_VARIANTS[kernel or "auto"],
                                int(bool(test_drop_first_copy))))


def _check_buffer(t, name, shape, dtype, device, contiguous=False):
    """A caller-supplied output: its shape, dtype and device must be those the
    library writes (it sizes every write from q and k)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dim() != len(shape) or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _device_copy(cu: torch.Tensor, device, stream):
    """cu_seqlens on the launch device, copied on the launch stream so that the
    copy is ordered before the kernel and its memory is not reused (by torch's
    caching allocator) while the kernel may still read it."""
    if stream is None or not isinstance(stream, torch.cuda.Stream):
        return cu.to(device)
    with torch.cuda.stream(stream):
        d = cu.to(device)
    if d is not cu:
        d.record_stream(stream)
    return d


_REJECTED = ("window_size", "softcap", "sink", "attention_mask", "block_mask", "score_mod",
             "aux_tensors", "seqused_k", "block_table", "num_splits", "alibi_slopes")


def ffpa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, attn_mask=None,
             dropout_p: float = 0.0, is_causal: bool = False, scale: float | None = None,
             enable_gqa: bool = False, *, return_lse: bool = False, out=None, lse=None,
             stream=None, kernel=None, status=None, wait_timeout_ns=None,
             test_drop_first_copy=False, **kwargs):
    """Dense attention forward through the C ABI ``ffpa_fwd_ex``.

    q [B,Hq,Nq,D], k/v [B,Hkv,Nkv,D] (bf16 or fp16, CUDA, D stride 1);
    attn_mask broadcastable to [B,Hq,Nq,Nkv] (bool: True participates;
    float32 or the q dtype: additive).  Returns O [B,Hq,Nq,D], or (O, LSE
    [B,Hq,Nq] fp32) with return_lse.  Follows the FFPA API reference,
    ``ffpa_attn.ffpa_attn_func``.

    Per-call options (ffpa_options): kernel ("auto", "single", "pair",
    "split", "dual"), status (a one-element int32 device tensor that receives
    FFPA_ERR_DEVICE_TIMEOUT if a wait of this call runs out; the caller
    zeroes it), wait_timeout_ns, and the test hook test_drop_first_copy."""
    if kwargs:
        raise TypeError(f"unexpected keyword arguments: {sorted(kwargs)}")
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported by this forward kernel")
    lib = load_library()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, D]")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    B, Hq, Nq, D = q.shape
    Bk, Hkv, Nkv, Dk = k.shape
    if tuple(v.shape) != (Bk, Hkv, Nkv, Dk) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    else:
        _check_buffer(out, "out", q.shape, q.dtype, q.device)
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_buffer(lse, "lse", (B, Hq, Nq), torch.float32, q.device, contiguous=True)
    mk, mptr, mstr, keep = _mask_args(attn_mask, q, B, Hq, Nq, Nkv)
    sc = None if scale is None else ctypes.byref(ctypes.c_float(float(scale)))
    opts = _options(q, kernel, status, wait_timeout_ns, test_drop_first_copy)
    st = lib.ffpa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         None if lse is None else lse.data_ptr(), _dtype_code(q),
                         B, Hq, Hkv, Nq, Nkv, D, _strides(q), _strides(k), _strides(v), _strides(out),
                         mptr, mk, mstr, sc, int(bool(is_causal)), int(bool(enable_gqa)),
                         _stream_handle(stream, q), opts)
    del keep
    if st != FFPA_OK:
        _raise(st, "ffpa_fwd")
    return (out, lse) if return_lse else out


def fp8_workspace_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int) -> int:
    """Bytes of the workspace ffpa_fwd_fp8 needs (0 for an unsupported shape)."""
    return int(load_library().ffpa_fwd_fp8_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D))


def fp8_workspace_views(ws: torch.Tensor, B, Hq, Hkv, Nq, Nkv, D):
    """Views of a uint8 workspace as the layout include/ffpa.h documents for
    ffpa_fwd_fp8: e4m3 codes of Q [B,Hq,Nqp,D], K [B,Hkv,Nkp,D], V transposed
    [B,Hkv,D,Nkp] (uint8) and the fp32 block scales of each."""
    nqb, nkb = (Nq + 127) // 128, (Nkv + 127) // 128
    nqp, nkp = nqb * 128, nkb * 128
    shapes = [((B, Hq, nqp, D), torch.uint8), ((B, Hkv, nkp, D), torch.uint8),
              ((B, Hkv, D, nkp), torch.uint8), ((B, Hq, nqb), torch.float32),
              ((B, Hkv, nkb), torch.float32), ((B, Hkv, nkb), torch.float32)]
    out, at = [], 0
    for shape, dt in shapes:
        n = math.prod(shape) * (4 if dt == torch.float32 else 1)
        out.append(ws[at:at + n].view(dt).view(shape))
        at += (n + 255) // 256 * 256
    return out


def ffpa_fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, attn_mask=None,
                 dropout_p: float = 0.0, is_causal: bool = False, scale: float | None = None,
                 enable_gqa: bool = False, *, return_lse: bool = False, out=None, lse=None,
                 workspace=None, stream=None, kernel=None, status=None, wait_timeout_ns=None,
                 test_drop_first_copy=False):
    """FP8 (e4m3) attention forward through the C ABI ``ffpa_fwd_fp8_ex``.

    Arguments as ffpa_fwd (bf16/fp16 in and out); D a multiple of 128.
    kernel: "single" forces the single-CTA FP8 kernel, "split" the column
    split (D = 256, 384, 512); by default the split runs at D = 384 and 512.
    workspace: a uint8 device tensor of at least fp8_workspace_bytes(...)
    bytes (allocated here when None); after the call it holds the e4m3
    codes and scales (fp8_workspace_views)."""
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported by this forward kernel")
    lib = load_library()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, D]")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    B, Hq, Nq, D = q.shape
    Bk, Hkv, Nkv, Dk = k.shape
    if tuple(v.shape) != (Bk, Hkv, Nkv, Dk) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    else:
        _check_buffer(out, "out", q.shape, q.dtype, q.device)
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_buffer(lse, "lse", (B, Hq, Nq), torch.float32, q.device, contiguous=True)
    need = int(lib.ffpa_fwd_fp8_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    elif workspace.dtype != torch.uint8 or workspace.dim() != 1 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous 1-D uint8 tensor")
    mk, mptr, mstr, keep = _mask_args(attn_mask, q, B, Hq, Nq, Nkv)
    sc = None if scale is None else ctypes.byref(ctypes.c_float(float(scale)))
    opts = _options(q, kernel, status, wait_timeout_ns, test_drop_first_copy)
    st = lib.ffpa_fwd_fp8_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             None if lse is None else lse.data_ptr(), _dtype_code(q),
                             B, Hq, Hkv, Nq, Nkv, D, _strides(q), _strides(k), _strides(v),
                             _strides(out), mptr, mk, mstr, sc, int(bool(is_causal)),
                             int(bool(enable_gqa)), workspace.data_ptr(),
                             workspace.numel(), _stream_handle(stream, q), opts)
    del keep
    if st != FFPA_OK:
        _raise(st, "ffpa_fwd_fp8")
    return (out, lse) if return_lse else out


def _mask_args(attn_mask, q, B, Hq, Nq, Nkv):
    """(kind, pointer, strides, keep-alive) of a mask broadcast to [B,Hq,Nq,Nkv]."""
    if attn_mask is None:
        return FFPA_MASK_NONE, None, None, None
    m = attn_mask
    if m.dim() > 4:
        raise ValueError("attn_mask has more than 4 dimensions")
    while m.dim() < 4:
        m = m.unsqueeze(0)
    try:
        m = m.expand(B, Hq, Nq, Nkv)
    except RuntimeError as e:
        raise ValueError(f"attn_mask {tuple(attn_mask.shape)} does not broadcast to "
                         f"{(B, Hq, Nq, Nkv)}") from e
    if m.device != q.device:
        raise ValueError("attn_mask must be on the same device as q")
    if m.dtype == torch.bool:
        mk = FFPA_MASK_BOOL
    elif m.dtype == torch.float32:
        mk = FFPA_MASK_ADD_F32
    elif m.dtype == q.dtype:
        mk = FFPA_MASK_ADD_QTYPE
    else:
        raise TypeError(f"attn_mask dtype {m.dtype} not supported (bool, float32 or {q.dtype})")
    return mk, m.data_ptr(), _strides(m), m


# Largest stored-tile workspace ffpa_bwd allocates by itself (workspace="auto"):
# at most this many bytes and at most a quarter of the device's free memory.
BWD_AUTO_WORKSPACE_MAX = 32 << 30


def bwd_workspace_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int,
                        is_causal: bool = False) -> int:
    """Bytes of the stored-tile backward's workspace (0: the shape does not take that path)."""
    return int(load_library().ffpa_bwd_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D, int(bool(is_causal))))


def _release_on(ws, workspace, stream):
    """A workspace allocated here is freed when the call returns: on a launch
    stream other than the current one, the caching allocator must not hand its
    memory out again before the kernels on that stream are done with it."""
    if ws is not None and isinstance(workspace, str) and isinstance(stream, torch.cuda.Stream):
        ws.record_stream(stream)


def varlen_bwd_workspace_bytes(cu_q, cu_k, Hq: int, Hkv: int, D: int, causal: bool = False) -> int:
    """Bytes of the varlen stored-tile backward's workspace for these sequences
    (cu_q, cu_k: host sequences of cumulative lengths; 0: the path does not apply)."""
    cq = (ctypes.c_int32 * len(cu_q))(*[int(x) for x in cu_q])
    ck = (ctypes.c_int32 * len(cu_k))(*[int(x) for x in cu_k])
    return int(load_library().ffpa_bwd_varlen_workspace_bytes(cq, ck, len(cu_q) - 1, Hq, Hkv, D,
                                                              int(bool(causal))))


def _bwd_workspace(workspace, need: int, device):
    """(pointer, bytes, tensor to keep) of the stored-tile workspace argument."""
    if workspace is None or need == 0:
        return None, 0, None
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be None, "auto" or a uint8 device tensor')
        if need > BWD_AUTO_WORKSPACE_MAX or need > torch.cuda.mem_get_info(device)[0] // 4:
            return None, 0, None
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if (not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8
            or not workspace.is_contiguous() or workspace.device != device):
        raise ValueError("workspace must be a contiguous uint8 tensor on q's device")
    return workspace.data_ptr(), workspace.numel(), workspace


def ffpa_bwd(dout: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
             out: torch.Tensor, lse: torch.Tensor, is_causal: bool = False,
             scale: float | None = None, enable_gqa: bool = False, attn_mask=None, *, dq=None,
             dk=None, dv=None, delta=None, return_delta: bool = False, workspace="auto",
             stream=None, status=None, wait_timeout_ns=None, test_drop_first_copy=False):
    """Dense attention backward through the C ABI ``ffpa_bwd_ws``.

    dout, q, out [B,Hq,Nq,D]; k, v [B,Hkv,Nkv,D]; lse [B,Hq,Nq] fp32 from the
    forward with the same attn_mask / is_causal / scale (the mask enters the
    recomputed scores; no gradient is formed for it).  Returns (dq, dk, dv),
    plus delta = rowsum(dout * out) [B,Hq,Nq] fp32 with return_delta.

    workspace: the stored-tile backward's scratch (see bwd_workspace_bytes):
    "auto" allocates it when the shape takes that path and it needs at most
    BWD_AUTO_WORKSPACE_MAX bytes and a quarter of the free device memory;
    None runs the slice kernels (S and dP recomputed per 256-column output
    slice); a uint8 device tensor is used when it is large enough."""
    lib = load_library()
    for name, t in (("dout", dout), ("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D [B, H, N, D]")
        if t.dtype != q.dtype:
            raise TypeError("dout, q, k, v and out must share one dtype")
    B, Hq, Nq, D = q.shape
    Bk, Hkv, Nkv, Dk = k.shape
    if (tuple(v.shape) != (Bk, Hkv, Nkv, Dk) or Bk != B or Dk != D
            or tuple(out.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape)):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}, "
                         f"out {tuple(out.shape)}, dout {tuple(dout.shape)}")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse must be a contiguous float32 [B, Hq, Nq] tensor")
    dq, dk, dv, delta = _grad_buffers(q, k, v, dq, dk, dv, delta, (B, Hq, Nq))
    mk, mptr, mstr, keep = _mask_args(attn_mask, q, B, Hq, Nq, Nkv)
    sc = None if scale is None else ctypes.byref(ctypes.c_float(float(scale)))
    opts = _options(q, None, status, wait_timeout_ns, test_drop_first_copy)
    need = int(lib.ffpa_bwd_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D, int(bool(is_causal))))
    ws_ptr, ws_bytes, ws_keep = _bwd_workspace(workspace, need, q.device)
    st = lib.ffpa_bwd_ws_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            delta.data_ptr(), _dtype_code(q), B, Hq, Hkv, Nq, Nkv, D, _strides(q),
                            _strides(k), _strides(v), _strides(out), _strides(dout), _strides(dq),
                            _strides(dk), _strides(dv), mptr, mk, mstr, sc, int(bool(is_causal)),
                            int(bool(enable_gqa)), ws_ptr, ws_bytes, _stream_handle(stream, q), opts)
    _release_on(ws_keep, workspace, stream)
    del keep, ws_keep
    if st != FFPA_OK:
        _raise(st, "ffpa_bwd")
    return (dq, dk, dv, delta) if return_delta else (dq, dk, dv)


def _grad_buffers(q, k, v, dq, dk, dv, delta, delta_shape):
    """The gradient outputs and delta: allocated when not given, else checked."""
    if dq is None:
        dq = torch.empty_like(q, memory_format=torch.contiguous_format)
    else:
        _check_buffer(dq, "dq", q.shape, q.dtype, q.device)
    if dk is None:
        dk = torch.empty_like(k, memory_format=torch.contiguous_format)
    else:
        _check_buffer(dk, "dk", k.shape, k.dtype, q.device)
    if dv is None:
        dv = torch.empty_like(v, memory_format=torch.contiguous_format)
    else:
        _check_buffer(dv, "dv", v.shape, v.dtype, q.device)
    if delta is None:
        delta = torch.empty(delta_shape, dtype=torch.float32, device=q.device)
    else:
        _check_buffer(delta, "delta", delta_shape, torch.float32, q.device, contiguous=True)
    return dq, dk, dv, delta


BWD_NOALLOC_MAX_ROWS = 1048576   # FFPA_BWD_NOALLOC_MAX_ROWS of include/ffpa.h


def ffpa_bwd_noalloc(dout: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                     out: torch.Tensor, lse: torch.Tensor, dq: torch.Tensor, dk: torch.Tensor,
                     dv: torch.Tensor, is_causal: bool = False, scale: float | None = None,
                     enable_gqa: bool = False, attn_mask=None, *, stream=None):
    """Dense backward through the C ABI ``ffpa_bwd_noalloc``, for callers that
    cannot allocate device memory: the per-row scratch of the backward lives in
    a fixed array inside the library (at most BWD_NOALLOC_MAX_ROWS = B*Hq*Nq
    rows), and the caller passes dq, dk and dv.  Nothing is allocated here
    either (a broadcast mask is passed as a strided view).  Calls on one device
    share that array: calls that overlap on the GPU race."""
    lib = load_library()
    B, Hq, Nq, D = q.shape
    Nkv = k.shape[2]
    if B * Hq * Nq > BWD_NOALLOC_MAX_ROWS:
        raise ValueError(f"B*Hq*Nq = {B * Hq * Nq} exceeds the {BWD_NOALLOC_MAX_ROWS} rows of the "
                         "library's fixed backward scratch; use ffpa_bwd with a delta buffer")
    _check_buffer(dq, "dq", q.shape, q.dtype, q.device)
    _check_buffer(dk, "dk", k.shape, k.dtype, q.device)
    _check_buffer(dv, "dv", v.shape, v.dtype, q.device)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse must be a contiguous float32 [B, Hq, Nq] tensor")
    mk, mptr, mstr, keep = _mask_args(attn_mask, q, B, Hq, Nq, Nkv)
    sc = None if scale is None else ctypes.byref(ctypes.c_float(float(scale)))
    st = lib.ffpa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), _dtype_code(q), B, Hq, k.shape[1], Nq, Nkv, D,
                              _strides(q), _strides(k), _strides(v), _strides(out),
                              _strides(dout), _strides(dq), _strides(dk), _strides(dv), mptr, mk,
                              mstr, sc, int(bool(is_causal)), int(bool(enable_gqa)),
                              _stream_handle(stream, q))
    del keep
    if st != FFPA_OK:
        _raise(st, "ffpa_bwd_noalloc")
    return dq, dk, dv


def _check_cu(cu: torch.Tensor, T: int, name: str) -> list[int]:
    if cu.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    if cu.dim() != 1 or cu.numel() < 2:
        raise ValueError(f"{name} must be 1-D with at least 2 entries")
    vals = cu.tolist()
    if vals[0] != 0 or vals[-1] != T or any(b < a for a, b in zip(vals, vals[1:])):
        raise ValueError(f"{name} must start at 0, end at {T} and be non-decreasing")
    return vals


def ffpa_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                    cu_seqlens_k: torch.Tensor | None, max_seqlen_q: int, max_seqlen_k: int, *,
                    dropout_p: float = 0.0, softmax_scale: float | None = None,
                    causal: bool = False, enable_gqa: bool = False, return_lse: bool = False,
                    out=None, lse=None, stream=None, kernel=None, status=None,
                    wait_timeout_ns=None, test_drop_first_copy=False, **kwargs):
    """Packed varlen attention forward through the C ABI ``ffpa_fwd_varlen``.

    q [Tq,Hq,D], k/v [Tk,Hkv,D]; cu_seqlens_* int32 [nseq+1] (cu_seqlens_k
    None reuses cu_seqlens_q).  Returns O [Tq,Hq,D], or (O, LSE [Hq,Tq])
    with return_lse.  Follows the FFPA API reference,
    ``ffpa_attn.ffpa_attn_varlen_func`` (including its rejected options)."""
    for name in _REJECTED:
        if kwargs.get(name) not in (None, False, (-1, -1), 0, 0.0):
            raise NotImplementedError(f"option {name} is not supported")
        kwargs.pop(name, None)
    if kwargs:
        raise TypeError(f"unexpected keyword arguments: {sorted(kwargs)}")
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported")
    lib = load_library()
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    if _dtype_code(q) < 0:
        raise TypeError(f"dtype {q.dtype} not supported (bf16 or fp16)")
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be 3-D [T, H, D]")
    Tq, Hq, D = q.shape
    Tk, Hkv, Dk = k.shape
    if tuple(v.shape) != (Tk, Hkv, Dk) or Dk != D:
        raise ValueError("shape mismatch between q, k and v")
    cq = _check_cu(cu_seqlens_q, Tq, "cu_seqlens_q")
    ck = cq if cu_seqlens_k is None else _check_cu(cu_seqlens_k, Tk, "cu_seqlens_k")
    if len(ck) != len(cq):
        raise ValueError("cu_seqlens_q and cu_seqlens_k describe different batch sizes")
    if cu_seqlens_k is None and Tk != Tq:
        raise ValueError("cu_seqlens_k=None needs Tk == Tq")
    if max(b - a for a, b in zip(cq, cq[1:])) > max_seqlen_q or \
            max(b - a for a, b in zip(ck, ck[1:])) > max_seqlen_k:
        raise ValueError("max_seqlen_* is smaller than a sequence length")
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    else:
        _check_buffer(out, "out", q.shape, q.dtype, q.device)
    if return_lse and lse is None:
        lse = torch.empty(Hq, Tq, dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_buffer(lse, "lse", (Hq, Tq), torch.float32, q.device, contiguous=True)
    cuq = _device_copy(cu_seqlens_q, q.device, stream)
    cuk = None if cu_seqlens_k is None else _device_copy(cu_seqlens_k, q.device, stream)
    sc = None if softmax_scale is None else ctypes.byref(ctypes.c_float(float(softmax_scale)))
    opts = _options(q, kernel, status, wait_timeout_ns, test_drop_first_copy)
    st = lib.ffpa_fwd_varlen_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                None if lse is None else lse.data_ptr(), _dtype_code(q),
                                Tq, Tk, Hq, Hkv, D, _strides(q), _strides(k), _strides(v),
                                _strides(out), cuq.data_ptr(),
                                None if cuk is None else cuk.data_ptr(), len(cq) - 1,
                                int(max_seqlen_q), int(max_seqlen_k), sc, int(bool(causal)),
                                int(bool(enable_gqa)), _stream_handle(stream, q), opts)
    if st != FFPA_OK:
        _raise(st, "ffpa_fwd_varlen")
    return (out, lse) if return_lse else out


def ffpa_bwd_varlen(dout: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    out: torch.Tensor, lse: torch.Tensor, cu_seqlens_q: torch.Tensor,
                    cu_seqlens_k: torch.Tensor | None, max_seqlen_q: int, max_seqlen_k: int, *,
                    softmax_scale: float | None = None, causal: bool = False,
                    enable_gqa: bool = False, dq=None, dk=None, dv=None, delta=None,
                    return_delta: bool = False, workspace="auto", stream=None, status=None,
                    wait_timeout_ns=None, test_drop_first_copy=False):
    """Packed varlen backward through the C ABI ``ffpa_bwd_varlen_ws``.

    dout, q, out [Tq,Hq,D]; k, v [Tk,Hkv,D]; lse [Hq,Tq] fp32 from
    ffpa_fwd_varlen with the same sequences, causal and scale.  Returns
    (dq, dk, dv), plus delta [Hq,Tq] fp32 with return_delta.  workspace: as
    for ffpa_bwd, sized by varlen_bwd_workspace_bytes of these sequences."""
    lib = load_library()
    for name, t in (("dout", dout), ("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dim() != 3:
            raise ValueError(f"{name} must be 3-D [T, H, D]")
        if t.dtype != q.dtype:
            raise TypeError("dout, q, k, v and out must share one dtype")
    Tq, Hq, D = q.shape
    Tk, Hkv, Dk = k.shape
    if (tuple(v.shape) != (Tk, Hkv, Dk) or Dk != D or tuple(out.shape) != tuple(q.shape)
            or tuple(dout.shape) != tuple(q.shape)):
        raise ValueError("shape mismatch between q, k, v, out and dout")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (Hq, Tq):
        raise ValueError("lse must be a contiguous float32 [Hq, Tq] tensor")
    cq = _check_cu(cu_seqlens_q, Tq, "cu_seqlens_q")
    ck = cq if cu_seqlens_k is None else _check_cu(cu_seqlens_k, Tk, "cu_seqlens_k")
    if len(ck) != len(cq):
        raise ValueError("cu_seqlens_q and cu_seqlens_k describe different batch sizes")
    if cu_seqlens_k is None and Tk != Tq:
        raise ValueError("cu_seqlens_k=None needs Tk == Tq")
    if max(b - a for a, b in zip(cq, cq[1:])) > max_seqlen_q or \
            max(b - a for a, b in zip(ck, ck[1:])) > max_seqlen_k:
        raise ValueError("max_seqlen_* is smaller than a sequence length")
    dq, dk, dv, delta = _grad_buffers(q, k, v, dq, dk, dv, delta, (Hq, Tq))
    need = varlen_bwd_workspace_bytes(cq, ck, Hq, Hkv, D, causal)
    ws_ptr, ws_bytes, ws_keep = _bwd_workspace(workspace, need, q.device)
    cuq = _device_copy(cu_seqlens_q, q.device, stream)
    cuk = None if cu_seqlens_k is None else _device_copy(cu_seqlens_k, q.device, stream)
    sc = None if softmax_scale is None else ctypes.byref(ctypes.c_float(float(softmax_scale)))
    opts = _options(q, None, status, wait_timeout_ns, test_drop_first_copy)
    st = lib.ffpa_bwd_varlen_ws_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), delta.data_ptr(), _dtype_code(q), Tq, Tk, Hq, Hkv, D,
                                   _strides(q), _strides(k), _strides(v), _strides(out),
                                   _strides(dout), _strides(dq), _strides(dk), _strides(dv),
                                   cuq.data_ptr(), None if cuk is None else cuk.data_ptr(), len(cq) - 1,
                                   int(max_seqlen_q), int(max_seqlen_k), sc, int(bool(causal)),
                                   int(bool(enable_gqa)), ws_ptr, ws_bytes, _stream_handle(stream, q), opts)
    _release_on(ws_keep, workspace, stream)
    del ws_keep
    if st != FFPA_OK:
        _raise(st, "ffpa_bwd_varlen")
    return (dq, dk, dv, delta) if return_delta else (dq, dk, dv)


def ffpa_last_device_error(stream=None) -> int:
    """Checked mode for calls made without a status word: synchronise the stream and
    return (and clear) the device's shared fallback status word (see ffpa.h)."""
    return load_library().ffpa_last_device_error(_stream_handle(stream))


def selected_kernel(D: int, varlen: bool = False, kernel: str = "auto") -> str:
    """Name of the kernel ("single", "pair", "split" or "dual") a call with `kernel` would use
    for head dim D (an unmasked call: with a caller's mask the dual-tile choice runs the
    single-CTA kernel)."""
    if kernel not in KERNEL_VARIANTS:
        raise ValueError(f"kernel must be one of {sorted(KERNEL_VARIANTS)}, got {kernel!r}")
    v = load_library().ffpa_selected_kernel(int(D), int(bool(varlen)), KERNEL_VARIANTS[kernel])
    if v < 0:
        raise ValueError(f"unsupported head dimension {D}")
    return {code: name for name, code in KERNEL_VARIANTS.items()}[v]


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
