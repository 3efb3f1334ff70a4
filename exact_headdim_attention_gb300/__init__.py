"""Exact scaled-dot-product attention (forward and backward) for large head dimensions on GB300.

The compute path is libffpa.so (hand-written sm_103a CUDA kernels behind the
C ABI in include/ffpa.h); this package only marshals torch tensors into that
ABI.  Build the library with ``python -m exact_headdim_attention_gb300.build``.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    FFPA_BF16,
    FFPA_ERR_CUDA,
    FFPA_ERR_DEVICE_TIMEOUT,
    FFPA_ERR_DTYPE,
    FFPA_ERR_INVALID,
    FFPA_ERR_UNSUPPORTED,
    FFPA_FP16,
    FFPA_MASK_ADD_F32,
    FFPA_MASK_ADD_QTYPE,
    FFPA_MASK_BOOL,
    FFPA_MASK_NONE,
    FFPA_OK,
    FFPAError,
    KERNEL_VARIANTS,
    Options,
    default_scale,
    BWD_AUTO_WORKSPACE_MAX,
    bwd_workspace_bytes,
    varlen_bwd_workspace_bytes,
    ffpa_bwd,
    ffpa_bwd_noalloc,
    BWD_NOALLOC_MAX_ROWS,
    ffpa_bwd_varlen,
    ffpa_fwd,
    ffpa_fwd_fp8,
    fp8_workspace_bytes,
    fp8_workspace_views,
    ffpa_fwd_varlen,
    ffpa_last_device_error,
    ffpa_status_string,
    lib_path,
    load_library,
    selected_kernel,
)
from .torch_ops import ffpa_attn_func, ffpa_attn_varlen_func  # noqa: F401,E402
