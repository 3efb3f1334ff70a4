"""Host-side checks of the C ABI: the library builds, loads and exports every
declared symbol, and every argument check returns the documented status
without touching a GPU (no compute call is made)."""
import ctypes
import json
import re
import subprocess
from pathlib import Path

import pytest
import torch

import exact_headdim_attention_gb300 as pkg
from exact_headdim_attention_gb300 import build as bld

ROOT = Path(__file__).resolve().parent.parent
GOLDEN = json.loads((Path(__file__).parent / "golden" / "api_errors.json").read_text())

FAKE = 0x7F0000000000          # 16-byte aligned, never dereferenced by host checks


@pytest.fixture(scope="module")
def lib():
    bld.build()
    return pkg.load_library()


def declared_symbols():
    text = (ROOT / "include" / "ffpa.h").read_text()
    return sorted(set(re.findall(r"\b(ffpa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert declared_symbols() == sorted(pkg.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(pkg.lib_path())], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ffpa_[a-z0-9_]+)\b", out))
    for name in declared_symbols():
        assert name in exported, f"{name} not exported"
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for s in range(6):
        txt = pkg.ffpa_status_string(s)
        assert txt.startswith("FFPA_")
    assert "unknown" in pkg.ffpa_status_string(99)


def _arr(vals):
    return (ctypes.c_int64 * len(vals))(*vals)


def dense_call(lib, dt=0, B=1, Hq=2, Hkv=2, Nq=128, Nkv=128, D=64, causal=0, enable_gqa=0,
               q=FAKE, qs=None, mask=None, mask_kind=0, mask_str=None, scale=None, o=FAKE,
               lse=None, options=None):
    def st(H, N):
        return _arr([H * N * D, N * D, D, 1])
    qs = qs or st(Hq, Nq)
    ks = st(Hkv, Nkv)
    sc = None if scale is None else ctypes.byref(ctypes.c_float(scale))
    if options is None:
        return lib.ffpa_fwd(q, FAKE, FAKE, o, lse, dt, B, Hq, Hkv, Nq, Nkv, D, qs, ks, ks,
                            st(Hq, Nq), mask, mask_kind, mask_str, sc, causal, enable_gqa, None)
    return lib.ffpa_fwd_ex(q, FAKE, FAKE, o, lse, dt, B, Hq, Hkv, Nq, Nkv, D, qs, ks, ks, st(Hq, Nq),
                           mask, mask_kind, mask_str, sc, causal, enable_gqa, None,
                           ctypes.byref(options))


def varlen_call(lib, dt=0, Tq=256, Tk=256, Hq=2, Hkv=2, D=64, nseq=2, causal=0, enable_gqa=0,
                cu=FAKE, max_q=128, max_k=128):
    def st(H):
        return _arr([H * D, D, 1])
    return lib.ffpa_fwd_varlen(FAKE, FAKE, FAKE, FAKE, None, dt, Tq, Tk, Hq, Hkv, D, st(Hq), st(Hkv),
                               st(Hkv), st(Hq), cu, None, nseq, max_q, max_k, None, causal,
                               enable_gqa, None)


@pytest.mark.parametrize("case", GOLDEN["dense"], ids=lambda c: c["case"])
def test_dense_documented_errors(lib, case):
    assert dense_call(lib, **case["override"]) == case["status"]


@pytest.mark.parametrize("case", GOLDEN["varlen"], ids=lambda c: c["case"])
def test_varlen_documented_errors(lib, case):
    assert varlen_call(lib, **case["override"]) == case["status"]


def test_dense_layout_and_pointer_checks(lib):
    INVALID = pkg.FFPA_ERR_INVALID
    assert dense_call(lib, q=None) == INVALID
    assert dense_call(lib, q=FAKE + 8) == INVALID                      # misaligned base
    assert dense_call(lib, o=FAKE + 2) == INVALID
    assert dense_call(lib, qs=_arr([2 * 128 * 64, 128 * 64, 64, 2])) == INVALID   # D stride != 1
    assert dense_call(lib, qs=_arr([2 * 128 * 68, 128 * 68, 68, 1])) == INVALID   # 136-byte rows
    assert dense_call(lib, B=-1) == INVALID
    assert dense_call(lib, Hkv=0) == INVALID
    assert dense_call(lib, mask_kind=9) == INVALID
    assert dense_call(lib, mask_kind=1, mask=None, mask_str=_arr([0, 0, 0, 1])) == INVALID
    assert dense_call(lib, mask_kind=2, mask=FAKE, mask_str=_arr([0, -1, 0, 1])) == INVALID
    assert dense_call(lib, scale=float("inf")) == INVALID
    assert dense_call(lib, scale=float("nan")) == INVALID
    # a mask pointer not aligned to its element type, an LSE not aligned to 4 bytes
    for kind, off in ((2, 2), (2, 1), (3, 1)):
        assert dense_call(lib, mask_kind=kind, mask=FAKE + off, mask_str=_arr([0, 0, 0, 1])) == INVALID
    assert dense_call(lib, lse=FAKE + 2) == INVALID


def test_options_are_checked(lib):
    """ffpa_options.kernel outside FFPA_VARIANT_AUTO..DUAL is rejected; the
    defaults (all zero) behave as the plain entry point."""
    bad = pkg.Options(None, 0, 7, 0)
    assert dense_call(lib, options=bad) == pkg.FFPA_ERR_INVALID
    assert dense_call(lib, options=pkg.Options(None, 0, 5, 0)) == pkg.FFPA_ERR_INVALID
    assert dense_call(lib, options=pkg.Options(None, 0, -1, 0)) == pkg.FFPA_ERR_INVALID
    assert dense_call(lib, options=pkg.Options(None, 0, 0, 0), D=32) == pkg.FFPA_ERR_UNSUPPORTED
    if not torch.cuda.is_available():
        assert dense_call(lib, options=pkg.Options(None, 0, 3, 0)) == dense_call(lib)

def test_check_order_dtype_first(lib):
    # a bad dtype is reported even when everything else is also wrong
    assert dense_call(lib, dt=3, D=32, Hq=3, Hkv=2, q=None) == pkg.FFPA_ERR_DTYPE
    # an unsupported head dim is reported before layout problems
    assert dense_call(lib, D=32, q=None) == pkg.FFPA_ERR_UNSUPPORTED


def test_varlen_pointer_checks(lib):
    assert varlen_call(lib, cu=None) == pkg.FFPA_ERR_INVALID
    assert varlen_call(lib, max_q=-1) == pkg.FFPA_ERR_INVALID


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    assert dense_call(lib) == pkg.FFPA_ERR_CUDA


def test_binding_maps_statuses_to_page_exceptions(lib):
    q = torch.zeros(1, 2, 4, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        pkg.ffpa_fwd(q, q, q)
    qb = q.bfloat16()
    with pytest.raises(NotImplementedError):
        pkg.ffpa_fwd(qb, qb, qb, dropout_p=0.1)
    with pytest.raises(TypeError):
        pkg.ffpa_fwd(qb, qb, qb, window_size=(1, 1))
    qd = torch.zeros(1, 2, 4, 32, dtype=torch.bfloat16)
    with pytest.raises(NotImplementedError):
        pkg.ffpa_fwd(qd, qd, qd)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd(qb, qb[:, :1].expand(1, 1, 4, 64), qb[:, :1])   # Hq != Hkv, no enable_gqa


def test_binding_rejects_malformed_cu_seqlens(lib):
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        pkg.ffpa_fwd_varlen(q, q, q, torch.tensor([0, 10], dtype=torch.int64), None, 10, 10)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd_varlen(q, q, q, torch.tensor([0, 4, 3, 10], dtype=torch.int32), None, 10, 10)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd_varlen(q, q, q, torch.tensor([0, 9], dtype=torch.int32), None, 10, 10)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd_varlen(q, q, q, torch.tensor([0, 10], dtype=torch.int32), None, 5, 10)
    with pytest.raises(NotImplementedError):
        pkg.ffpa_fwd_varlen(q, q, q, torch.tensor([0, 10], dtype=torch.int32), None, 10, 10,
                            softcap=1.0)


def test_kernel_variant_names(lib):
    for name in ("single", "pair", "split", "dual", "auto"):
        pkg.selected_kernel(512, kernel=name)
    with pytest.raises(ValueError):
        pkg.selected_kernel(512, kernel="fastest")
    assert lib.ffpa_selected_kernel(512, 0, 7) == -1        # out of range
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd(q, q, q, kernel="fastest")


def test_selected_kernel_follows_the_choice(lib):
    assert pkg.selected_kernel(512) == "split"
    assert pkg.selected_kernel(512, varlen=True) == "split"
    assert pkg.selected_kernel(256) == "pair"
    assert pkg.selected_kernel(256, varlen=True) == "single"
    assert pkg.selected_kernel(1024) == "split"                    # cluster of 4 CTAs
    assert pkg.selected_kernel(768) == "split"                     # cluster of 3 CTAs
    assert pkg.selected_kernel(768, varlen=True) == "split"
    assert pkg.selected_kernel(640) == "split"                     # padded to 12 chunks, C = 3
    assert pkg.selected_kernel(320) == "split"                     # padded to 6 chunks, C = 2
    assert pkg.selected_kernel(320, varlen=True) == "split"
    assert pkg.selected_kernel(192) == "single"                    # one output slice, S once
    assert pkg.selected_kernel(192, kernel="split") == "split"
    assert pkg.selected_kernel(1024, kernel="single") == "single"
    assert pkg.selected_kernel(512, kernel="pair") == "pair"
    assert pkg.selected_kernel(384, kernel="pair") == "single"      # pair kernel does not take D=384
    assert pkg.selected_kernel(384, kernel="split") == "split"
    assert pkg.selected_kernel(640, kernel="split") == "split"
    assert pkg.selected_kernel(64, kernel="split") == "single"     # the split needs two chunks
    assert pkg.selected_kernel(512) == "split"                     # no choice outlives a call
    assert lib.ffpa_selected_kernel(100, 0, 0) == -1
    with pytest.raises(ValueError):
        pkg.selected_kernel(100)                          # not a multiple of 8
    assert pkg.selected_kernel(96) == "single"            # zero-padded to two chunks
    # dual tile: dense D = 64 and 128 only
    assert pkg.selected_kernel(64) == "dual"
    assert pkg.selected_kernel(128) == "dual"
    assert pkg.selected_kernel(128, varlen=True) == "single"
    assert pkg.selected_kernel(128, kernel="dual") == "dual"
    assert pkg.selected_kernel(256, kernel="dual") == "single"
    assert pkg.selected_kernel(128, kernel="single") == "single"
    assert pkg.selected_kernel(128, kernel="split") == "split"
    assert pkg.selected_kernel(120, kernel="dual") == "single"


def bwd_call(lib, dt=0, B=1, Hq=2, Hkv=2, Nq=128, Nkv=128, D=64, causal=0, enable_gqa=0,
             lse=FAKE, delta=FAKE, dk=FAKE, qs=None, scale=None, mask=None, mask_kind=0, mask_str=None):
    def st(H, N):
        return _arr([H * N * D, N * D, D, 1])
    qs = qs or st(Hq, Nq)
    ks = st(Hkv, Nkv)
    sc = None if scale is None else ctypes.byref(ctypes.c_float(scale))
    return lib.ffpa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, lse, FAKE, dk, FAKE, delta, dt, B, Hq, Hkv, Nq,
                        Nkv, D, qs, ks, ks, qs, qs, qs, ks, ks, mask, mask_kind, mask_str, sc, causal,
                        enable_gqa, None)


@pytest.mark.parametrize("case", GOLDEN["dense"], ids=lambda c: c["case"])
def test_bwd_documented_errors(lib, case):
    """The backward takes the forward's arguments and applies the same checks."""
    assert bwd_call(lib, **case["override"]) == case["status"]


def test_bwd_layout_and_pointer_checks(lib):
    INVALID = pkg.FFPA_ERR_INVALID
    assert bwd_call(lib, lse=None) == INVALID
    assert bwd_call(lib, delta=None) == INVALID
    assert bwd_call(lib, dk=FAKE + 4) == INVALID                                  # misaligned output
    assert bwd_call(lib, qs=_arr([2 * 128 * 64, 128 * 64, 64, 2])) == INVALID     # D stride != 1
    assert bwd_call(lib, scale=float("nan")) == INVALID
    assert bwd_call(lib, dt=5, lse=None) == pkg.FFPA_ERR_DTYPE
    assert bwd_call(lib, B=0, lse=None) == pkg.FFPA_OK                           # nothing to write
    assert bwd_call(lib, mask_kind=9) == INVALID
    assert bwd_call(lib, mask_kind=1, mask=None, mask_str=_arr([0, 0, 0, 1])) == INVALID
    assert bwd_call(lib, mask_kind=2, mask=FAKE, mask_str=_arr([0, -1, 0, 1])) == INVALID


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_bwd_valid_call_without_gpu_reports_cuda_error(lib):
    assert bwd_call(lib) == pkg.FFPA_ERR_CUDA


def test_bwd_workspace_bytes(lib):
    """The stored-tile workspace: a 32 KB block of zeros, then P and dS as one
    32 KB block (128 x 128 16-bit values) per (b, hq, query tile, key tile)
    each; zero where the path does not apply."""
    wb = pkg.bwd_workspace_bytes
    assert wb(1, 16, 16, 4096, 4096, 512) == (2 * 16 * 32 * 32 + 1) * 32768
    assert wb(2, 8, 2, 300, 129, 256) == (2 * 2 * 8 * 3 * 2 + 1) * 32768
    assert wb(1, 4, 1, 1, 1, 384) == (2 * 4 + 1) * 32768
    for D in (64, 192, 320, 448, 576, 768, 1024):
        assert wb(1, 2, 2, 256, 256, D) == 0, D          # the slice kernels only
    assert wb(1, 2, 2, 256, 256, 128) == (2 * 2 * 2 * 2 + 1) * 32768
    assert wb(1, 2, 2, 0, 256, 512) == 0                 # no query rows
    assert wb(1, 2, 2, 256, 0, 512) == 0                 # no keys
    assert wb(1, 3, 2, 256, 256, 512) == 0               # not a grouping
    assert wb(1 << 16, 1 << 8, 1, 1 << 17, 128, 512) == 0   # more than 2^30 blocks


def _stored_tiles_brute(Nq, Nkv):
    """Key tiles of each query tile that some row sees (lower-right causal), summed."""
    total = 0
    for qt in range(-(-Nq // 128)):
        last_row = min(Nq, (qt + 1) * 128) - 1
        last_key = min(Nkv - 1, last_row + (Nkv - Nq))
        total += last_key // 128 + 1
    return total


def test_bwd_workspace_bytes_causal(lib):
    """Under causal masking only the visible key tiles are stored: the block
    count is the brute-force sum over query tiles; non-causal keeps all."""
    wb = pkg.bwd_workspace_bytes
    for Nq, Nkv in ((4096, 4096), (300, 300), (129, 1000), (1, 1), (1, 129), (127, 129), (256, 1024),
                    (1000, 1000), (640, 641)):
        for B, Hq in ((1, 1), (2, 8)):
            want = (2 * B * Hq * _stored_tiles_brute(Nq, Nkv) + 1) * 32768
            assert wb(B, Hq, Hq, Nq, Nkv, 512, True) == want, (Nq, Nkv)
            assert wb(B, Hq, Hq, Nq, Nkv, 512, False) == (2 * B * Hq * (-(-Nq // 128)) * (-(-Nkv // 128)) + 1) * 32768
    assert wb(1, 2, 2, 300, 200, 512, True) == 0      # causal needs Nkv >= Nq
    assert wb(1, 16, 16, 4096, 4096, 512, True) == (2 * 16 * (32 * 33 // 2) + 1) * 32768


def test_varlen_bwd_workspace_bytes(lib):
    """Varlen: a 1 KB-rounded header of nseq + 1 int64, a zero block, and P and
    dS blocks summed over the sequences (brute force per sequence, lower-right
    causal within each; sequences with fewer keys than queries included)."""
    vb = pkg.varlen_bwd_workspace_bytes
    def want(cq, ck, Hq, causal):
        blocks = 0
        for s in range(len(cq) - 1):
            lq, lk = cq[s + 1] - cq[s], ck[s + 1] - ck[s]
            if lq == 0 or lk == 0:
                continue
            if not causal:
                blocks += Hq * (-(-lq // 128)) * (-(-lk // 128))
                continue
            for qt in range(-(-lq // 128)):
                last_row = min(lq, (qt + 1) * 128) - 1
                last_key = min(lk - 1, last_row + (lk - lq))
                blocks += Hq * (last_key // 128 + 1 if last_key >= 0 else 0)
        hdr = -(-((len(cq)) * 8) // 1024) * 1024
        return hdr + (2 * blocks + 1) * 32768 if blocks else 0
    cases = [([0, 300, 428, 429, 879], None), ([0, 100, 300, 300, 364], [0, 150, 350, 380, 680]),
             ([0, 50, 60, 317], [0, 20, 30, 290]), ([0, 4096], None), ([0, 1, 2], [0, 1, 130])]
    for cq, ck in cases:
        ck = ck or cq
        for causal in (False, True):
            for Hq in (1, 4):
                assert vb(cq, ck, Hq, 1, 512, causal) == want(cq, ck, Hq, causal), (cq, ck, causal)
    assert vb([0, 300], [0, 300], 2, 2, 64, False) == 0           # the slice kernels only
    assert vb([0, 0, 0], [0, 0, 0], 2, 2, 512, False) == 0        # nothing to store
    assert vb([0, 300], [0, 300], 3, 2, 512, False) == 0          # not a grouping


def bwd_ws_call(lib, ws, ws_bytes, D=512, dt=0):
    def st(N):
        return _arr([2 * N * D, N * D, D, 1])
    s = st(128)
    return lib.ffpa_bwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dt, 1, 2, 2, 128,
                           128, D, s, s, s, s, s, s, s, s, None, 0, None, None, 0, 0, ws, ws_bytes, None)


def test_bwd_ws_checks(lib):
    need = pkg.bwd_workspace_bytes(1, 2, 2, 128, 128, 512)
    # a workspace that would be used must be 16-byte aligned
    assert bwd_ws_call(lib, FAKE + 8, need) == pkg.FFPA_ERR_INVALID
    # argument errors come first, as for ffpa_bwd
    assert bwd_ws_call(lib, FAKE, need, D=100) == pkg.FFPA_ERR_UNSUPPORTED
    assert bwd_ws_call(lib, FAKE, need, dt=7) == pkg.FFPA_ERR_DTYPE
    if not torch.cuda.is_available():
        # a misaligned workspace that is too small is not used, so not checked
        assert bwd_ws_call(lib, FAKE + 8, need - 1) == pkg.FFPA_ERR_CUDA
        assert bwd_ws_call(lib, FAKE, need) == pkg.FFPA_ERR_CUDA
        assert bwd_ws_call(lib, None, 0) == pkg.FFPA_ERR_CUDA


def test_binding_checks_caller_outputs(lib):
    """Caller-supplied outputs must have the shape, dtype and device the library
    writes: the C side sizes every write from q and k."""
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    for bad in (torch.zeros(1, 2, 3, 64, dtype=torch.bfloat16),      # fewer rows
                torch.zeros(1, 2, 4, 64, dtype=torch.float16),       # other dtype
                torch.zeros(2, 4, 64, dtype=torch.bfloat16),         # rank 3
                torch.zeros(1, 2, 4, 32, dtype=torch.bfloat16)):     # narrower D
        with pytest.raises(ValueError):
            pkg.ffpa_fwd(q, q, q, out=bad)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd(q, q, q, lse=torch.zeros(1, 2, 3))
    with pytest.raises(ValueError):
        pkg.ffpa_fwd(q, q, q, lse=torch.zeros(1, 2, 4, dtype=torch.float64))
    with pytest.raises(ValueError):
        pkg.ffpa_fwd(q, q, q, status=torch.zeros(1, dtype=torch.int64))
    qv = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 10], dtype=torch.int32)
    with pytest.raises(ValueError):
        pkg.ffpa_fwd_varlen(qv, qv, qv, cu, None, 10, 10, out=qv[:9])
    with pytest.raises(ValueError):
        pkg.ffpa_fwd_varlen(qv, qv, qv, cu, None, 10, 10, lse=torch.zeros(10, 2))   # [T, H] not [H, T]
    lse = torch.zeros(1, 2, 4)
    for name, bad in (("dq", q[:, :1]), ("dk", q.half()), ("dv", q[..., :32]),
                      ("delta", torch.zeros(1, 2, 4, dtype=torch.float64))):
        with pytest.raises(ValueError):
            pkg.ffpa_bwd(q, q, q, q, q, lse, **{name: bad})
    with pytest.raises(ValueError):
        pkg.ffpa_bwd_varlen(qv, qv, qv, qv, qv, torch.zeros(2, 10), cu, None, 10, 10, dq=qv[:, :1])


def test_bwd_binding_checks(lib):
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 4)
    with pytest.raises(ValueError):
        pkg.ffpa_bwd(q, q, q, q, q, lse.double())                 # lse must be float32
    with pytest.raises(ValueError):
        pkg.ffpa_bwd(q, q, q, q, q[:, :, :3], lse)                # out shape
    with pytest.raises(TypeError):
        pkg.ffpa_bwd(q.half(), q, q, q, q, lse)                   # mixed dtypes


def test_fine_head_dims_dense_only(lib):
    """Dense head dims divisible by 8 are accepted (zero-padded chunks, single-CTA
    kernel); varlen and the backward keep whole 64-column chunks."""
    UNSUP = pkg.FFPA_ERR_UNSUPPORTED
    assert dense_call(lib, D=72) != UNSUP
    assert dense_call(lib, D=1000) != UNSUP
    assert dense_call(lib, D=100) == UNSUP
    assert varlen_call(lib, D=72) == UNSUP
    assert bwd_call(lib, D=72) == UNSUP
    assert pkg.selected_kernel(72) == "single"
    assert pkg.selected_kernel(520) == "single"
    with pytest.raises(ValueError):
        pkg.selected_kernel(72, varlen=True)
    assert pkg.selected_kernel(120, kernel="split") == "single"
    assert pkg.selected_kernel(192 + 8, kernel="pair") == "single"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_fine_head_dim_valid_call_without_gpu(lib):
    assert dense_call(lib, D=120) == pkg.FFPA_ERR_CUDA


def bwd_varlen_call(lib, dt=0, Tq=256, Tk=256, Hq=2, Hkv=2, D=64, nseq=2, causal=0, enable_gqa=0,
                    cu=FAKE, max_q=128, max_k=128, lse=FAKE, delta=FAKE):
    def st(H):
        return _arr([H * D, D, 1])
    qs, ks = st(Hq), st(Hkv)
    return lib.ffpa_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, lse, FAKE, FAKE, FAKE, delta, dt, Tq, Tk, Hq,
                               Hkv, D, qs, ks, ks, qs, qs, qs, ks, ks, cu, None, nseq, max_q, max_k,
                               None, causal, enable_gqa, None)


@pytest.mark.parametrize("case", GOLDEN["varlen"], ids=lambda c: c["case"])
def test_bwd_varlen_documented_errors(lib, case):
    """The varlen backward applies the varlen forward's checks."""
    assert bwd_varlen_call(lib, **case["override"]) == case["status"]


def test_bwd_varlen_pointer_checks(lib):
    INVALID = pkg.FFPA_ERR_INVALID
    assert bwd_varlen_call(lib, cu=None) == INVALID
    assert bwd_varlen_call(lib, lse=None) == INVALID
    assert bwd_varlen_call(lib, delta=None) == INVALID
    assert bwd_varlen_call(lib, max_q=-1) == INVALID
    assert bwd_varlen_call(lib, Tq=0, Tk=0, lse=None) == pkg.FFPA_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_bwd_varlen_valid_call_without_gpu(lib):
    assert bwd_varlen_call(lib) == pkg.FFPA_ERR_CUDA
