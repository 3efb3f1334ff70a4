"""The torch custom operators over the C ABI (forward, and the backward kernels
through autograd; the gradients themselves are checked on the GPU in
test_gpu_backward.py).

CPU: registration (including the autograd formulas), shape-only fake
implementations, rejected options.
GPU: eager calls through torch.ops against the float64 oracle, and a
torch.compile(fullgraph=True) trace through the operator."""
import pytest
import torch
from torch._subclasses.fake_tensor import FakeTensorMode

import exact_headdim_attention_gb300 as pkg
from exact_headdim_attention_gb300 import torch_ops
from exact_headdim_attention_gb300 import workloads as wl


def test_ops_registered():
    assert hasattr(torch.ops.ffpa, "attn_fwd") and hasattr(torch.ops.ffpa, "attn_varlen_fwd")
    assert pkg.ffpa_attn_func is torch_ops.ffpa_attn_func


def test_autograd_formulas_registered():
    """Both operators carry a backward (the binding's ffpa_bwd / ffpa_bwd_varlen)."""
    for op, bwd, setup in ((torch_ops.attn_fwd, torch_ops._attn_fwd_backward,
                            torch_ops._attn_fwd_setup_context),
                           (torch_ops.attn_varlen_fwd, torch_ops._attn_varlen_backward,
                            torch_ops._attn_varlen_setup_context)):
        assert getattr(op, "_backward_fn", bwd) is bwd
        assert getattr(op, "_setup_context_fn", setup) is setup
    for name in ("ffpa::attn_fwd", "ffpa::attn_varlen_fwd"):
        assert torch._C._dispatch_has_kernel_for_dispatch_key(name, "Autograd")


def test_fake_shapes_dense_and_varlen():
    with FakeTensorMode():
        q = torch.empty(2, 8, 100, 512, dtype=torch.bfloat16)
        k = torch.empty(2, 2, 300, 512, dtype=torch.bfloat16)
        o, lse = torch.ops.ffpa.attn_fwd(q, k, k, None, True, 0.1, True)
        assert o.shape == q.shape and o.dtype == q.dtype
        assert lse.shape == (2, 8, 100) and lse.dtype == torch.float32
        qv = torch.empty(500, 8, 256, dtype=torch.float16)
        cu = torch.empty(4, dtype=torch.int32)
        o, lse = torch.ops.ffpa.attn_varlen_fwd(qv, qv, qv, cu, None, 300, 300, True, None, False)
        assert o.shape == qv.shape and lse.shape == (8, 500)


def test_dropout_rejected():
    q = torch.empty(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(NotImplementedError):
        pkg.ffpa_attn_func(q, q, q, dropout_p=0.1)
    qv = torch.empty(4, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(NotImplementedError):
        pkg.ffpa_attn_varlen_func(qv, qv, qv, torch.tensor([0, 4], dtype=torch.int32), None, 4, 4,
                                  dropout_p=0.5)


@pytest.mark.gpu
def test_op_eager_matches_oracle():
    import oracle
    from tests.gpu_util import check, device_ok
    dev = torch.device("cuda:0")
    q, k, v, g = wl.draw_dense(1, 4, 2, 200, 330, 512, seed=61)
    m = torch.rand(1, 1, 200, 330, generator=g) < 0.8
    o, lse = pkg.ffpa_attn_func(q.to(dev), k.to(dev), v.to(dev), attn_mask=m.to(dev),
                                is_causal=True, enable_gqa=True, return_lse=True)
    device_ok()
    o_ref, l_ref = oracle.attn_dense(q, k, v, attn_mask=m, is_causal=True)
    check(o, lse, o_ref, l_ref, "torch.ops.ffpa.attn_fwd")


@pytest.mark.gpu
def test_varlen_op_matches_oracle():
    import oracle
    from tests.gpu_util import check, device_ok
    dev = torch.device("cuda:0")
    lq = [70, 257, 3]
    q, k, v, cq, ck = wl.draw_varlen(lq, lq, 4, 4, 256, seed=62)
    o, lse = pkg.ffpa_attn_varlen_func(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), None, max(lq),
                                       max(lq), causal=True, return_lse=True)
    device_ok()
    o_ref, l_ref = oracle.attn_varlen(q, k, v, cq, None, causal=True)
    check(o, lse, o_ref, l_ref, "torch.ops.ffpa.attn_varlen_fwd")


@pytest.mark.gpu
def test_compile_fullgraph_through_the_op():
    dev = torch.device("cuda:0")
    q, k, v, _ = wl.draw_dense(1, 2, 2, 256, 256, 320, seed=63)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)

    def f(q, k, v):
        return pkg.ffpa_attn_func(q * 1.0, k, v, scale=0.05) + 1.0

    compiled = torch.compile(f, fullgraph=True, backend="aot_eager")
    torch.testing.assert_close(compiled(q, k, v), f(q, k, v), rtol=0, atol=0)
