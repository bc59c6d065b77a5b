"""window_softmax_decomposed under torch.autograd: the forward equals plan.forward bit for bit, the gradients that
autograd delivers equal plan.backward's bit for bit (for any upstream gradient layout), and they match the fp64
oracle's backward within the gradient bar of tests/test_backward_gpu.py."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

GRAD_REL = 5e-3
GRAD_ABS = 2e-2  # times max |reference| of the slice

CASES = [configs.TINY,
         configs.Workload("ag_front_d128", B=2, H=3, D=128, T=9, S=40, K=2, r=1, G=70, global_pos=1, seed=61),
         configs.Workload("ag_dense_d64", B=1, H=2, D=64, T=5, S=30, K=2, r=3, G=0, global_pos=0, seed=62)]


def leaves(w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    return [t.detach().clone().requires_grad_(True) for t in (q, k, v)]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_autograd_matches_plan_backward_and_oracle(cuda, w):
    q, k, v = leaves(w)
    dout = inputs.make_dout(w).to("cuda")
    out = cuda.window_softmax_decomposed(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    out.backward(dout)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out_ref, lse = plan.forward_lse(q.detach(), k.detach(), v.detach())
        grads = plan.backward(q.detach(), k.detach(), v.detach(), out_ref, dout, lse)
        assert plan.check_error() == 0
    finally:
        plan.close()
    assert torch.equal(out.detach(), out_ref)
    for name, a, b in zip(("dq", "dk", "dv"), (q.grad, k.grad, v.grad), grads):
        assert torch.equal(a, b), f"{w.name} {name}: autograd differs from plan.backward"
    want = ref.window_attention_backward(q.detach(), k.detach(), v.detach(), dout, w.T, w.S, w.K, w.r, w.G,
                                         w.global_pos)
    for name, g, r in zip(("dq", "dk", "dv"), (q.grad, k.grad, v.grad), want):
        g = g.float().cpu().double().numpy()
        for b in range(r.shape[0]):
            for h in range(r.shape[2]):
                gs, rs = g[b, :, h], r[b, :, h]
                rel = np.linalg.norm(gs - rs) / max(np.linalg.norm(rs), 1e-30)
                ab = np.abs(gs - rs).max() / max(np.abs(rs).max(), 1e-30)
                assert rel <= GRAD_REL and ab <= GRAD_ABS, f"{w.name} {name} b{b} h{h}: rel {rel:.2e} abs {ab:.2e}"


def test_expanded_upstream_gradient_and_partial_requires_grad(cuda):
    # loss = out.sum(): autograd hands the backward an expanded (stride 0) gradient of ones; only k needs a gradient
    w = configs.TINY
    q, k, v = leaves(w)
    q.requires_grad_(False)
    v.requires_grad_(False)
    out = cuda.window_softmax_decomposed(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    out.float().sum().backward()
    assert q.grad is None and v.grad is None
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out_ref, lse = plan.forward_lse(q.detach(), k.detach(), v.detach())
        ones = torch.ones_like(out_ref)
        _, dk, _ = plan.backward(q.detach(), k.detach(), v.detach(), out_ref, ones, lse)
    finally:
        plan.close()
    assert torch.equal(k.grad, dk)


def test_head_major_layout(cuda):
    # [B, H, L, D] physical order seen through a [B, L, H, D] view: the plan takes the strides as they are
    w = configs.Workload("ag_head_major", B=1, H=2, D=64, T=6, S=20, K=2, r=1, G=12, global_pos=0, seed=63)
    q, k, v = (t.detach().permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3).requires_grad_(True)
               for t in inputs.make_qkv(w, device="cuda"))
    dout = inputs.make_dout(w).to("cuda")
    out = cuda.window_softmax_decomposed(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    out.backward(dout)
    want = ref.window_attention_backward(q.detach(), k.detach(), v.detach(), dout, w.T, w.S, w.K, w.r, w.G,
                                         w.global_pos)
    for g, r in zip((q.grad, k.grad, v.grad), want):
        g = g.float().cpu().double().numpy()
        assert np.linalg.norm(g - r) / np.linalg.norm(r) <= GRAD_REL
