"""The plan entry points inside CUDA graphs: a forward (and a forward with row log-sum-exp plus the backward)
captured once and replayed on fresh inputs copied into the captured tensors must give exactly what eager calls
give on those inputs, replay after replay (each launch leaves the plan's work counter as it found it). The capture
runs on another stream than the plan's previous eager call, which must not make the captured call wait on an
event recorded outside the capture; eager calls on yet another stream still work after it. Calls that cannot be
captured (a first backward, which allocates its workspace; the host-buffer forward; the error check, which
synchronises) are refused with WA_ERR_UNSUPPORTED and queue nothing, so the capture stays valid."""
import ctypes

import pytest
import torch

from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

# 2 x 4 slices; 5 chunks of 2 frames x 200 tokens (window items with one and two query tiles) and 300 globals
# (split items, so the merge kernel is captured too)
W = configs.Workload("graph_small", B=2, H=4, D=128, T=9, S=200, K=2, r=1, G=300, global_pos=0, seed=91)
# a geometry no other test uses: plans are shared through the process-wide plan cache, and this test needs a plan
# on which no backward has run yet
W_FRESH = configs.Workload("graph_fresh", B=1, H=3, D=128, T=7, S=200, K=2, r=1, G=260, global_pos=1, seed=92)
WA_ERR_UNSUPPORTED = 2


def new_plan(wa, w):
    return wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)


def test_forward_graph_replays_equal_eager_calls(cuda):
    w = W
    plan = new_plan(cuda, w)
    try:
        q, k, v = inputs.make_qkv(w, device="cuda")
        out = torch.empty_like(q)
        plan.forward(q, k, v, out=out)  # eager, on the default stream: the capture below runs on a side stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.forward(q, k, v, out=out)
        for seed in (101, 102, 103):
            q2, k2, v2 = inputs.make_qkv(w, seed=seed, device="cuda")
            q.copy_(q2)
            k.copy_(k2)
            v.copy_(v2)
            out.fill_(float("nan"))
            g.replay()
            want = plan.forward(q2, k2, v2)
            torch.cuda.synchronize()
            assert torch.equal(out, want), f"replay with seed {seed} differs from the eager call"
        other = torch.cuda.Stream()
        with torch.cuda.stream(other):
            again = plan.forward(q2, k2, v2)
        other.synchronize()
        assert torch.equal(again, want)
        assert plan.check_error() == 0
    finally:
        plan.close()


def test_fp8_forward_graph(cuda):
    """The e4m3 forward (scales fixed at capture, as every launch argument is) replays like its eager call."""
    w = W
    plan = new_plan(cuda, w)
    try:
        q, k, v = inputs.make_qkv(w, device="cuda")
        sq, sk = 8.0 / 448.0, 8.0 / 448.0  # N(0, 1) draws stay below 8: nothing leaves the e4m3 range
        q8, k8 = (q.float() / sq).to(torch.float8_e4m3fn), (k.float() / sk).to(torch.float8_e4m3fn)
        out = torch.empty_like(v)
        plan.forward_fp8(q8, k8, v, sq, sk, out=out)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.forward_fp8(q8, k8, v, sq, sk, out=out)
        for seed in (121, 122):
            q2, k2, v2 = inputs.make_qkv(w, seed=seed, device="cuda")
            q8.copy_((q2.float() / sq).to(torch.float8_e4m3fn))
            k8.copy_((k2.float() / sk).to(torch.float8_e4m3fn))
            v.copy_(v2)
            out.fill_(float("nan"))
            g.replay()
            want = plan.forward_fp8(q8.clone(), k8.clone(), v2, sq, sk)
            torch.cuda.synchronize()
            assert torch.equal(out, want), f"seed {seed}"
        assert plan.check_error() == 0
    finally:
        plan.close()


def test_forward_lse_and_backward_graph(cuda):
    w = W
    plan = new_plan(cuda, w)
    try:
        q, k, v = inputs.make_qkv(w, device="cuda")
        dout = inputs.make_dout(w, device="cuda")
        out, lse = plan.forward_lse(q, k, v)
        plan.backward(q, k, v, out, dout, lse)  # eager first call: allocates the backward workspace
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            out_g, lse_g = plan.forward_lse(q, k, v)
            grads_g = plan.backward(q, k, v, out_g, dout, lse_g)
        for seed in (111, 112):
            q2, k2, v2 = inputs.make_qkv(w, seed=seed, device="cuda")
            d2 = inputs.make_dout(w, seed=seed, device="cuda")
            for dst, src in ((q, q2), (k, k2), (v, v2), (dout, d2)):
                dst.copy_(src)
            g.replay()
            out_e, lse_e = plan.forward_lse(q2, k2, v2)
            grads_e = plan.backward(q2, k2, v2, out_e, d2, lse_e)
            torch.cuda.synchronize()
            assert torch.equal(out_g, out_e) and torch.equal(lse_g, lse_e), f"seed {seed}: forward differs"
            for name, a, b in zip(("dq", "dk", "dv"), grads_g, grads_e):
                assert torch.equal(a, b), f"seed {seed}: {name} differs"
        assert plan.check_error() == 0
    finally:
        plan.close()


def test_uncapturable_calls_are_refused_inside_a_capture(cuda):
    w = W_FRESH
    plan = new_plan(cuda, w)
    L = cuda.lib()
    P = ctypes.c_void_p
    try:
        q, k, v = inputs.make_qkv(w, device="cuda")
        dout = inputs.make_dout(w, device="cuda")
        out, lse = plan.forward_lse(q, k, v)
        grads = [torch.empty_like(q) for _ in range(3)]
        host = [torch.zeros(q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(4)]
        out2 = torch.empty_like(q)
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            # no backward has run on this plan yet: its workspace would have to be allocated inside the capture
            st_bwd = L.wa_backward(plan.handle, *(P(t.data_ptr()) for t in (q, k, v, out, dout, lse, *grads)),
                                   P(side.cuda_stream))
            st_host = L.wa_forward_host(plan.handle, *(P(t.data_ptr()) for t in host), P(side.cuda_stream))
            st_check = L.wa_plan_check_error(plan.handle, P(side.cuda_stream))
            plan.forward(q, k, v, out=out2)  # the capture is still valid and records this call
        assert (st_bwd, st_host, st_check) == (WA_ERR_UNSUPPORTED,) * 3
        out2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out2, out)
        # outside a capture the same calls run
        plan.backward(q, k, v, out, dout, lse)
        assert plan.check_error() == 0
    finally:
        plan.close()
