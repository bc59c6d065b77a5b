"""wa_forward_static: the forward pass for callers that may not allocate device memory (for example a framework
that only hands out memory from its own accounted pool, or code under a fixed device-memory budget). Its scratch
is a library-owned static device array, so it is checked here against the plan-based wa_forward on the same
inputs, on two calls in a row with different geometries, so that a stale scratch from the first call cannot
leak into the second. Named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

REL_TOL = 5e-3
ABS_TOL = 3e-2


def static_forward(wa, w, q, k, v):
    out = torch.full_like(q, float("nan"))  # a work item left out would leave NaN rows behind
    lay = wa.make_layout(w.B, w.L, w.H, w.D, w.global_pos)
    s = torch.cuda.current_stream().cuda_stream
    st = wa.lib().wa_forward_static(w.T, w.S, w.K, w.r, w.G, ctypes.byref(lay), ctypes.c_void_p(q.data_ptr()),
                                    ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                    ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(s))
    assert st == 0, wa.wa_status_string(st)
    torch.cuda.synchronize()
    return out


def plan_forward(wa, w, q, k, v):
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out = plan.forward(q, k, v)
        assert plan.check_error() == 0
    finally:
        plan.close()
    return out


def close(a, b):
    a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
    for bi in range(a.shape[0]):
        for h in range(a.shape[2]):
            x, y = a[bi, :, h], b[bi, :, h]
            assert np.linalg.norm(x - y) / np.linalg.norm(y) <= REL_TOL
            assert np.abs(x - y).max() <= ABS_TOL


def test_static_scratch_matches_plan_forward_twice(cuda):
    for w in (configs.MEDIUM, configs.RAGGED):  # two calls in a row, different geometries and scratch layouts
        q, k, v = inputs.make_qkv(w, device="cuda")
        close(static_forward(cuda, w, q, k, v), plan_forward(cuda, w, q, k, v))
    w = configs.MEDIUM  # and once more on the first geometry, over the second call's leftover scratch
    q, k, v = inputs.make_qkv(w, seed=77, device="cuda")
    close(static_forward(cuda, w, q, k, v), plan_forward(cuda, w, q, k, v))


def test_static_scratch_rejects_oversized_geometry(cuda):
    # 200,000 global rows: the global-leg workspace alone exceeds the 32 MiB array; nothing may be launched
    T, S, K, r, G = 1, 8, 1, 0, 200000
    L = T * S + G
    q = torch.zeros(1, L, 1, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lay = cuda.make_layout(1, L, 1, 128, 0)
    st = cuda.lib().wa_forward_static(T, S, K, r, G, ctypes.byref(lay), ctypes.c_void_p(q.data_ptr()),
                                      ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                      ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(0))
    assert st == 2  # WA_ERR_UNSUPPORTED
    torch.cuda.synchronize()


# 1,000 window groups of one query tile each plus 63 global split items: 1,063 work items per (b, h), so the
# allocation-free call writes its work list with two expansion launches (800 per launch)
MANY_GROUPS = configs.Workload("many_groups", B=1, H=2, D=64, T=1000, S=64, K=1, r=0, G=64, global_pos=0, seed=71)
# head dim 64 with the globals before the frames
D64_FRONT = configs.Workload("d64_front", B=2, H=3, D=64, T=13, S=37, K=4, r=2, G=130, global_pos=1, seed=72)


def test_dynamic_claiming_matches_static_striding(cuda):
    """A plan's forward lets each CTA claim its next work item from a counter (the last CTA of a launch rewinds it);
    wa_forward_static writes the same items into its scratch on the device and hands them out by static striding.
    Same items and the same arithmetic per item: the results agree bit for bit, over several launches in a row on
    one plan (a counter left unrewound would make the next launch skip its items and leave the NaN in place)."""
    for w in (configs.MEDIUM, configs.RAGGED, MANY_GROUPS, D64_FRONT):
        plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
        try:
            for seed in (5, 6, 7):
                q, k, v = inputs.make_qkv(w, seed=seed, device="cuda")
                out = torch.full_like(q, float("nan"))
                plan.forward(q, k, v, out=out)
                assert plan.check_error() == 0
                assert torch.equal(out, static_forward(cuda, w, q, k, v))
        finally:
            plan.close()


def test_static_forward_in_a_cuda_graph(cuda):
    """After a first call in the context (it looks up the array's address), the allocation-free forward can be
    captured: the work list travels in the launches' parameters, so every replay rewrites it on the device and
    reads nothing from the host. Two replays on fresh inputs equal eager calls bit for bit (MANY_GROUPS: two
    expansion launches per call)."""
    w = MANY_GROUPS
    q, k, v = inputs.make_qkv(w, device="cuda")
    static_forward(cuda, w, q, k, v)
    out = torch.empty_like(q)
    lay = cuda.make_layout(w.B, w.L, w.H, w.D, w.global_pos)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream().cuda_stream
        st = cuda.lib().wa_forward_static(w.T, w.S, w.K, w.r, w.G, ctypes.byref(lay), ctypes.c_void_p(q.data_ptr()),
                                          ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                          ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(s))
    assert st == 0, cuda.wa_status_string(st)
    for seed in (31, 32):
        q2, k2, v2 = inputs.make_qkv(w, seed=seed, device="cuda")
        q.copy_(q2)
        k.copy_(k2)
        v.copy_(v2)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, static_forward(cuda, w, q2, k2, v2)), f"seed {seed}"
