"""Failure paths on the GPU, without faulting it: the device watchdog (a bounded wait that a test-only flag makes
run out), a failed workspace allocation (injected on the host) and the plan cache's reference counting."""
import os

import pytest
import torch

from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu


def test_watchdog_timeout_is_reported_and_device_stays_usable(cuda):
    w = configs.MEDIUM
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        good = plan.forward(q, k, v)
        assert plan.check_error() == 0
        plan.set_debug_flags(1)  # one key tile is never loaded: its consumer's wait runs out
        plan.forward(q, k, v)
        assert plan.check_error() == 5  # WA_ERR_DEVICE_TIMEOUT
        plan.set_debug_flags(0)
        again = plan.forward(q, k, v)
        assert plan.check_error() == 0
        assert torch.equal(good, again)
    finally:
        plan.set_debug_flags(0)
        plan.close()


def test_failed_allocation_is_reported_without_leak(cuda):
    os.environ["WA_TEST_FAIL_ALLOC"] = "1"
    try:
        with pytest.raises(cuda.WAError) as e:
            cuda.Plan(5, 33, 2, 1, 17, 1, 1, 128, 0)  # a geometry no other test caches
        assert e.value.status == 3  # WA_ERR_OOM
    finally:
        del os.environ["WA_TEST_FAIL_ALLOC"]
    p = cuda.Plan(5, 33, 2, 1, 17, 1, 1, 128, 0)
    p.close()


def test_plan_cache_refcount_and_eviction(cuda):
    lib = cuda.lib()
    geos = [(4, 16 + i, 2, 1, 8) for i in range(6)]
    plans = [cuda.Plan(*g, 1, 1, 128, 0) for g in geos]
    assert lib.wa_cache_size() <= 4  # plans beyond the cap stay uncached while every cached one is in use
    again = cuda.Plan(*geos[0], 1, 1, 128, 0)
    assert again.handle.value == plans[0].handle.value
    assert lib.wa_plan_refcount(again.handle) == 2
    again.close()
    assert lib.wa_plan_refcount(plans[0].handle) == 1
    for p in plans:
        p.close()
    # unreferenced plans are evicted least-recently-used first as new geometries arrive
    extra = [cuda.Plan(4, 40 + i, 2, 1, 8, 1, 1, 128, 0) for i in range(4)]
    assert lib.wa_cache_size() == 4
    for p in extra:
        p.close()


def test_forward_argument_errors(cuda):
    w = configs.TINY
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    lib = cuda.lib()
    try:
        s = torch.cuda.current_stream().cuda_stream
        import ctypes
        P = ctypes.c_void_p
        # out aliasing q
        assert lib.wa_forward(plan.handle, P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(q.data_ptr()),
                              P(s)) == 1
        # misaligned pointer
        assert lib.wa_forward(plan.handle, P(q.data_ptr() + 2), P(k.data_ptr()), P(v.data_ptr()),
                              P(torch.empty_like(q).data_ptr()), P(s)) == 1
        assert plan.check_error() == 0
    finally:
        plan.close()


def test_failed_host_path_set_up_is_undone_and_retried(cuda):
    # the host-buffer forward sets up its device copies on first use; a failed allocation there must leave nothing
    # half set up, so that the next call sets it up again and gives the plain forward's result
    w = configs.Workload("host_retry", B=1, H=2, D=128, T=6, S=100, K=2, r=1, G=40, global_pos=0, seed=91)
    q, k, v = inputs.make_qkv(w)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        want = plan.forward(q.cuda(), k.cuda(), v.cuda()).cpu()
        os.environ["WA_TEST_FAIL_ALLOC"] = "1"
        try:
            with pytest.raises(cuda.WAError) as e:
                plan.forward_host(q, k, v)
            assert e.value.status == 3  # WA_ERR_OOM
        finally:
            del os.environ["WA_TEST_FAIL_ALLOC"]
        for _ in range(2):
            got = plan.forward_host(q, k, v)
            assert torch.equal(got, want)
        assert plan.check_error() == 0
    finally:
        plan.close()
