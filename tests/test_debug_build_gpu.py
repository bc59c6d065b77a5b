"""The index-checking debug build (``libwa_debug.so``: the sources compiled with -DWA_DEBUG, where each kernel's
item claimer bounds-checks every work item before any copy or store uses it). It stands in for a memory checker:
on Tiny, Medium and Ragged (forward, row log-sum-exp, backward, and the e4m3 forward on Medium and Ragged) no check
fires and every result equals the production library's bit for bit; a test hook that moves one work item's key
segment past the end of the sequence is caught and reported as WA_ERR_DEVICE_BOUNDS, and the next call is clean."""
import contextlib

import pytest
import torch

from chunk_windowed_softmax_gb300 import _build, configs, inputs

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def library(wa, path):
    """Route the binding to another build of the library for the duration of the block."""
    saved = (wa._lib_handle, wa.LIB_PATH)
    wa._lib_handle, wa.LIB_PATH = None, path
    try:
        yield wa
    finally:
        wa._lib_handle, wa.LIB_PATH = saved


def run_all(wa, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out = plan.forward(q, k, v)
        out2, lse = plan.forward_lse(q, k, v)
        grads = plan.backward(q, k, v, out2, dout, lse)
        res = [out, out2, lse, *grads]
        if w.D == 128:
            sq = float(q.float().abs().max()) / 448.0
            sk = float(k.float().abs().max()) / 448.0
            res.append(plan.forward_fp8((q.float() / sq).to(torch.float8_e4m3fn),
                                        (k.float() / sk).to(torch.float8_e4m3fn), v, sq, sk))
        st = plan.check_error()
    finally:
        plan.close()
    torch.cuda.synchronize()
    return st, res


@pytest.fixture(scope="module")
def debug_lib(cuda):
    return _build.build(debug=True)


@pytest.mark.parametrize("w", [configs.TINY, configs.MEDIUM, configs.RAGGED], ids=lambda w: w.name)
def test_debug_build_checks_pass_and_results_match(cuda, debug_lib, w):
    st, want = run_all(cuda, w)
    assert st == 0
    with library(cuda, debug_lib) as dbg:
        st, got = run_all(dbg, w)
    assert st == 0, f"a device-side index check fired: {cuda.wa_status_string(st)}"
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_debug_build_catches_an_out_of_range_segment(cuda, debug_lib):
    w = configs.MEDIUM
    q, k, v = inputs.make_qkv(w, device="cuda")
    with library(cuda, debug_lib) as dbg:
        plan = dbg.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
        try:
            plan.set_debug_flags(8)  # the first item of CTA 0 gets a key segment past the sequence
            plan.forward(q, k, v)
            assert plan.check_error() == 6  # WA_ERR_DEVICE_BOUNDS
            plan.set_debug_flags(0)
            out = plan.forward(q, k, v)
            assert plan.check_error() == 0
        finally:
            plan.close()
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        assert torch.equal(out, plan.forward(q, k, v))
    finally:
        plan.close()
