"""wa_forward_host: the forward on host buffers, pipelined over head groups (copies in, compute, copies out on three
streams). Its results must equal the device-resident forward bit for bit (the same kernels and work items, only
regrouped by head), and therefore the fp64 oracle within the forward's bar."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs
from test_parity_gpu import check_slices, relayout, strides_of

pytestmark = pytest.mark.gpu


def device_forward(wa, w, q, k, v):
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos, strides=strides_of(q))
    try:
        out = plan.forward(q.cuda(), k.cuda(), v.cuda())
        assert plan.check_error() == 0
    finally:
        plan.close()
    return out.cpu()


@pytest.mark.parametrize("w", [configs.MEDIUM, configs.RAGGED,
                               configs.Workload("host_h3_heads", B=1, H=3, D=64, T=9, S=40, K=2, r=1, G=30,
                                                global_pos=0, seed=61)],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_forward_matches_device_forward(cuda, w, pinned):
    q, k, v = inputs.make_qkv(w, device="cuda")
    want = device_forward(cuda, w, q, k, v)
    qh, kh, vh = (t.cpu().pin_memory() if pinned else t.cpu() for t in (q, k, v))
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        got = plan.forward_host(qh, kh, vh)
        again = plan.forward_host(qh, kh, vh)  # the staging buffers are reused
        assert plan.check_error() == 0
    finally:
        plan.close()
    assert not got.is_cuda
    assert torch.equal(got, want) and torch.equal(again, want)


def test_host_forward_against_oracle(cuda):
    w = configs.MEDIUM
    q, k, v = inputs.make_qkv(w)
    out = cuda.forward(q.pin_memory(), k.pin_memory(), v.pin_memory(), w.T, w.S, w.K, w.r, w.G, w.global_pos)
    want = ref.window_attention(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    check_slices({(0, h): out[0, :, h].float().numpy() for h in range(w.H)},
                 {(0, h): want[0, :, h] for h in range(w.H)}, "host forward")


def test_host_forward_single_group_layout(cuda):
    """A layout whose head slices are not one strided block ([B, H, L, D] physical) runs as one group."""
    w = configs.Workload("host_bhld", B=2, H=3, D=128, T=6, S=50, K=2, r=1, G=20, global_pos=1, seed=62)
    q, k, v = inputs.make_qkv(w, device="cuda")
    qs, ks, vs = (relayout(t, "bhld") for t in (q, k, v))
    want = device_forward(cuda, w, qs, ks, vs)
    qh, kh, vh = (t.cpu() for t in (qs, ks, vs))
    assert strides_of(qh) == strides_of(qs)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos, strides=strides_of(qs))
    try:
        got = plan.forward_host(qh, kh, vh)
        assert plan.check_error() == 0
    finally:
        plan.close()
    assert torch.equal(got, want)
