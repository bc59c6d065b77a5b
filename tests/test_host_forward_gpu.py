"""wa_forward_host: the forward on host buffers, pipelined over pieces of the sequence (copies in, compute, copies out
on separate streams; each launch runs the work items whose rows have arrived). Its results must equal the
device-resident forward bit for bit (the same kernels and work items, only regrouped by launch), and therefore the
fp64 oracle within the forward's bar."""
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs
from test_parity_gpu import check_slices, relayout, strides_of

pytestmark = pytest.mark.gpu


def prime_with_nan(plan, q):
    """Run one host forward on all-NaN inputs, so that the plan's device staging holds NaN wherever the next call has
    not copied its own rows yet: a launch that reads a row before it has arrived then shows NaN in its output."""
    nan = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, pin_memory=q.is_pinned()).fill_(float("nan"))
    plan.forward_host(nan, nan, nan)
    assert plan.check_error() == 0


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
        prime_with_nan(plan, qh)
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


def host_layout(t, kind):
    """Same logical [B, L, H, D] tensor in a physical layout whose rows are still one block of heads."""
    B, L, H, D = t.shape
    if kind == "rowpad":  # rows padded to a larger pitch, heads adjacent inside a row
        big = torch.zeros(B, L, H * D + 64, dtype=t.dtype, device=t.device)
        big[:, :, :H * D] = t.reshape(B, L, H * D)
        return big[:, :, :H * D].unflatten(2, (H, D))
    if kind == "lbhd":  # batch entries interleaved between sequence rows
        return t.permute(1, 0, 2, 3).contiguous().permute(1, 0, 2, 3)
    raise ValueError(kind)


PIECE_CASES = [
    (configs.Workload("host_no_globals", B=1, H=2, D=128, T=9, S=100, K=2, r=1, G=0, global_pos=0, seed=63), None),
    (configs.Workload("host_radius_covers_all", B=1, H=2, D=128, T=7, S=90, K=2, r=9, G=40, global_pos=0, seed=64),
     None),
    (configs.Workload("host_radius0_front", B=2, H=2, D=64, T=8, S=70, K=3, r=0, G=200, global_pos=1, seed=65), None),
    (configs.Workload("host_one_token_frames", B=1, H=3, D=128, T=300, S=1, K=7, r=2, G=5, global_pos=1, seed=66),
     None),
    (configs.Workload("host_rowpad", B=2, H=3, D=128, T=11, S=40, K=2, r=2, G=24, global_pos=0, seed=67), "rowpad"),
    (configs.Workload("host_lbhd", B=2, H=2, D=64, T=10, S=30, K=3, r=1, G=16, global_pos=1, seed=68), "lbhd"),
    (configs.Workload("host_one_head_rowpad", B=1, H=1, D=128, T=12, S=33, K=1, r=3, G=7, global_pos=0, seed=69),
     "rowpad"),
    (configs.Workload("host_long_globals", B=1, H=8, D=128, T=40, S=64, K=1, r=0, G=1100, global_pos=0, seed=70),
     None),  # the host path's 2 global splits against the device plan's 1; the head ranges of the first and last
             # pieces merge their global rows separately
]


def same_lists(cuda, w, strides):
    """Whether the host path runs the device plan's work list (it keeps shorter global splits when the global rows
    are plentiful)."""
    lay = cuda.make_layout(w.B, w.L, w.H, w.D, w.global_pos, strides)
    _, _, dev = cuda.wa_geometry_describe(w.T, w.S, w.K, w.r, w.G, lay, with_items=True)
    return cuda.wa_host_schedule_describe(w.T, w.S, w.K, w.r, w.G, lay)["items"] == dev


def check_against_device(cuda, w, got, want, strides):
    """Bit for bit when the two lists are the same; otherwise the frame rows bit for bit and the global rows (whose
    split merge differs) within the oracle bar of the parity tests."""
    if same_lists(cuda, w, strides):
        assert torch.equal(got, want)
        return
    g0 = 0 if w.global_pos else w.T * w.S
    frames = torch.ones(w.L, dtype=torch.bool)
    frames[g0:g0 + w.G] = False
    assert torch.equal(got[:, frames], want[:, frames])
    for b in range(w.B):
        for h in range(w.H):
            a = got[b, g0:g0 + w.G, h].double()
            r = want[b, g0:g0 + w.G, h].double()
            assert (a - r).norm() / r.norm() <= 5e-3 and (a - r).abs().max() <= 3e-2


@pytest.mark.parametrize("w,kind", PIECE_CASES, ids=[c[0].name for c in PIECE_CASES])
def test_host_forward_pieces(cuda, w, kind):
    """Geometries and row layouts that change the pieces: no globals, one group, front globals, many small chunks,
    padded rows, batch entries between rows, a single head."""
    q, k, v = inputs.make_qkv(w, device="cuda")
    if kind is not None:
        q, k, v = (host_layout(t, kind) for t in (q, k, v))
    want = device_forward(cuda, w, q, k, v)
    qh, kh, vh = (torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, pin_memory=True) for t in (q, k, v))
    for h, d in zip((qh, kh, vh), (q, k, v)):
        h.copy_(d)
    assert strides_of(qh) == strides_of(q)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos, strides=strides_of(q))
    try:
        prime_with_nan(plan, qh)
        got = plan.forward_host(qh, kh, vh)
        assert plan.check_error() == 0
    finally:
        plan.close()
    check_against_device(cuda, w, got, want.cpu() if want.is_cuda else want, strides_of(q))
