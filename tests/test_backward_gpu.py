"""Backward-pass support of the CUDA path against the fp64 CPU oracle: the forward's row log-sum-exp output, and
the gradients dq, dk, dv of sum(out * dout).

Bars (float64 oracle on the same bf16 inputs):
  * lse: |lse_gpu - lse_ref| <= 2e-3 for every row (fp32 running sums over at most ~1e5 terms);
  * gradients: per (b, h) slice ||g_gpu - g_ref||_F / ||g_ref||_F <= 5e-3 and max |g_gpu - g_ref| <= 2e-2 *
    max |g_ref|: the forward's relative bar. dS and P enter the tensor-core products as bf16, one rounding more
    than the forward; the measured worst cases are 3.9e-3 relative and 6.9e-3 of the slice maximum (the sharpened
    global keys), about 2.4e-3 and 3-5e-3 elsewhere.
"""
import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

LSE_TOL = 2e-3


def gpu_lse(wa, w, q, k, v):
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        out_plain = plan.forward(q, k, v)
        assert plan.check_error() == 0
        assert torch.equal(out, out_plain), "the lse output must not change the forward result"
    finally:
        plan.close()
    return lse.cpu().double().numpy()


LSE_CASES = [configs.TINY, configs.MEDIUM, configs.RAGGED,
             configs.Workload("lse_front_d64", B=2, H=2, D=64, T=10, S=60, K=3, r=1, G=130, global_pos=1, seed=31),
             configs.Workload("lse_many_splits", B=1, H=2, D=128, T=40, S=64, K=1, r=0, G=300, global_pos=0, seed=32)]


@pytest.mark.parametrize("w", LSE_CASES, ids=lambda w: w.name)
def test_forward_lse_full(cuda, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    got = gpu_lse(cuda, w, q, k, v)
    want = ref.row_logsumexp(q, k, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    err = np.abs(got - want).max()
    assert err <= LSE_TOL, f"{w.name}: max |lse error| {err:.3e}"


# --------------------------------------------------------------------------------------------------- gradients
GRAD_REL = 5e-3
GRAD_ABS = 2e-2  # times max |reference| of the slice


def gpu_backward(wa, w, q, k, v, dout):
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        dq, dk, dv = plan.backward(q, k, v, out, dout, lse)
        assert plan.check_error() == 0
    finally:
        plan.close()
    return dq, dk, dv


def check_grads(got, want, label):
    """got: (dq, dk, dv) GPU tensors; want: float64 arrays. The bar applies per (b, h) slice and tensor."""
    worst = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, want):
        g = g.float().cpu().double().numpy()
        for b in range(r.shape[0]):
            for h in range(r.shape[2]):
                gs, rs = g[b, :, h], r[b, :, h]
                rel = np.linalg.norm(gs - rs) / max(np.linalg.norm(rs), 1e-30)
                ab = np.abs(gs - rs).max() / max(np.abs(rs).max(), 1e-30)
                wr, wa_ = worst.get(name, (0.0, 0.0))
                worst[name] = (max(wr, rel), max(wa_, ab))
    msg = ", ".join(f"{n}: rel {a:.2e} abs {b:.2e}" for n, (a, b) in worst.items())
    print(f"{label}: {msg}")
    for n, (rel, ab) in worst.items():
        assert rel <= GRAD_REL and ab <= GRAD_ABS, f"{label} {n}: {msg}"


GRAD_CASES = [
    configs.TINY,
    configs.MEDIUM,
    configs.Workload("bwd_ragged", B=2, H=2, D=128, T=50, S=60, K=4, r=2, G=77, global_pos=1, seed=41),
    configs.Workload("bwd_no_globals", B=1, H=2, D=128, T=9, S=100, K=2, r=1, G=0, global_pos=0, seed=42),
    configs.Workload("bwd_many_splits", B=1, H=2, D=128, T=40, S=64, K=1, r=0, G=300, global_pos=0, seed=43),
    configs.Workload("bwd_d64_front", B=2, H=2, D=64, T=13, S=37, K=4, r=2, G=130, global_pos=1, seed=44),
    configs.Workload("bwd_one_token_frames", B=1, H=2, D=128, T=300, S=1, K=7, r=2, G=5, global_pos=1, seed=45),
    configs.Workload("bwd_single_row", B=1, H=1, D=128, T=1, S=1, K=1, r=0, G=0, global_pos=0, seed=46),
    configs.Workload("bwd_radius_covers_all", B=1, H=2, D=128, T=7, S=90, K=2, r=9, G=40, global_pos=0, seed=47),
    configs.Workload("bwd_sharp_globals", B=1, H=2, D=128, T=12, S=64, K=3, r=1, G=256, global_pos=0, seed=48,
                     k_global_scale=4.0),
    # at least 1024 global rows: doubled split length (2 splits), partial last global tile
    configs.Workload("bwd_long_globals", B=1, H=2, D=128, T=40, S=64, K=1, r=0, G=1100, global_pos=0, seed=49),
    # B*H*L not a multiple of 4 (1 and 3 mod 4; bwd_one_token_frames has 2 mod 4): the split partials of the global
    # rows, written with 16-byte stores, sit behind the B*H*L fp32 row dots in one workspace and must still start on
    # a 16-byte boundary
    configs.Workload("bwd_rows_1_mod_4", B=1, H=1, D=128, T=4, S=41, K=2, r=1, G=5, global_pos=0, seed=54),
    configs.Workload("bwd_rows_3_mod_4_d64", B=1, H=3, D=64, T=7, S=13, K=3, r=0, G=2, global_pos=1, seed=55),
]


@pytest.mark.parametrize("w", GRAD_CASES, ids=lambda w: w.name)
def test_backward_full(cuda, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    got = gpu_backward(cuda, w, q, k, v, dout)
    want = ref.window_attention_backward(q, k, v, dout, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    check_grads(got, want, w.name)


def test_backward_deterministic_and_streams(cuda):
    w = configs.MEDIUM
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        a = plan.backward(q, k, v, out, dout, lse)
        s2 = torch.cuda.Stream()
        with torch.cuda.stream(s2):
            b = plan.backward(q, k, v, out, dout, lse)
        torch.cuda.synchronize()
        assert plan.check_error() == 0
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    finally:
        plan.close()


def test_backward_matches_autograd_of_dense_masked_attention(cuda):
    """Independent of the oracle's loop: torch autograd (float64, CPU) through dense attention with the kept-set
    mask built by brute force from the chunk rule."""
    w = configs.Workload("bwd_dense", B=1, H=2, D=64, T=8, S=20, K=2, r=1, G=24, global_pos=0, seed=49)
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    got = gpu_backward(cuda, w, q, k, v, dout)
    L = w.L
    chunk = [(i // w.S) // w.K if i < w.F else -1 for i in range(L)]
    mask = torch.zeros(L, L, dtype=torch.bool)
    for i in range(L):
        for j in range(L):
            mask[i, j] = chunk[i] < 0 or chunk[j] < 0 or abs(chunk[i] - chunk[j]) <= w.r
    qd, kd, vd = (t.double().cpu().requires_grad_(True) for t in (q, k, v))
    s = torch.einsum("blhd,bmhd->bhlm", qd, kd) / np.sqrt(w.D)
    p = torch.softmax(s.masked_fill(~mask, float("-inf")), dim=-1)
    o = torch.einsum("bhlm,bmhd->blhd", p, vd)
    (o * dout.double().cpu()).sum().backward()
    check_grads(got, [t.grad.numpy() for t in (qd, kd, vd)], "dense autograd")


@pytest.mark.parametrize("flag", [2, 4], ids=["dq_kernel", "dkdv_kernel"])
def test_backward_watchdog(cuda, flag):
    """A copy that never arrives: the bounded wait expires, the kernel unwinds and the error is reported; the next
    backward on the same plan is correct."""
    w = configs.Workload("bwd_watchdog", B=1, H=2, D=128, T=6, S=64, K=2, r=1, G=32, global_pos=0, seed=50)
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        plan.set_debug_flags(flag)
        plan.backward(q, k, v, out, dout, lse)
        assert plan.check_error() == 5  # WA_ERR_DEVICE_TIMEOUT
        plan.set_debug_flags(0)
        got = plan.backward(q, k, v, out, dout, lse)
        assert plan.check_error() == 0
    finally:
        plan.close()
    want = ref.window_attention_backward(q, k, v, dout, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    check_grads(got, want, "after watchdog")


def test_backward_h3_sampled(cuda):
    """The full H3 layer (56 heads, L = 99,968) in the benchmark's launch configuration; the oracle checks one head
    on a sample: dq of chunk 0, a middle chunk and all global rows; dk, dv of the keys of a middle chunk (each
    needs every query that keeps it: three chunks of frames and all global queries)."""
    w = configs.H3
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    got = gpu_backward(cuda, w, q, k, v, dout)
    h = 27
    qh, kh, vh, doh = (t[:, :, h:h + 1].cpu() for t in (q, k, v, dout))
    gq, gk, gv = (t[0, :, h].float().cpu().double().numpy() for t in got)
    del q, k, v, dout, got
    mid = w.nc // 2
    q_frames = ref.chunk_frames(0, w.T, w.K) + ref.chunk_frames(mid, w.T, w.K)
    k_frames = ref.chunk_frames(mid, w.T, w.K)
    rdq, rdk, rdv = ref.window_attention_backward_rows(qh, kh, vh, doh, w.T, w.S, w.K, w.r, w.G, w.global_pos, 0, 0,
                                                       q_frames=q_frames, global_q=True, k_frames=k_frames)
    for name, g, ref_rows in (("dq", gq, rdq), ("dk", gk, rdk), ("dv", gv, rdv)):
        rows = sorted(ref_rows)
        want = np.stack([ref_rows[r] for r in rows])
        have = g[rows]
        rel = np.linalg.norm(have - want) / np.linalg.norm(want)
        ab = np.abs(have - want).max() / np.abs(want).max()
        print(f"h3 {name} ({len(rows)} rows): rel {rel:.2e} abs {ab:.2e}")
        assert rel <= GRAD_REL and ab <= GRAD_ABS, f"h3 {name}: rel {rel:.3e} abs {ab:.3e}"


@pytest.mark.parametrize("kind", ["bhld", "padded"])
def test_backward_strided_layouts(cuda, kind):
    """The plan's strides apply to every tensor of the backward: q, k, v, out, dout and the three gradients."""
    from test_parity_gpu import relayout, strides_of
    w = configs.Workload("bwd_strided", B=2, H=3, D=128, T=6, S=50, K=2, r=1, G=20, global_pos=1, seed=51)
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    qs, ks, vs, ds = (relayout(t, kind) for t in (q, k, v, dout))
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos, strides=strides_of(qs))
    try:
        out, lse = plan.forward_lse(qs, ks, vs)
        grads = plan.backward(qs, ks, vs, out, ds, lse)
        assert plan.check_error() == 0
        assert all(tuple(g.stride()) == tuple(qs.stride()) for g in grads)
    finally:
        plan.close()
    want = ref.window_attention_backward(q, k, v, dout, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    check_grads(grads, want, f"strided {kind}")


def test_backward_argument_errors(cuda):
    """Synchronous argument checks: nothing is launched for a misaligned pointer or outputs that overlap inputs."""
    w = configs.TINY
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        s = torch.cuda.current_stream().cuda_stream
        args = [q, k, v, out, dout, lse, dq, dk, dv]
        ptrs = [t.data_ptr() for t in args]
        bad = list(ptrs)
        bad[0] += 2  # q misaligned
        with pytest.raises(cuda.WAError):
            cuda.wa_backward(plan.handle, *bad, s)
        bad = list(ptrs)
        bad[6] = ptrs[7]  # dq overlaps dk
        with pytest.raises(cuda.WAError):
            cuda.wa_backward(plan.handle, *bad, s)
        bad = list(ptrs)
        bad[8] = ptrs[0]  # dv overlaps q
        with pytest.raises(cuda.WAError):
            cuda.wa_backward(plan.handle, *bad, s)
        cuda.wa_backward(plan.handle, *ptrs, s)  # the valid call still works
        assert plan.check_error() == 0
    finally:
        plan.close()


@pytest.mark.parametrize("w", __import__("test_parity_gpu").random_geometries(12, seed=8), ids=lambda w: w.name)
def test_backward_random_geometries(cuda, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    got = gpu_backward(cuda, w, q, k, v, dout)
    want = ref.window_attention_backward(q, k, v, dout, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    check_grads(got, want, w.name)
