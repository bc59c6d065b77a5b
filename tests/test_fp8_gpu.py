"""Parity of the e4m3-score path (wa_forward_fp8) against the fp64 oracle on the dequantised inputs.

q and k are quantised per tensor to float8 e4m3 (scale = amax / 448, the format's largest finite value); the
oracle sees exactly the represented values, q_scale * q8 and k_scale * k8 (in float64), and the bf16 v. The bar
is the bf16 path's: per (b, h) relative Frobenius error <= 5e-3 and per-element absolute error <= 3e-2."""
import ctypes

import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

REL_TOL = 5e-3
ABS_TOL = 3e-2


def quantise(t):
    scale = float(t.float().abs().max()) / 448.0
    return (t.float() / scale).to(torch.float8_e4m3fn), scale


def check(got, want, label):
    worst_rel, worst_abs = 0.0, 0.0
    for key, w in want.items():
        g = got[key]
        worst_rel = max(worst_rel, np.linalg.norm(g - w) / np.linalg.norm(w))
        worst_abs = max(worst_abs, np.abs(g - w).max())
    assert worst_rel <= REL_TOL and worst_abs <= ABS_TOL, f"{label}: rel {worst_rel:.3e} abs {worst_abs:.3e}"


def run(wa, w, heads=None, chunks=None):
    q, k, v = inputs.make_qkv(w, device="cuda")
    q8, sq = quantise(q)
    k8, sk = quantise(k)
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out = plan.forward_fp8(q8, k8, v, sq, sk)
        assert plan.check_error() == 0
    finally:
        plan.close()
    qd = (q8.float() * sq).double().cpu()
    kd = (k8.float() * sk).double().cpu()
    vc = v.cpu()
    got_all = out.float().cpu().numpy()
    got, want = {}, {}
    if heads is None:
        full = ref.window_attention(qd, kd, vc, w.T, w.S, w.K, w.r, w.G, w.global_pos)
        for b in range(w.B):
            for h in range(w.H):
                got[(b, h)], want[(b, h)] = got_all[b, :, h], full[b, :, h]
    else:
        for h in heads:
            frames = [t for c in chunks for t in ref.chunk_frames(c, w.T, w.K)]
            res = ref.window_attention_rows(qd, kd, vc, w.T, w.S, w.K, w.r, w.G, w.global_pos, 0, h, frames=frames,
                                            global_rows=True)
            rows = sorted(res)
            want[(0, h)] = np.stack([res[r] for r in rows])
            got[(0, h)] = got_all[0, rows, h]
    check(got, want, w.name + " fp8")


@pytest.mark.parametrize("w", [configs.MEDIUM, configs.RAGGED,
                               configs.Workload("fp8_sharp", B=1, H=2, D=128, T=12, S=64, K=3, r=1, G=256,
                                                global_pos=0, seed=31, k_global_scale=4.0)],
                         ids=lambda w: w.name)
def test_fp8_full(cuda, w):
    run(cuda, w)


def test_fp8_h3_sampled(cuda):
    w = configs.H3
    run(cuda, w, heads=(0, 55), chunks=(0, w.nc // 2, w.nc - 1))


def test_fp8_rejects_bad_scales_and_head_dim(cuda):
    lib = cuda.lib()
    w = configs.TINY  # D = 64: the e4m3 path needs D = 128
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        buf = torch.zeros(w.B, w.L, w.H, w.D, dtype=torch.bfloat16, device="cuda")
        o = torch.empty_like(buf)
        P = ctypes.c_void_p
        args = (plan.handle, P(buf.data_ptr()), P(buf.data_ptr()), P(buf.data_ptr()), P(o.data_ptr()))
        assert lib.wa_forward_fp8(*args, 1.0, 1.0, None) == 2   # WA_ERR_UNSUPPORTED
        assert lib.wa_forward_fp8(*args, 0.0, 1.0, None) == 1   # WA_ERR_INVALID
        assert lib.wa_forward_fp8(*args, 1.0, float("nan"), None) == 1
    finally:
        plan.close()


def random_fp8_geometries(n, seed):
    """Seeded random geometries for the e4m3 path (D = 128): ragged chunks, both global placements, r past nc."""
    import random
    rnd = random.Random(seed)
    out = []
    for i in range(n):
        T = rnd.randint(1, 14)
        K = rnd.randint(1, 5)
        nc = -(-T // K)
        out.append(configs.Workload(f"fp8_rand{i}", B=rnd.randint(1, 2), H=rnd.randint(1, 3), D=128, T=T,
                                    S=rnd.randint(1, 97), K=K, r=rnd.randint(0, nc + 1),
                                    G=rnd.choice([0, 1, rnd.randint(2, 300)]), global_pos=rnd.randint(0, 1),
                                    seed=4000 + i))
    return out


@pytest.mark.parametrize("w", random_fp8_geometries(10, seed=9), ids=lambda w: w.name)
def test_fp8_random_geometries(cuda, w):
    run(cuda, w)
