"""Backward-pass support of the CUDA path against the fp64 CPU oracle: the forward's row log-sum-exp output, and
the gradients dq, dk, dv of sum(out * dout).

Bars (float64 oracle on the same bf16 inputs):
  * lse: |lse_gpu - lse_ref| <= 2e-3 for every row (fp32 running sums over at most ~1e5 terms);
  * gradients: per (b, h) slice ||g_gpu - g_ref||_F / ||g_ref||_F <= 1e-2 and max |g_gpu - g_ref| <= 5e-2 *
    max |g_ref| (dS and P enter the tensor-core products as bf16, one rounding more than the forward).
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
