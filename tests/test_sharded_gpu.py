"""Head ranges on one GPU: the heads of a layer computed range by range (as the ranks of a head-sharded run each
compute theirs) assemble into exactly the output of one call over every head, and a range matches the oracle."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs, sharded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [configs.MEDIUM, configs.RAGGED], ids=lambda w: w.name)
def test_head_ranges_assemble_to_full_call(cuda, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        full = plan.forward(q, k, v)
        assert plan.check_error() == 0
    finally:
        plan.close()
    for ranges in ([(h, 1) for h in range(w.H)], [(0, w.H // 2), (w.H // 2, w.H - w.H // 2)], [(0, 3), (3, w.H - 3)]):
        # in place: views of the full tensors (plan layout H = nh, the full strides, pointers at head h0)
        out = torch.full_like(q, float("nan"))
        for h0, nh in ranges:
            sharded.forward_heads(q, k, v, h0, nh, w.T, w.S, w.K, w.r, w.G, w.global_pos, out=out)
        assert torch.equal(out, full), f"{ranges}: strided head ranges"
        # as a head-sharded rank holds them: contiguous [B, L, nh, D] copies
        parts = []
        for h0, nh in ranges:
            sel = slice(h0, h0 + nh)
            p = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, nh, w.D, w.global_pos)
            try:
                parts.append(p.forward(q[:, :, sel].contiguous(), k[:, :, sel].contiguous(), v[:, :, sel].contiguous()))
            finally:
                p.close()
        assert torch.equal(torch.cat(parts, dim=2), full), f"{ranges}: contiguous head shards"


def test_head_range_matches_oracle(cuda):
    w = configs.RAGGED
    q, k, v = inputs.make_qkv(w, device="cuda")
    h0, nh = 5, 3
    out = sharded.forward_heads(q, k, v, h0, nh, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    sel = slice(h0, h0 + nh)
    want = ref.window_attention(q[:, :, sel].cpu(), k[:, :, sel].cpu(), v[:, :, sel].cpu(), w.T, w.S, w.K, w.r, w.G,
                                w.global_pos)
    got = out[:, :, sel].float().cpu().numpy()
    for b in range(w.B):
        for h in range(nh):
            x, y = got[b, :, h], want[b, :, h]
            assert np.linalg.norm(x - y) / np.linalg.norm(y) <= 5e-3 and np.abs(x - y).max() <= 3e-2


def test_sharded_forward_single_rank_is_the_plain_call(cuda):
    """One rank (no process group): sharded_forward is the plain forward of the whole layer."""
    w = configs.MEDIUM
    q, k, v = inputs.make_qkv(w, device="cuda")
    got = sharded.sharded_forward(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        assert torch.equal(got, plan.forward(q, k, v))
    finally:
        plan.close()
