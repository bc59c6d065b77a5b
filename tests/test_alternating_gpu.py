"""Items with a single query tile run with alternating key tiles: key tile j goes to tile slot j % 2 and the two
halves are merged by log-sum-exp in the epilogue. These geometries are chosen so that the plan mixes, on every
CTA, two-tile items, alternating items with an even and an odd number of key tiles (slot 0 then takes one more),
alternating global-split items, and single-tile items with one key tile (which run alone); they are compared
with the fp64 oracle for the output (bf16 and e4m3 scores) and the row log-sum-exp."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs

REL_TOL, ABS_TOL, LSE_TOL = 5e-3, 3e-2, 2e-3

CASES = [
    # groups of 300 rows: one two-tile item and one of 44 rows, against 3 or 4 key tiles (the first group's window
    # touches the globals); the 50 global rows: one tile against four splits of 4 key tiles (alternating) and a
    # last split of 1 (alone); 32 heads: 608 items on 152 CTAs
    configs.Workload("alt_mixed", B=1, H=32, D=128, T=7, S=300, K=1, r=0, G=50, global_pos=1, seed=81),
    # groups of 64 rows (single tiles) over windows of 2 or 3 chunks of 64 rows: 1-2 key tiles per segment
    configs.Workload("alt_short", B=2, H=8, D=128, T=12, S=64, K=1, r=1, G=20, global_pos=0, seed=82),
    # D = 64; single-tile groups whose key range is one tile (the lone path) next to alternating ones
    configs.Workload("alt_d64", B=1, H=16, D=64, T=9, S=40, K=2, r=0, G=24, global_pos=1, seed=83),
]


def describe_kinds(wa, w):
    lay = wa.make_layout(w.B, w.L, w.H, w.D, w.global_pos)
    _, _, items = wa.wa_geometry_describe(w.T, w.S, w.K, w.r, w.G, lay, with_items=True)
    kinds = set()
    for bh, kind, qlo, qhi, a, b, c, d in items:
        nt = sum(-(-(hi - lo) // 128) for lo, hi in ((a, b), (c, d)) if hi > lo)
        kinds.add(("pair" if qhi - qlo > 128 else ("alternating" if nt >= 2 else "lone"), kind, nt % 2))
    return kinds


def test_cases_hold_the_intended_item_kinds(walib):
    every = set().union(*(describe_kinds(walib, w) for w in CASES))
    assert {k[0] for k in every} == {"pair", "alternating", "lone"}
    assert ("alternating", 0, 0) in every and ("alternating", 0, 1) in every  # even and odd key-tile counts
    assert any(k[:2] == ("alternating", 1) for k in every)  # global-split items alternate too
    k0 = describe_kinds(walib, CASES[0])
    assert {k[0] for k in k0} == {"pair", "alternating", "lone"}  # all three kinds in one launch


def compare(got, want, label):
    worst_rel = worst_abs = 0.0
    for key in want:
        g, r = got[key], want[key]
        worst_rel = max(worst_rel, np.linalg.norm(g - r) / np.linalg.norm(r))
        worst_abs = max(worst_abs, np.abs(g - r).max())
    assert worst_rel <= REL_TOL and worst_abs <= ABS_TOL, f"{label}: rel {worst_rel:.3e} abs {worst_abs:.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_alternating_items_bf16_and_lse(cuda, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    check_bf16_and_lse(cuda, w, q, k, v)


# Hot scores: q and k times 4 (exact in bf16), so the scores' standard deviation is 16 and the lazy reference max
# is raised again and again: in pair items, in both halves of alternating items (whose halves then merge across
# very different references) and in the global splits.
HOT = configs.Workload("alt_hot", B=1, H=4, D=128, T=10, S=150, K=2, r=1, G=200, global_pos=0, seed=84)


def test_hot_case_holds_alternating_items(walib):
    assert {k[0] for k in describe_kinds(walib, HOT)} >= {"pair", "alternating"}


@pytest.mark.gpu
def test_hot_scores_bf16_and_lse(cuda):
    w = HOT
    q, k, v = inputs.make_qkv(w, device="cuda")
    check_bf16_and_lse(cuda, w, q * 4, k * 4, v)


def check_bf16_and_lse(cuda, w, q, k, v):
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        again = plan.forward(q, k, v)
        assert plan.check_error() == 0
    finally:
        plan.close()
    assert torch.equal(out, again)
    want = ref.window_attention(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    got = out.float().cpu().numpy()
    compare({(b, h): got[b, :, h] for b in range(w.B) for h in range(w.H)},
            {(b, h): want[b, :, h] for b in range(w.B) for h in range(w.H)}, w.name)
    want_lse = ref.row_logsumexp(q, k, w.T, w.S, w.K, w.r, w.G, w.global_pos)
    err = np.abs(lse.cpu().double().numpy() - want_lse).max()
    assert err <= LSE_TOL, f"{w.name}: max |lse error| {err:.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("w", [c for c in CASES if c.D == 128], ids=lambda w: w.name)
def test_alternating_items_e4m3(cuda, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    sq = float(q.float().abs().max()) / 448.0
    sk = float(k.float().abs().max()) / 448.0
    q8 = (q.float() / sq).to(torch.float8_e4m3fn)
    k8 = (k.float() / sk).to(torch.float8_e4m3fn)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out = plan.forward_fp8(q8, k8, v, sq, sk)
        assert plan.check_error() == 0
    finally:
        plan.close()
    qd = (q8.float() * sq).double().cpu()
    kd = (k8.float() * sk).double().cpu()
    want = ref.window_attention(qd, kd, v.cpu(), w.T, w.S, w.K, w.r, w.G, w.global_pos)
    got = out.float().cpu().numpy()
    compare({(b, h): got[b, :, h] for b in range(w.B) for h in range(w.H)},
            {(b, h): want[b, :, h] for b in range(w.B) for h in range(w.H)}, w.name + " e4m3")
