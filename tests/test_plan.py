"""The host-side plan (C++, through the C ABI's host-only wa_geometry_describe), checked on the CPU against a
Python restatement of the grouping rule and against the oracle's kept sets."""
import random

import numpy as np
import pytest

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs


def groups_restated(T, S, K, r, G, gp):
    """Chunks with identical clamped windows merge into one group (VDN-Minimax-H3 article, section 三)."""
    nc = -(-T // K)
    f0, g0 = (G, 0) if gp else (0, T * S)
    out = []
    for c in range(nc):
        lo, hi = max(0, c - r), min(nc - 1, c + r)
        q = (f0 + c * K * S, f0 + min(T, (c + 1) * K) * S)
        kv = (f0 + lo * K * S, f0 + min(T, (hi + 1) * K) * S)
        if out and out[-1][2] == (lo, hi):
            out[-1][0] = (out[-1][0][0], q[1])
        else:
            out.append([q, kv, (lo, hi)])
    return [(q, kv) for q, kv, _ in out]


def describe(wa, T, S, K, r, G, gp, B=1, H=1, D=128, items=False):
    lay = wa.make_layout(B, T * S + G, H, D, gp)
    return wa.wa_geometry_describe(T, S, K, r, G, lay, with_items=items)


GEOS = [(6, 16, 2, 1, 8, 0), (24, 256, 4, 1, 256, 0), (50, 300, 4, 2, 77, 1), (102, 960, 3, 1, 2048, 0),
        (7, 5, 3, 2, 4, 1), (5, 3, 7, 0, 2, 0), (9, 4, 2, 9, 3, 1), (12, 2, 1, 0, 0, 0), (11, 130, 2, 1, 129, 1)]


@pytest.mark.parametrize("geo", GEOS)
def test_groups_match_restatement(walib, geo):
    T, S, K, r, G, gp = geo
    info, groups, _ = describe(walib, *geo)
    want = groups_restated(*geo)
    assert info["n_groups"] == len(want)
    f0, g0 = (G, 0) if gp else (0, T * S)
    for g, (q, kv) in zip(groups, want):
        assert (g["q_lo"], g["q_hi"]) == q
        segs = sorted([(g["kv0_lo"], g["kv0_hi"]), (g["kv1_lo"], g["kv1_hi"])])
        segs = [s for s in segs if s[1] > s[0]]
        # the union of the segments is the frame window plus the globals, with no overlap
        cover = np.zeros(T * S + G, dtype=int)
        for lo, hi in segs:
            cover[lo:hi] += 1
        expect = np.zeros(T * S + G, dtype=int)
        expect[kv[0]:kv[1]] = 1
        expect[g0:g0 + G] = 1
        np.testing.assert_array_equal(cover, expect)


def random_geos(n, seed):
    rnd = random.Random(seed)
    return [(rnd.randint(1, 40), rnd.randint(1, 300), rnd.randint(1, 6), rnd.randint(0, 3), rnd.randint(0, 300),
             rnd.randint(0, 1)) for _ in range(n)]


@pytest.mark.parametrize("geo", GEOS + random_geos(12, 5))
def test_items_cover_every_row_once_with_its_kept_set(walib, geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    B, H = 2, 3
    info, _, items = describe(walib, *geo, B=B, H=H, items=True)
    f0, g0 = (G, 0) if gp else (0, T * S)
    # window rows: exactly one item per (bh, row); global rows: exactly one item per (bh, row, split)
    win = np.zeros((B * H, L), dtype=int)
    glob = {}
    for bh, kind, qlo, qhi, a, b, c, d in items:
        assert 0 < qhi - qlo <= 256
        segs = [(a, b), (c, d)]
        keys = np.zeros(L, dtype=bool)
        for lo, hi in segs:
            assert not keys[lo:hi].any()
            keys[lo:hi] = True
        if kind == 0:
            win[bh, qlo:qhi] += 1
            # every row of the item has exactly this kept set (rows with identical kept sets form a group)
            for row in (qlo, qhi - 1):
                t = (row - f0) // S
                want = np.zeros(L, dtype=bool)
                want[ref.kept_set_of_frame(t, T, S, K, r, G, gp)] = True
                np.testing.assert_array_equal(keys, want)
        else:
            assert g0 <= qlo and qhi <= g0 + G
            glob.setdefault((bh, qlo, qhi), np.zeros(L, dtype=int))
            glob[(bh, qlo, qhi)][keys] += 1
    assert (win[:, f0:f0 + T * S] == 1).all()
    assert win[:, g0:g0 + G].sum() == 0
    if G:
        rows = np.zeros((B * H, L), dtype=int)
        for (bh, qlo, qhi), cover in glob.items():
            assert (cover == 1).all()  # the splits of one global tile cover every key exactly once
            rows[bh, qlo:qhi] += 1
        assert (rows[:, g0:g0 + G] == 1).all()
    else:
        assert not glob
    assert info["n_splits"] >= 1


@pytest.mark.parametrize("w", [configs.TINY, configs.MEDIUM, configs.H3, configs.RAGGED] + configs.sweep()[::5])
def test_kept_pairs_match_oracle(walib, w):
    info, _, _ = describe(walib, w.T, w.S, w.K, w.r, w.G, w.global_pos, B=w.B, H=w.H, D=w.D)
    assert info["kept_pairs"] == ref.kept_pairs(w.T, w.S, w.K, w.r, w.G, w.global_pos)
    assert info["global_pairs"] == w.G * w.L
    assert info["L"] == w.L
    assert info["n_chunks"] == w.nc


def test_h3_plan_shape(walib):
    w = configs.H3
    info, groups, _ = describe(walib, w.T, w.S, w.K, w.r, w.G, w.global_pos, B=w.B, H=w.H, D=w.D)
    assert info["n_groups"] == 34  # 102 latent frames / 3 per chunk; every chunk has a distinct window
    assert all(g["q_hi"] - g["q_lo"] == 2880 for g in groups)
    # the last window touches the globals at the back: one contiguous key segment
    assert (groups[-1]["kv1_hi"] - groups[-1]["kv1_lo"]) == 0 and groups[-1]["kv0_hi"] == w.L
    assert info["workspace_bytes"] == w.B * w.H * w.G * info["n_splits"] * (w.D + 1) * 4


def test_radius_beyond_chunks_is_one_group(walib):
    info, groups, _ = describe(walib, 10, 7, 3, 5, 4, 0)
    assert info["n_groups"] == 1
    assert (groups[0]["q_lo"], groups[0]["q_hi"]) == (0, 70)


def test_profile_summaries_parse():
    """bench.py reads the kernel-source hash and the DRAM traffic from the committed ncu summaries."""
    import os
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    for path, key in ((bench.PROFILE_SUMMARY, "dram bytes per full H3 launch"),
                      (bench.BWD_PROFILE_SUMMARY, "dk/dv dram bytes per full H3 launch"),
                      (bench.FP8_PROFILE_SUMMARY, "dram bytes per full H3 launch")):
        fields = bench.profile_fields(path)
        assert len(fields["kernel source sha256[:16]"]) == 16
        assert float(fields[key]) > 1e9
