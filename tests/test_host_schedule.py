"""The host-buffer forward's piece schedule (host only, no GPU).

The sequence is copied in as pieces (blocks of rows x heads) and launch p runs after piece p has arrived, so the
schedule is correct when
- the pieces partition the rows [0, L) x heads [0, H) (every element copied exactly once), the global rows first;
- every work item runs in the launch of the latest piece holding a row it reads for its head, where the kernel
  reads whole 128-row tiles from the start of each of its ranges (q rows, key segment 0, key segment 1; rows past L
  read as zeros): earlier would read rows that have not arrived, later would stall the pipeline;
- every frame row of out is copied back exactly once per head, after every item that writes it has run (the
  global rows are copied after the merge);
and it pipelines: at H3 sizes one piece per window group, with the first group's rows and the globals split into
two head ranges (the first launch starts after half of that copy) and the last frame piece into four (each
quarter's global rows are merged and copied back right behind its launch).
"""
import numpy as np
import pytest

import chunk_windowed_softmax_gb300 as wa
from chunk_windowed_softmax_gb300 import configs

TILE = 128


def describe(T, S, K, r, G, B, H, D, global_pos, strides=None):
    L = T * S + G
    layout = wa.make_layout(B, L, H, D, global_pos, strides)
    info, groups, _ = wa.wa_geometry_describe(T, S, K, r, G, layout, with_groups=True)
    sched = wa.wa_host_schedule_describe(T, S, K, r, G, layout)
    return L, info, groups, sched["items"], sched


def read_ranges(item, L):
    """Rows the kernel reads for one work item: whole tiles from the start of each range, capped at L."""
    out = []
    for lo, hi in ((item[2], item[3]), (item[4], item[5]), (item[6], item[7])):
        if hi > lo:
            out.append((lo, min(L, lo + -(-(hi - lo) // TILE) * TILE)))
    return out


def check_schedule(T, S, K, r, G, B, H, D, global_pos, strides=None):
    L, info, groups, items, sched = describe(T, S, K, r, G, B, H, D, global_pos, strides)
    pieces, launch = sched["pieces"], sched["item_launch"]
    F = T * S
    g0, f0 = (0, G) if global_pos else (F, 0)
    # pieces partition [0, L) x [0, H)
    piece_of = np.full((L, H), -1, dtype=np.int32)
    for p, (lo, hi, h_lo, h_hi) in enumerate(pieces):
        assert 0 <= lo < hi <= L and 0 <= h_lo < h_hi <= H
        assert (piece_of[lo:hi, h_lo:h_hi] == -1).all(), "pieces overlap"
        piece_of[lo:hi, h_lo:h_hi] = p
    assert (piece_of >= 0).all(), "an element is never copied"
    if sched["row_pieces"] and G > 0:
        assert pieces[0][:2] == (g0, g0 + G) and pieces[0][2] == 0
    # each item runs exactly when the last piece it reads (for its head) has arrived
    assert len(launch) == len(items)
    for it, p in zip(items, launch):
        h = it[0] % H
        need = max(int(piece_of[lo:hi, h].max()) for lo, hi in read_ranges(it, L))
        assert p == need, (it, p, need)
    # out: every row of each head copied back once, after all its writers (a global row: after every split item of
    # its head, whose partial outputs the merge reads)
    if sched["row_pieces"]:
        copied = np.full((L, H), -1, dtype=np.int32)
        for p, lo, hi, h_lo, h_hi in sched["out"]:
            assert 0 <= lo < hi <= L and 0 <= h_lo < h_hi <= H
            assert (lo, hi) == (g0, g0 + G) or f0 <= lo < hi <= f0 + F
            assert (copied[lo:hi, h_lo:h_hi] == -1).all(), "a block of out is copied back twice"
            copied[lo:hi, h_lo:h_hi] = p
        assert (copied >= 0).all(), "a row of out is never copied back"
        for it, p in zip(items, launch):
            rows = slice(it[2], it[3]) if it[1] == 0 else slice(g0, g0 + G)
            assert (copied[rows, it[0] % H] >= p).all(), "out rows copied back before an item they need ran"
    else:
        assert pieces == [(0, L, 0, H)] and sched["out"] == [] and set(launch) <= {0}
    return L, info, groups, sched


GEOMETRIES = [
    (6, 16, 2, 1, 8, 1, 2, 64, 0),        # Tiny
    (24, 256, 4, 1, 256, 1, 8, 128, 0),   # Medium
    (50, 300, 4, 2, 77, 2, 16, 128, 1),   # Ragged (front globals, two batch entries)
    (9, 100, 2, 1, 0, 1, 2, 128, 0),      # no globals
    (7, 90, 2, 9, 40, 1, 2, 128, 0),      # the radius covers every chunk: one group
    (8, 70, 3, 0, 200, 2, 2, 64, 1),      # radius 0, front globals
    (3, 50, 5, 1, 9, 1, 2, 128, 0),       # one chunk longer than T
    (300, 1, 7, 2, 5, 1, 3, 128, 1),      # one-token frames
    (11, 40, 2, 2, 24, 2, 3, 128, 0),
    (5, 200, 1, 0, 300, 1, 1, 64, 0),     # r = 0: each group's last query tile reads past its own chunk
    (40, 64, 1, 0, 1100, 1, 8, 128, 0),   # 1100 global rows: doubled split length, per-head-range merges
]


@pytest.mark.parametrize("geo", GEOMETRIES, ids=lambda g: "T{}_S{}_K{}_r{}_G{}_B{}_H{}_D{}_p{}".format(*g))
def test_schedule_is_valid(geo):
    check_schedule(*geo)


def test_schedule_row_padded_and_batch_interleaved_layouts():
    T, S, K, r, G, B, H, D = 11, 40, 2, 2, 24, 2, 3, 128
    L = T * S + G
    check_schedule(T, S, K, r, G, B, H, D, 0, strides=(L * (H * D + 64), H * D + 64, D))  # padded rows
    check_schedule(T, S, K, r, G, B, H, D, 1, strides=(H * D, B * H * D, D))  # batch entries between rows


def test_schedule_single_piece_when_heads_are_not_adjacent():
    T, S, K, r, G, B, H, D = 6, 50, 2, 1, 20, 2, 3, 128
    L = T * S + G
    _, _, _, sched = check_schedule(T, S, K, r, G, B, H, D, 1, strides=(H * L * D, D, L * D))  # [B, H, L, D]
    assert not sched["row_pieces"]


def test_schedule_pipelines_h3():
    w = configs.H3
    L, info, groups, sched = check_schedule(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    KS = w.K * w.S
    pieces = sched["pieces"]
    assert sched["row_pieces"]
    half = w.H // 2
    # the globals and the first window group's rows, each in two head ranges, alternating so that the first
    # group's first heads can start after half of that copy
    assert [p[2:] for p in pieces[:4]] == [(0, half), (0, half), (half, w.H), (half, w.H)]
    assert pieces[0][:2] == pieces[2][:2] == (w.L - w.G, w.L)
    first = pieces[1][:2]
    assert pieces[3][:2] == first and first[0] == 0 and (w.r + 1) * KS <= first[1] <= (w.r + 1) * KS + TILE
    # then one piece per window group (all heads), ending where its reads end; the last two groups (windows
    # [31, 33] and [32, 33]) both read to the end of the frames and share the last piece, which comes in four head
    # ranges
    quarter = [(w.H * i // 4, w.H * (i + 1) // 4) for i in range(4)]
    assert info["n_groups"] == 34 and len(pieces) == 4 + 31 + 4
    assert all(p[2:] == (0, w.H) for p in pieces[4:-4])
    assert [p[2:] for p in pieces[-4:]] == quarter and len({p[:2] for p in pieces[-4:]}) == 1
    assert pieces[-1][1] == w.L - w.G
    assert all(abs((hi - lo) - KS) <= TILE for lo, hi, _, _ in pieces[4:-4])
    # the global rows of each quarter of the heads are merged and copied back right behind that quarter's launch
    merges = [o for o in sched["out"] if o[1:3] == (w.L - w.G, w.L)]
    assert [o[3:] for o in merges] == quarter and [o[0] for o in merges] == list(range(len(pieces) - 4, len(pieces)))
    launches = sched["item_launch"]
    assert max(launches) == len(pieces) - 1
    assert min(launches) == 1  # the first window group's first heads run after the second piece


def test_schedule_caps_the_piece_count():
    # 400 one-token chunks with r = 0: 400 window groups, merged into at most 64 pieces
    L, info, groups, sched = check_schedule(400, 1, 1, 0, 3, 1, 2, 64, 0)
    assert info["n_groups"] == 400
    assert len(sched["pieces"]) == 64


def test_host_list_keeps_short_global_splits():
    # the host-buffer forward's own work list: the plan's window items unchanged, the global leg in key splits half
    # as long when the global rows are plentiful (H3: 5 splits where the device plan has 3)
    w = configs.H3
    layout = wa.make_layout(w.B, w.L, w.H, w.D, w.global_pos)
    info, _, dev_items = wa.wa_geometry_describe(w.T, w.S, w.K, w.r, w.G, layout, with_items=True)
    host_items = wa.wa_host_schedule_describe(w.T, w.S, w.K, w.r, w.G, layout)["items"]
    assert info["n_splits"] == 3
    assert sorted(i for i in host_items if i[1] == 0) == sorted(i for i in dev_items if i[1] == 0)
    per_tile = {}
    for it in host_items:
        if it[1] == 1:
            per_tile.setdefault((it[0], it[2]), []).append((it[4], it[5]))
    assert len(per_tile) == w.H * w.G // 256
    for segs in per_tile.values():
        segs.sort()
        assert len(segs) == 5 and segs[0][0] == 0 and segs[-1][1] == w.L
        assert all(a[1] == b[0] for a, b in zip(segs, segs[1:]))
    # with few global rows the two lists are the same
    m = configs.MEDIUM
    lay = wa.make_layout(m.B, m.L, m.H, m.D, m.global_pos)
    _, _, dev_m = wa.wa_geometry_describe(m.T, m.S, m.K, m.r, m.G, lay, with_items=True)
    assert wa.wa_host_schedule_describe(m.T, m.S, m.K, m.r, m.G, lay)["items"] == dev_m
