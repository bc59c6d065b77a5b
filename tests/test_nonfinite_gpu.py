"""A row's result depends only on the tokens of its kept set (VDN-Minimax-H3 window-attention article, section 一:
the kept set of a frame query is its chunk window plus the globals; section 三: each row's softmax is normalised
over exactly that set). Tokens outside it may hold anything, Inf and NaN included.

The kernels read whole 128-row tiles, so the last tile of a key segment also holds rows past the segment's end:
frames of the next chunk, or the first frames after globals placed at the front. These tests plant Inf and NaN
exactly there and check that every row whose kept set excludes the planted rows is bit-identical to a run on clean
inputs (and finite, and within the oracle's tolerance), for the bf16 forward, the e4m3 forward and the backward.
"""
import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu


def frames_clean_of(w, planted):
    """Frames whose kept set contains none of the planted sequence rows."""
    bad = set(int(x) for x in planted)
    return [t for t in range(w.T)
            if not bad.intersection(ref.kept_set_of_frame(t, w.T, w.S, w.K, w.r, w.G, w.global_pos).tolist())]


def frame_row_index(w, frames):
    return np.concatenate([ref.frame_rows(t, w.S, w.f0) for t in frames]) if frames else np.zeros(0, np.int64)


def plan_groups(wa, w):
    """The window groups of the library's own plan (host-only wa_geometry_describe)."""
    lay = wa.make_layout(w.B, w.L, w.H, w.D, w.global_pos)
    return wa.wa_geometry_describe(w.T, w.S, w.K, w.r, w.G, lay)[1]


def tail_rows(w, g):
    """Rows that the last 128-row tile of each key segment of window group g reads past the segment's end and that
    lie outside the group's kept set (sequence rows past L are zero-filled by the copy and not counted)."""
    t0 = (g["q_lo"] - w.f0) // w.S
    kept = set(ref.kept_set_of_frame(t0, w.T, w.S, w.K, w.r, w.G, w.global_pos).tolist())
    rows = set()
    for lo, hi in ((g["kv0_lo"], g["kv0_hi"]), (g["kv1_lo"], g["kv1_hi"])):
        if hi > lo:
            rows.update(range(hi, min(w.L, lo + -(-(hi - lo) // 128) * 128)))
    return np.array(sorted(rows - kept), dtype=np.int64)


def group_frames(w, g):
    return list(range((g["q_lo"] - w.f0) // w.S, (g["q_hi"] - w.f0) // w.S))


def targets(wa, w):
    """(group, planted rows) for every window group with a ragged tail outside its kept set."""
    out = []
    for g in plan_groups(wa, w):
        rows = tail_rows(w, g)
        if len(rows):
            out.append((g, rows))
    assert out, "the geometry must give some group a tile that reads past its segment"
    return out


def plant(t, rows, value):
    t = t.clone()
    t[:, rows] = value
    return t


FWD_CASES = [
    # globals before the frames: the global segment's last tile reads frames 0..; windows of 600 rows end mid-tile
    configs.Workload("nf_front", B=1, H=2, D=128, T=12, S=100, K=2, r=1, G=77, global_pos=1, seed=51),
    # globals after the frames, D = 64 (four value slots), windows of 3 x 70 rows
    configs.Workload("nf_back_d64", B=2, H=1, D=64, T=15, S=70, K=1, r=1, G=40, global_pos=0, seed=52),
]


@pytest.mark.parametrize("w", FWD_CASES, ids=lambda w: w.name)
def test_forward_rows_ignore_nonfinite_outside_kept_set(cuda, w):
    q, k, v = inputs.make_qkv(w, device="cuda")
    want = ref.window_attention(q.cpu(), k.cpu(), v.cpu(), w.T, w.S, w.K, w.r, w.G, w.global_pos)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        a = plan.forward(q, k, v)
        for g, rows in targets(cuda, w):
            clean = frames_clean_of(w, rows)
            assert set(group_frames(w, g)) <= set(clean)
            keep = torch.as_tensor(frame_row_index(w, clean), device="cuda")
            for kval, vval in ((float("inf"), float("nan")), (float("nan"), float("-inf"))):
                b = plan.forward(q, plant(k, rows, kval), plant(v, rows, vval))
                assert plan.check_error() == 0
                assert torch.equal(a[:, keep], b[:, keep]), f"group {g}: rows outside the planted rows' reach changed"
                assert torch.isfinite(b[:, keep].float()).all()
            # and those rows are the oracle's (which never looks outside a kept set)
            got, sel = b.float().cpu().numpy(), keep.cpu().numpy()
            for bi in range(w.B):
                for h in range(w.H):
                    x, y = got[bi, sel, h], want[bi, sel, h]
                    assert np.linalg.norm(x - y) / np.linalg.norm(y) <= 5e-3 and np.abs(x - y).max() <= 3e-2
    finally:
        plan.close()


def test_fp8_forward_rows_ignore_nonfinite_outside_kept_set(cuda):
    w = FWD_CASES[0]
    q, k, v = inputs.make_qkv(w, device="cuda")
    sq = float(q.float().abs().max()) / 448.0
    sk = float(k.float().abs().max()) / 448.0
    q8 = (q.float() / sq).to(torch.float8_e4m3fn)
    k8 = (k.float() / sk).to(torch.float8_e4m3fn)
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        a = plan.forward_fp8(q8, k8, v, sq, sk)
        for g, rows in targets(cuda, w):
            keep = torch.as_tensor(frame_row_index(w, frames_clean_of(w, rows)), device="cuda")
            k8_nan = k8.clone()
            k8_nan.view(torch.uint8)[:, rows] = 0x7F  # e4m3fn NaN (the format has no infinity)
            b = plan.forward_fp8(q8, k8_nan, plant(v, rows, float("inf")), sq, sk)
            assert plan.check_error() == 0
            assert torch.equal(a[:, keep], b[:, keep]), f"group {g}"
            assert torch.isfinite(b[:, keep].float()).all()
    finally:
        plan.close()


def test_backward_dq_ignores_nonfinite_keys_outside_kept_set(cuda):
    """Keys and values planted with Inf / NaN past a window's end: dq of every row that does not keep them is
    unchanged (the global rows keep everything, and through them so does every key's dk, dv)."""
    w = FWD_CASES[0]
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        dq, _, _ = plan.backward(q, k, v, out, dout, lse)
        for g, rows in targets(cuda, w):
            keep = torch.as_tensor(frame_row_index(w, frames_clean_of(w, rows)), device="cuda")
            k2, v2 = plant(k, rows, float("inf")), plant(v, rows, float("nan"))
            out2, lse2 = plan.forward_lse(q, k2, v2)
            dq2, _, _ = plan.backward(q, k2, v2, out2, dout, lse2)
            assert plan.check_error() == 0
            assert torch.equal(dq[:, keep], dq2[:, keep]), f"group {g}"
            assert torch.isfinite(dq2[:, keep].float()).all()
    finally:
        plan.close()


@pytest.mark.parametrize("D", [128, 64])
def test_backward_dkdv_ignore_nonfinite_queries_outside_kept_set(cuda, D):
    """No globals. Read key-major, a key group's query segment is its own window (the kept relation is symmetric),
    so the rows its last query tile reads past the window's end are queries that do not keep these keys. Those
    queries (q = Inf) and their upstream gradients (dout = NaN) are planted: dq of every other row and dk, dv of every
    key that no planted query keeps are unchanged."""
    w = configs.Workload(f"nf_bwd_d{D}", B=1, H=2, D=D, T=12, S=100, K=2, r=1, G=0, global_pos=0, seed=53)
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    try:
        out, lse = plan.forward_lse(q, k, v)
        g1 = plan.backward(q, k, v, out, dout, lse)
        for g, rows in targets(cuda, w):
            # a key is touched by a planted query exactly when that query keeps it: keys of frames whose kept set
            # (= the queries that keep them) holds no planted row are clean
            key_frames = frames_clean_of(w, rows)
            assert set(group_frames(w, g)) <= set(key_frames)
            keys = torch.as_tensor(frame_row_index(w, key_frames), device="cuda")
            others = torch.as_tensor(np.setdiff1d(np.arange(w.L), rows), device="cuda")
            q2, do2 = plant(q, rows, float("inf")), plant(dout, rows, float("nan"))
            out2, lse2 = plan.forward_lse(q2, k, v)
            g2 = plan.backward(q2, k, v, out2, do2, lse2)
            assert plan.check_error() == 0
            assert torch.equal(g1[0][:, others], g2[0][:, others]), f"group {g}: dq"
            for name, a, b in zip(("dk", "dv"), g1[1:], g2[1:]):
                assert torch.equal(a[:, keys], b[:, keys]), f"group {g}: {name}"
                assert torch.isfinite(b[:, keys].float()).all()
    finally:
        plan.close()
