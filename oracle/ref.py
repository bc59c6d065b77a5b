"""CPU oracle for chunk-aligned window softmax attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline / reference arm may import this
module. The CUDA library never does, and this module imports nothing from it: the two share no code. It is
plain, slow and written to be checked by eye, in float64.

What is computed (the VDN-Minimax-H3 window-attention article, lqnn.cn):
  * section 一 (why window attention): the packed sequence holds T latent frames of S spatial tokens each plus G
    global text/audio tokens. Frames are grouped into chunks of K latent frames; a query of frame t, in chunk
    c = floor(t / K), may see only the whole chunks in [c - radius, c + radius]; the global tokens stay fully
    connected (every query sees them, and a global query sees every token).
  * section 三 (the decomposed idea): the result is mathematically identical to the masked kernel: each query's
    softmax is normalised over exactly its kept set; the article keeps an eager per-frame loop as the
    correctness baseline, which is the shape of ``window_attention`` below.
Readings where the article is silent, each the plainest one the rest of the article supports:
  * chunks past either end of the sequence do not exist: the window is clamped, not shifted (section 一 speaks of
    the whole chunks in the range, i.e. the ones that exist);
  * T need not be a multiple of K: the last chunk is partial and otherwise ordinary (every K frames form a chunk);
  * globals sit after the frame tokens (global_pos = 0) or before them (global_pos = 1); either placement gives the
    same result up to that permutation of the rows;
  * scores are scaled by 1/sqrt(D); non-causal; no bias, softcap or dropout (the article mentions none).

The backward (window_attention_backward, row_logsumexp) follows the same loop and is pinned by
tests/test_oracle_backward.py: central finite differences of the forward above, and torch autograd through a
float64 dense attention in the cases that reduce to one.

Every function here is pinned by tests/test_oracle.py against facts that do not come from this file
(brute force over an explicit mask, a library dense-attention routine in the special cases that reduce to it,
closed forms and invariants), so no function is "parity unpinned".
"""
import math

import numpy as np


# ----------------------------------------------------------------------------------------------- geometry
def num_chunks(T, K):
    """Number of chunks: ceil(T / K) (the last chunk may hold fewer than K frames)."""
    return (T + K - 1) // K


def frame_offset(G, global_pos):
    """Index of the first frame token: 0 when the globals come after the frames, G when they come first."""
    return G if global_pos else 0


def global_offset(T, S, global_pos):
    """Index of the first global token: T*S when the globals come after the frames, 0 when they come first."""
    return 0 if global_pos else T * S


def frame_rows(t, S, f0):
    """Sequence indices of the S tokens of latent frame t (frame-major packing, section 一)."""
    return np.arange(f0 + t * S, f0 + (t + 1) * S, dtype=np.int64)


def window_chunks(c, r, nc):
    """Chunks visible from chunk c: the chunks of [c - r, c + r] that exist (section 一, window_bounds)."""
    return list(range(max(0, c - r), min(nc - 1, c + r) + 1))


def kept_set_of_frame(t, T, S, K, r, G, global_pos):
    """Sorted sequence indices a query token of frame t attends to: its window's frames plus all globals."""
    nc = num_chunks(T, K)
    f0 = frame_offset(G, global_pos)
    g0 = global_offset(T, S, global_pos)
    c = t // K
    idx = []
    for cc in window_chunks(c, r, nc):
        for tt in range(cc * K, min(T, (cc + 1) * K)):
            idx.append(frame_rows(tt, S, f0))
    idx.append(np.arange(g0, g0 + G, dtype=np.int64))
    return np.sort(np.concatenate(idx))


def kept_set_of_global(T, S, G):
    """A global query attends to the whole packed sequence (section 一: globals stay fully connected)."""
    return np.arange(T * S + G, dtype=np.int64)


# ------------------------------------------------------------------------------------------------ softmax
def attend(q_rows, k_kept, v_kept, scale):
    """Plain attention of some query rows over one kept set, float64.

    q_rows [n, D], k_kept / v_kept [m, D]. Scores s = q.k * scale; p = exp(s - max s) / sum exp(.) over the kept
    set only; out = p @ v. Returns (out [n, D], p [n, m]).
    """
    s = (q_rows @ k_kept.T) * scale
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    p = e / e.sum(axis=1, keepdims=True)
    return p @ v_kept, p


def _as64(x):
    if hasattr(x, "detach"):  # a torch tensor: upcast through float32 (exact for bf16)
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def window_attention(q, k, v, T, S, K, r, G, global_pos, return_probs=False):
    """Chunk-aligned window softmax attention over a packed sequence, by an eager per-frame loop.

    q, k, v: [B, L, H, D] with L = T*S + G (numpy or torch; upcast to float64 from the same values the GPU sees).
    Returns out [B, L, H, D] float64. With ``return_probs`` it also returns a dict mapping (b, h, row) to
    (kept indices, probabilities) for every row (debug mode; tiny inputs only).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, L, H, D = q.shape
    assert L == T * S + G, "sequence length must be T*S + G"
    scale = 1.0 / math.sqrt(D)
    out = np.zeros_like(q)
    probs = {} if return_probs else None
    f0 = frame_offset(G, global_pos)
    g0 = global_offset(T, S, global_pos)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                kept = kept_set_of_frame(t, T, S, K, r, G, global_pos)
                rows = frame_rows(t, S, f0)
                o, p = attend(q[b, rows, h], k[b, kept, h], v[b, kept, h], scale)
                out[b, rows, h] = o
                if return_probs:
                    for i, row in enumerate(rows):
                        probs[(b, h, int(row))] = (kept, p[i])
            if G:
                kept = kept_set_of_global(T, S, G)
                rows = np.arange(g0, g0 + G, dtype=np.int64)
                o, p = attend(q[b, rows, h], k[b, kept, h], v[b, kept, h], scale)
                out[b, rows, h] = o
                if return_probs:
                    for i, row in enumerate(rows):
                        probs[(b, h, int(row))] = (kept, p[i])
    return (out, probs) if return_probs else out


def window_attention_rows(q, k, v, T, S, K, r, G, global_pos, b, h, frames=(), global_rows=False):
    """The same computation restricted to one (b, h) slice and to the listed frames (and global rows).

    ``global_rows``: False (none), True (all G), or a sequence of global-token numbers g in [0, G) (row g0 + g).
    Rows are independent, so each returned row equals the matching row of ``window_attention``. Returns a dict
    {row index: output row (float64 [D])}. Used to check large workloads on a sample of rows.
    """
    D = q.shape[-1]
    scale = 1.0 / math.sqrt(D)
    f0 = frame_offset(G, global_pos)
    g0 = global_offset(T, S, global_pos)
    res = {}
    for t in frames:
        kept = kept_set_of_frame(t, T, S, K, r, G, global_pos)
        rows = frame_rows(t, S, f0)
        o, _ = attend(_as64(q[b, rows, h]), _as64(k[b, kept, h]), _as64(v[b, kept, h]), scale)
        for i, row in enumerate(rows):
            res[int(row)] = o[i]
    if global_rows is not False and G:
        kept = kept_set_of_global(T, S, G)
        if global_rows is True:
            rows = np.arange(g0, g0 + G, dtype=np.int64)
        else:
            rows = g0 + np.asarray(sorted(set(int(g) for g in global_rows)), dtype=np.int64)
            assert rows.size == 0 or (rows.min() >= g0 and rows.max() < g0 + G), "global rows lie in [0, G)"
        kk, vv = _as64(k[b, kept, h]), _as64(v[b, kept, h])
        for lo in range(0, G, 256):  # bounded score blocks: G x L may not fit in memory at once
            sel = rows[lo:lo + 256]
            o, _ = attend(_as64(q[b, sel, h]), kk, vv, scale)
            for i, row in enumerate(sel):
                res[int(row)] = o[i]
    return res


def chunk_frames(c, T, K):
    """Latent frames of chunk c."""
    return list(range(c * K, min(T, (c + 1) * K)))


def kept_pairs(T, S, K, r, G, global_pos=0):
    """Number of kept (query, key) pairs of one (b, h) slice, counted from the kept sets themselves."""
    n = 0
    for t in range(T):
        n += S * len(kept_set_of_frame(t, T, S, K, r, G, global_pos))
    return n + G * (T * S + G)


# ------------------------------------------------------------------------------------------------ backward
def row_logsumexp(q, k, T, S, K, r, G, global_pos):
    """LSE_i = ln sum_{j in kept(i)} exp(q_i.k_j / sqrt(D)) for every row, float64 [B, H, L]."""
    q, k = _as64(q), _as64(k)
    B, L, H, D = q.shape
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, H, L))
    f0, g0 = frame_offset(G, global_pos), global_offset(T, S, global_pos)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                kept = kept_set_of_frame(t, T, S, K, r, G, global_pos)
                rows = frame_rows(t, S, f0)
                s = (q[b, rows, h] @ k[b, kept, h].T) * scale
                mx = s.max(axis=1, keepdims=True)
                out[b, h, rows] = (mx + np.log(np.exp(s - mx).sum(axis=1, keepdims=True)))[:, 0]
            if G:
                rows = np.arange(g0, g0 + G)
                s = (q[b, rows, h] @ k[b, :, h].T) * scale
                mx = s.max(axis=1, keepdims=True)
                out[b, h, rows] = (mx + np.log(np.exp(s - mx).sum(axis=1, keepdims=True)))[:, 0]
    return out


def window_attention_backward(q, k, v, dout, T, S, K, r, G, global_pos):
    """Gradients (dq, dk, dv) of sum(out * dout) for the chunk-window attention, float64, by the same per-frame loop.

    For a row i with kept set J (scale c = 1/sqrt(D)): p = softmax_J(c q_i.k_j); o_i = sum p_j v_j. Then
    dv_j += p_j dout_i; dp_j = dout_i.v_j; ds_j = p_j (dp_j - sum_j' p_j' dp_j'); dq_i = c sum_j ds_j k_j;
    dk_j += c ds_j q_i (the chain rule through the softmax restricted to J).
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    B, L, H, D = q.shape
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    f0, g0 = frame_offset(G, global_pos), global_offset(T, S, global_pos)

    def rows_backward(b, h, rows, kept):
        _, p = attend(q[b, rows, h], k[b, kept, h], v[b, kept, h], scale)
        do = dout[b, rows, h]
        dv[b, kept, h] += p.T @ do
        dp = do @ v[b, kept, h].T
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dq[b, rows, h] += scale * (ds @ k[b, kept, h])
        dk[b, kept, h] += scale * (ds.T @ q[b, rows, h])

    for b in range(B):
        for h in range(H):
            for t in range(T):
                rows_backward(b, h, frame_rows(t, S, f0), kept_set_of_frame(t, T, S, K, r, G, global_pos))
            if G:
                rows_backward(b, h, np.arange(g0, g0 + G), kept_set_of_global(T, S, G))
    return dq, dk, dv


def window_attention_backward_rows(q, k, v, dout, T, S, K, r, G, global_pos, b, h, q_frames=(), global_q=False,
                                   k_frames=()):
    """The backward of one (b, h) slice restricted to some rows, for checking large workloads on a sample.

    Returns (dq, dk, dv), three dicts {row index: float64 [D]}: dq for the rows of ``q_frames`` (and for the global
    rows when ``global_q``), dk and dv for the rows of ``k_frames``. A query row's dq needs only its own kept set;
    a key row's dk and dv need every query that keeps it. Those queries are found by testing each frame's kept set
    (and every global query keeps every key), and each is handled as in ``window_attention_backward``; so every
    returned row equals the matching row of that function.
    """
    D = q.shape[-1]
    scale = 1.0 / math.sqrt(D)
    f0, g0 = frame_offset(G, global_pos), global_offset(T, S, global_pos)
    qs, ks, vs, ds = (_as64(x[b, :, h]) for x in (q, k, v, dout))
    key_rows = np.concatenate([frame_rows(t, S, f0) for t in k_frames]) if k_frames else np.zeros(0, np.int64)
    dq, dk, dv = {}, {}, {}
    dk_acc = np.zeros((len(key_rows), D))
    dv_acc = np.zeros((len(key_rows), D))

    def block(rows, kept, want_dq):
        _, p = attend(qs[rows], ks[kept], vs[kept], scale)
        dp = ds[rows] @ vs[kept].T
        dsc = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        if want_dq:
            g = scale * (dsc @ ks[kept])
            for i, row in enumerate(rows):
                dq[int(row)] = g[i]
        if len(key_rows):
            pos = {int(x): i for i, x in enumerate(kept)}
            cols = [pos.get(int(x), -1) for x in key_rows]
            sel = np.array([c >= 0 for c in cols])
            if sel.any():
                c = np.array([x for x in cols if x >= 0])
                dv_acc[sel] += p[:, c].T @ ds[rows]
                dk_acc[sel] += scale * (dsc[:, c].T @ qs[rows])

    for t in range(T):
        kept = kept_set_of_frame(t, T, S, K, r, G, global_pos)
        needed_for_keys = len(key_rows) > 0 and np.isin(key_rows, kept).any()
        if t in q_frames or needed_for_keys:
            block(frame_rows(t, S, f0), kept, t in q_frames)
    if G and (global_q or len(key_rows)):
        kept = kept_set_of_global(T, S, G)
        rows = np.arange(g0, g0 + G, dtype=np.int64)
        for lo in range(0, G, 256):  # bounded score blocks: G x L may not fit in memory at once
            block(rows[lo:lo + 256], kept, global_q)
    for i, row in enumerate(key_rows):
        dk[int(row)] = dk_acc[i]
        dv[int(row)] = dv_acc[i]
    return dq, dk, dv
