"""Pins for the CPU oracle (CPU only).

The oracle is checked against facts that do not come from its own code:
  * brute force: an explicit L x L mask built by a separate pairwise rule, then a masked dense softmax in pure
    Python loops (no numpy matmul), on tiny random geometries with both global placements;
  * hand-drawn masks from the article's window rule (tests/golden/);
  * special cases that reduce to a library routine (torch scaled_dot_product_attention in float64): a radius
    covering every chunk gives full dense attention; radius 0 without globals gives block-diagonal attention;
  * closed forms (k = 0 gives the mean of v over the kept set; constant v; one-hot v gives zero outside the
    window) and invariants (global rows ignore K and r; front/back placement is a permutation; permuting tokens
    inside a chunk permutes only that chunk's rows; row sums are 1 over exactly the kept set);
  * planted mistakes: plausible bugs put into a copy of the oracle must fail the brute-force pin.
"""
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle.ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------- brute force
def is_global(x, T, S, G, global_pos):
    return x < G if global_pos else x >= T * S


def frame_of(x, S, G, global_pos):
    return (x - G) // S if global_pos else x // S


def brute_mask(T, S, K, r, G, global_pos):
    """Pairwise rule, written independently of the oracle: kept iff either token is global, or the two frames'
    chunks are at most r apart (VDN-Minimax-H3 article, section 一)."""
    L = T * S + G
    m = np.zeros((L, L), dtype=bool)
    for i in range(L):
        for j in range(L):
            if is_global(i, T, S, G, global_pos) or is_global(j, T, S, G, global_pos):
                m[i, j] = True
            else:
                ci = frame_of(i, S, G, global_pos) // K
                cj = frame_of(j, S, G, global_pos) // K
                m[i, j] = abs(ci - cj) <= r
    return m


def brute_attention(q, k, v, mask):
    """Masked dense softmax attention in pure Python loops. q, k, v: float64 [B, L, H, D]."""
    B, L, H, D = q.shape
    scale = 1.0 / math.sqrt(D)
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            for i in range(L):
                s = {}
                for j in range(L):
                    if mask[i, j]:
                        acc = 0.0
                        for d in range(D):
                            acc += q[b, i, h, d] * k[b, j, h, d]
                        s[j] = acc * scale
                mx = max(s.values())
                e = {j: math.exp(x - mx) for j, x in s.items()}
                z = sum(e.values())
                for d in range(D):
                    out[b, i, h, d] = sum(e[j] * v[b, j, h, d] for j in e) / z
    return out


def rand_qkv(rng, B, L, H, D):
    return [rng.standard_normal((B, L, H, D)) for _ in range(3)]


def tiny_geometries(n, seed):
    rnd = random.Random(seed)
    geos = []
    for _ in range(n):
        T = rnd.randint(1, 7)
        S = rnd.randint(1, 5)
        K = rnd.randint(1, 3)
        r = rnd.randint(0, 2)
        G = rnd.randint(0, 4)
        gp = rnd.randint(0, 1)
        geos.append((T, S, K, r, G, gp))
    # corners: a single chunk, K > T, radius beyond the chunk count, no globals
    geos += [(1, 3, 1, 0, 2, 0), (3, 2, 5, 0, 1, 1), (7, 1, 2, 4, 0, 0), (5, 2, 2, 1, 0, 1)]
    return geos


@pytest.mark.parametrize("geo", tiny_geometries(24, seed=7))
def test_brute_force(geo):
    T, S, K, r, G, gp = geo
    rng = np.random.default_rng(hash(geo) % (2 ** 32))
    q, k, v = rand_qkv(rng, 1, T * S + G, 2, 4)
    want = brute_attention(q, k, v, brute_mask(T, S, K, r, G, gp))
    got = ref.window_attention(q, k, v, T, S, K, r, G, gp)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def load_mask(name):
    rows = [ln.strip() for ln in open(os.path.join(GOLDEN, name)) if ln.strip() and not ln.startswith("#")]
    return np.array([[c == "1" for c in ln] for ln in rows])


@pytest.mark.parametrize("name,geo", [
    ("mask_T6_S1_K2_r1_G1_back.txt", (6, 1, 2, 1, 1, 0)),
    ("mask_T5_S1_K2_r1_G2_front.txt", (5, 1, 2, 1, 2, 1)),
    ("mask_T3_S2_K1_r0_G0.txt", (3, 2, 1, 0, 0, 0)),
])
def test_hand_drawn_masks(name, geo):
    T, S, K, r, G, gp = geo
    want = load_mask(name)
    L = T * S + G
    # the oracle's kept sets, laid out as a mask
    got = np.zeros((L, L), dtype=bool)
    f0 = G if gp else 0
    g0 = 0 if gp else T * S
    for t in range(T):
        for i in range(f0 + t * S, f0 + (t + 1) * S):
            got[i, ref.kept_set_of_frame(t, T, S, K, r, G, gp)] = True
    for i in range(g0, g0 + G):
        got[i, ref.kept_set_of_global(T, S, G)] = True
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(brute_mask(*geo), want)
    # and the probabilities' support in debug mode is exactly the drawn mask
    rng = np.random.default_rng(3)
    q, k, v = rand_qkv(rng, 1, L, 1, 4)
    _, probs = ref.window_attention(q, k, v, *geo, return_probs=True)
    for i in range(L):
        kept, p = probs[(0, 0, i)]
        supp = np.zeros(L, dtype=bool)
        supp[kept[p > 0]] = True
        np.testing.assert_array_equal(supp, want[i])


# --------------------------------------------------------------------------- library special cases
def sdpa64(q, k, v):
    """torch's dense scaled-dot-product attention in float64; inputs [L, D] (one slice)."""
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[0, 0].numpy()


@pytest.mark.parametrize("geo", [(6, 3, 2, 2, 3, 0), (7, 2, 3, 5, 4, 1), (4, 4, 1, 3, 0, 0), (9, 2, 4, 2, 1, 1)])
def test_radius_covering_all_chunks_is_dense(geo):
    T, S, K, r, G, gp = geo
    assert r >= ref.num_chunks(T, K) - 1
    rng = np.random.default_rng(11)
    q, k, v = rand_qkv(rng, 2, T * S + G, 3, 8)
    got = ref.window_attention(q, k, v, *geo)
    for b in range(2):
        for h in range(3):
            np.testing.assert_allclose(got[b, :, h], sdpa64(q[b, :, h], k[b, :, h], v[b, :, h]), atol=1e-12)


@pytest.mark.parametrize("geo", [(6, 3, 2, 0, 0, 0), (7, 2, 3, 0, 0, 1), (5, 4, 1, 0, 0, 0)])
def test_radius0_no_globals_is_block_diagonal(geo):
    T, S, K, r, G, gp = geo
    rng = np.random.default_rng(12)
    q, k, v = rand_qkv(rng, 1, T * S, 2, 8)
    got = ref.window_attention(q, k, v, *geo)
    for c in range(ref.num_chunks(T, K)):
        lo, hi = c * K * S, min(T, (c + 1) * K) * S
        for h in range(2):
            want = sdpa64(q[0, lo:hi, h], k[0, lo:hi, h], v[0, lo:hi, h])
            np.testing.assert_allclose(got[0, lo:hi, h], want, atol=1e-12)


# ------------------------------------------------------------------------- closed forms, invariants
GEOS = [(6, 3, 2, 1, 3, 0), (7, 2, 3, 1, 4, 1), (5, 2, 2, 0, 2, 0), (8, 1, 3, 2, 1, 1)]


@pytest.mark.parametrize("geo", GEOS)
def test_zero_keys_give_mean_of_kept_values(geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    rng = np.random.default_rng(13)
    q, _, v = rand_qkv(rng, 1, L, 2, 5)
    k = np.zeros_like(q)
    got = ref.window_attention(q, k, v, *geo)
    mask = brute_mask(*geo)
    for i in range(L):
        np.testing.assert_allclose(got[0, i], v[0, mask[i]].mean(axis=0), atol=1e-12)


@pytest.mark.parametrize("geo", GEOS)
def test_constant_values_pass_through(geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    rng = np.random.default_rng(14)
    q, k, _ = rand_qkv(rng, 1, L, 2, 5)
    c = rng.standard_normal(5)
    v = np.broadcast_to(c, (1, L, 2, 5)).copy()
    got = ref.window_attention(q, k, v, *geo)
    np.testing.assert_allclose(got, v, atol=1e-12)


@pytest.mark.parametrize("geo", GEOS)
def test_one_hot_value_is_attention_mass(geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    rng = np.random.default_rng(15)
    q, k, _ = rand_qkv(rng, 1, L, 1, 4)
    mask = brute_mask(*geo)
    for j in range(L):
        v = np.zeros((1, L, 1, 4))
        v[0, j, 0, 0] = 1.0
        got = ref.window_attention(q, k, v, *geo)[0, :, 0, 0]
        assert np.all(got[~mask[:, j]] == 0.0)  # no mass on token j from queries that do not keep it
        assert np.all(got[mask[:, j]] > 0.0)
        assert np.all(got <= 1.0)


@pytest.mark.parametrize("geo", GEOS)
def test_row_sums_are_one_over_exactly_the_kept_set(geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    rng = np.random.default_rng(16)
    q, k, v = rand_qkv(rng, 1, L, 2, 4)
    _, probs = ref.window_attention(q, k, v, *geo, return_probs=True)
    mask = brute_mask(*geo)
    for (b, h, i), (kept, p) in probs.items():
        assert abs(p.sum() - 1.0) < 1e-12
        np.testing.assert_array_equal(np.sort(kept), np.flatnonzero(mask[i]))
    assert len(probs) == 2 * L


def test_global_rows_ignore_chunking():
    T, S, G = 6, 3, 3
    rng = np.random.default_rng(17)
    q, k, v = rand_qkv(rng, 1, T * S + G, 2, 4)
    outs = [ref.window_attention(q, k, v, T, S, K, r, G, 0)[:, T * S:] for K in (1, 2, 4) for r in (0, 1, 3)]
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], atol=1e-13)


@pytest.mark.parametrize("geo", [(6, 3, 2, 1, 3), (7, 2, 3, 0, 4), (5, 1, 2, 2, 1)])
def test_front_back_placement_is_a_permutation(geo):
    T, S, K, r, G = geo
    F = T * S
    rng = np.random.default_rng(18)
    q, k, v = rand_qkv(rng, 1, F + G, 2, 4)
    back = ref.window_attention(q, k, v, T, S, K, r, G, 0)
    perm = np.concatenate([np.arange(F, F + G), np.arange(F)])  # front index -> back index
    front = ref.window_attention(q[:, perm], k[:, perm], v[:, perm], T, S, K, r, G, 1)
    np.testing.assert_allclose(front, back[:, perm], atol=1e-12)


@pytest.mark.parametrize("geo", [(6, 3, 2, 1, 3, 0), (7, 2, 3, 1, 2, 1)])
def test_permuting_inside_a_chunk_permutes_only_its_rows(geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    f0 = G if gp else 0
    rng = np.random.default_rng(19)
    q, k, v = rand_qkv(rng, 1, L, 2, 4)
    base = ref.window_attention(q, k, v, *geo)
    lo, hi = f0 + K * S, f0 + min(T, 2 * K) * S  # chunk 1
    perm = np.arange(L)
    perm[lo:hi] = lo + rng.permutation(hi - lo)
    out = ref.window_attention(q[:, perm], k[:, perm], v[:, perm], *geo)
    np.testing.assert_allclose(out, base[:, perm], atol=1e-12)


def closed_form_kept_pairs(T, S, K, r, G):
    """Sum over chunks of rows_c * (window tokens_c + G), plus G * L for the global rows."""
    nc = -(-T // K)
    tot = 0
    for c in range(nc):
        rows = (min(T, (c + 1) * K) - c * K) * S
        w = (min(T, (min(nc - 1, c + r) + 1) * K) - max(0, c - r) * K) * S
        tot += rows * (w + G)
    return tot + G * (T * S + G)


@pytest.mark.parametrize("geo", [(6, 16, 2, 1, 8), (24, 256, 4, 1, 256), (50, 300, 4, 2, 77), (102, 960, 3, 1, 2048),
                                 (34, 960, 1, 0, 2048), (7, 5, 3, 2, 4)])
def test_kept_pair_count(geo):
    T, S, K, r, G = geo
    n = ref.kept_pairs(T, S, K, r, G)
    assert n == closed_form_kept_pairs(T, S, K, r, G)
    if geo[:5] == (6, 16, 2, 1, 8):  # the tiny workload, counted by hand: 32*(72+104+72) + 8*104 per head
        assert n == 8768
    if T * S + G < 40:
        assert n == brute_mask(T, S, K, r, G, 0).sum() == brute_mask(T, S, K, r, G, 1).sum()


def test_row_sample_matches_full():
    T, S, K, r, G, gp = 9, 4, 2, 1, 5, 1
    rng = np.random.default_rng(20)
    q, k, v = rand_qkv(rng, 2, T * S + G, 3, 8)
    full = ref.window_attention(q, k, v, T, S, K, r, G, gp)
    got = ref.window_attention_rows(q, k, v, T, S, K, r, G, gp, b=1, h=2, frames=[0, 4, 8], global_rows=True)
    assert len(got) == 3 * S + G
    for row, o in got.items():
        np.testing.assert_allclose(o, full[1, row, 2], atol=1e-13)


def test_bf16_torch_inputs_are_upcast_exactly():
    g = torch.Generator().manual_seed(0)
    q, k, v = (torch.randn(1, 14, 2, 8, generator=g).bfloat16() for _ in range(3))
    a = ref.window_attention(q, k, v, 3, 4, 2, 0, 2, 0)
    b = ref.window_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), 3, 4, 2, 0, 2, 0)
    np.testing.assert_array_equal(a, b)


# -------------------------------------------------------------------------------- planted mistakes
def _mutant_window_chunks_off_by_one(c, r, nc):
    return list(range(max(0, c - r), min(nc - 1, c + r + 1) + 1))


def _mutant_window_chunks_shifted(c, r, nc):  # a fixed-width window shifted at the edges instead of clamped
    lo = min(max(0, c - r), max(0, nc - 1 - 2 * r))
    return list(range(lo, min(nc, lo + 2 * r + 1)))


def _mutant_attend_no_scale(q_rows, k_kept, v_kept, scale):
    s = q_rows @ k_kept.T
    e = np.exp(s - s.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    return p @ v_kept, p


def _mutant_attend_transposed_v(q_rows, k_kept, v_kept, scale):
    s = (q_rows @ k_kept.T) * scale
    e = np.exp(s - s.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    return (p @ v_kept[::-1]), p


def _mutant_global_offset(T, S, global_pos):
    return 0 if not global_pos else T * S


@pytest.mark.parametrize("attr,mutant", [
    ("window_chunks", _mutant_window_chunks_off_by_one),
    ("window_chunks", _mutant_window_chunks_shifted),
    ("attend", _mutant_attend_no_scale),
    ("attend", _mutant_attend_transposed_v),
    ("global_offset", _mutant_global_offset),
])
def test_planted_mistakes_are_caught(monkeypatch, attr, mutant):
    monkeypatch.setattr(ref, attr, mutant)
    caught = False
    for geo in tiny_geometries(10, seed=99):
        T, S, K, r, G, gp = geo
        rng = np.random.default_rng(5)
        q, k, v = rand_qkv(rng, 1, T * S + G, 1, 4)
        try:
            got = ref.window_attention(q, k, v, *geo)
        except (ValueError, IndexError, AssertionError):
            caught = True
            break
        want = brute_attention(q, k, v, brute_mask(*geo))
        if not np.allclose(got, want, atol=1e-12):
            caught = True
            break
    assert caught, f"planted mistake in {attr} went unnoticed"


@pytest.mark.parametrize("gp", [0, 1])
def test_row_sample_global_subset_matches_full(gp):
    """A subset of the global rows (numbered 0..G-1 from the first global token) gives exactly those rows, each equal
    to the full oracle's row; the whole list gives the same rows as global_rows=True."""
    T, S, K, r, G = 7, 3, 2, 1, 9
    rng = np.random.default_rng(21 + gp)
    q, k, v = rand_qkv(rng, 1, T * S + G, 2, 8)
    full = ref.window_attention(q, k, v, T, S, K, r, G, gp)
    g0 = ref.global_offset(T, S, gp)
    sub = [G - 1, 0, 4]
    got = ref.window_attention_rows(q, k, v, T, S, K, r, G, gp, b=0, h=1, frames=[3], global_rows=sub)
    assert sorted(got) == sorted(ref.frame_rows(3, S, ref.frame_offset(G, gp)).tolist() + [g0 + g for g in sub])
    for row, o in got.items():
        np.testing.assert_allclose(o, full[0, row, 1], atol=1e-13)
    every = ref.window_attention_rows(q, k, v, T, S, K, r, G, gp, b=0, h=1, global_rows=list(range(G)))
    alln = ref.window_attention_rows(q, k, v, T, S, K, r, G, gp, b=0, h=1, global_rows=True)
    assert sorted(every) == sorted(alln) == list(range(g0, g0 + G))
    for row in every:
        np.testing.assert_array_equal(every[row], alln[row])
