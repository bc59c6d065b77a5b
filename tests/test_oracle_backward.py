"""Pins for the oracle's backward and row log-sum-exp (CPU only).

- Central finite differences of the forward oracle: d/dx sum(out * dout) for every input element, on tiny random
  geometries with both global placements (independent of the gradient formula).
- Library special case: with a radius covering every chunk the layer is dense attention, so torch autograd
  through float64 scaled_dot_product_attention gives the gradients; with r = 0 and no globals it is per-chunk.
- The row log-sum-exp against scipy's logsumexp over the brute-force kept mask.
- Planted mistakes in the backward must fail the finite-difference pin.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle.ref as ref
from test_oracle import brute_mask, rand_qkv, tiny_geometries


def finite_difference(q, k, v, dout, geo, eps=1e-6):
    grads = []
    for which in range(3):
        x = [q, k, v][which]
        g = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            fp = (ref.window_attention(q, k, v, *geo) * dout).sum()
            x[idx] = old - eps
            fm = (ref.window_attention(q, k, v, *geo) * dout).sum()
            x[idx] = old
            g[idx] = (fp - fm) / (2 * eps)
        grads.append(g)
    return grads


@pytest.mark.parametrize("geo", tiny_geometries(6, seed=41) + [(5, 2, 2, 1, 2, 1), (4, 3, 1, 0, 0, 0)])
def test_backward_matches_finite_differences(geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    rng = np.random.default_rng(abs(hash(geo)) % 2 ** 32)
    q, k, v = rand_qkv(rng, 1, L, 1, 3)
    dout = rng.standard_normal(q.shape)
    got = ref.window_attention_backward(q, k, v, dout, *geo)
    want = finite_difference(q, k, v, dout, geo)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, atol=1e-6, rtol=1e-6)


def sdpa_grads(q, k, v, dout):
    """Gradients of dense float64 attention by torch autograd; inputs [L, D] (one slice)."""
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None])[0, 0]
    (o * torch.tensor(dout)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("geo", [(6, 3, 2, 2, 3, 0), (7, 2, 3, 5, 4, 1)])
def test_backward_dense_special_case(geo):
    T, S, K, r, G, gp = geo
    rng = np.random.default_rng(51)
    q, k, v = rand_qkv(rng, 1, T * S + G, 2, 8)
    dout = rng.standard_normal(q.shape)
    dq, dk, dv = ref.window_attention_backward(q, k, v, dout, *geo)
    for h in range(2):
        wq, wk, wv = sdpa_grads(q[0, :, h], k[0, :, h], v[0, :, h], dout[0, :, h])
        np.testing.assert_allclose(dq[0, :, h], wq, atol=1e-12)
        np.testing.assert_allclose(dk[0, :, h], wk, atol=1e-12)
        np.testing.assert_allclose(dv[0, :, h], wv, atol=1e-12)


def test_backward_block_diagonal_special_case():
    T, S, K = 6, 3, 2
    rng = np.random.default_rng(52)
    q, k, v = rand_qkv(rng, 1, T * S, 1, 8)
    dout = rng.standard_normal(q.shape)
    dq, dk, dv = ref.window_attention_backward(q, k, v, dout, T, S, K, 0, 0, 0)
    for c in range(3):
        sl = slice(c * K * S, (c + 1) * K * S)
        wq, wk, wv = sdpa_grads(q[0, sl, 0], k[0, sl, 0], v[0, sl, 0], dout[0, sl, 0])
        np.testing.assert_allclose(dq[0, sl, 0], wq, atol=1e-12)
        np.testing.assert_allclose(dk[0, sl, 0], wk, atol=1e-12)
        np.testing.assert_allclose(dv[0, sl, 0], wv, atol=1e-12)


@pytest.mark.parametrize("geo", tiny_geometries(8, seed=43))
def test_row_logsumexp_against_scipy(geo):
    T, S, K, r, G, gp = geo
    L = T * S + G
    rng = np.random.default_rng(53)
    q, k, _ = rand_qkv(rng, 2, L, 2, 4)
    got = ref.row_logsumexp(q, k, *geo)
    mask = brute_mask(*geo)
    for b in range(2):
        for h in range(2):
            s = q[b, :, h] @ k[b, :, h].T / 2.0  # 1/sqrt(4)
            want = np.array([logsumexp(s[i, mask[i]]) for i in range(L)])
            np.testing.assert_allclose(got[b, h], want, atol=1e-12)


def _backward_with_mistake(q, k, v, dout, T, S, K, r, G, gp, mistake):
    """A copy of the per-row gradient with one plausible mistake planted (used only to show the pin catches it)."""
    q, k, v, dout = (np.asarray(x, np.float64) for x in (q, k, v, dout))
    B, L, H, D = q.shape
    c = 1.0 / np.sqrt(D)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    f0, g0 = (G, 0) if gp else (0, T * S)
    groups = [(ref.frame_rows(t, S, f0), ref.kept_set_of_frame(t, T, S, K, r, G, gp)) for t in range(T)]
    if G:
        groups.append((np.arange(g0, g0 + G), ref.kept_set_of_global(T, S, G)))
    for rows, kept in groups:
        _, p = ref.attend(q[0, rows, 0], k[0, kept, 0], v[0, kept, 0], c)
        do = dout[0, rows, 0]
        dv[0, kept, 0] += p.T @ do
        dp = do @ v[0, kept, 0].T
        ds = p * dp if mistake == "no_centring" else p * (dp - (p * dp).sum(axis=1, keepdims=True))
        sc = 1.0 if mistake == "no_scale" else c
        dq[0, rows, 0] += sc * (ds @ k[0, kept, 0])
        dk[0, kept, 0] += sc * (ds.T @ (do if mistake == "dk_from_dout" else q[0, rows, 0]))
    return dq, dk, dv


@pytest.mark.parametrize("mistake", ["no_centring", "no_scale", "dk_from_dout"])
def test_planted_backward_mistakes_are_caught(mistake):
    geo = (5, 2, 2, 1, 2, 0)
    rng = np.random.default_rng(54)
    q, k, v = rand_qkv(rng, 1, 12, 1, 3)
    dout = rng.standard_normal(q.shape)
    want = finite_difference(q, k, v, dout, geo)
    got = _backward_with_mistake(q, k, v, dout, *geo, mistake)
    assert not all(np.allclose(g, w, atol=1e-6) for g, w in zip(got, want))
    clean = _backward_with_mistake(q, k, v, dout, *geo, None)
    assert all(np.allclose(g, w, atol=1e-6) for g, w in zip(clean, want))


@pytest.mark.parametrize("geo", [(7, 3, 2, 1, 4, 0), (9, 2, 3, 1, 5, 1), (6, 4, 1, 0, 0, 0), (5, 3, 2, 3, 2, 1)])
def test_backward_rows_equal_full_backward(geo):
    """The row-restricted backward (used on samples of large workloads) returns exactly the rows of the full one."""
    T, S, K, r, G, gp = geo
    L = T * S + G
    rng = np.random.default_rng(sum(geo) + 7)
    q, k, v = rand_qkv(rng, 2, L, 2, 4)
    dout = rng.standard_normal(q.shape)
    full = ref.window_attention_backward(q, k, v, dout, *geo)
    f0 = G if gp else 0
    g0 = 0 if gp else T * S
    for b, h in ((0, 1), (1, 0)):
        q_frames, k_frames = (0, T // 2), (T - 1, T // 2)
        dq, dk, dv = ref.window_attention_backward_rows(q, k, v, dout, *geo, b, h, q_frames=q_frames,
                                                        global_q=G > 0, k_frames=k_frames)
        q_rows = [f0 + t * S + i for t in q_frames for i in range(S)] + list(range(g0, g0 + G))
        k_rows = [f0 + t * S + i for t in k_frames for i in range(S)]
        assert sorted(dq) == sorted(set(q_rows)) and sorted(dk) == sorted(set(k_rows)) == sorted(dv)
        for row in q_rows:
            np.testing.assert_allclose(dq[row], full[0][b, row, h], rtol=1e-12, atol=1e-12)
        for row in k_rows:
            np.testing.assert_allclose(dk[row], full[1][b, row, h], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(dv[row], full[2][b, row, h], rtol=1e-12, atol=1e-12)
