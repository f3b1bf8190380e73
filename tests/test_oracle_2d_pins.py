"""Pins of the fp64 oracle's 2-D circulant attention (no GPU).

Page: "Vision Transformers are Circulant Attention Learners" — the attention
map is modelled as a BCCB matrix (block circulant with circulant blocks),
whose product with a vector is a 2-D circular convolution, O = σ(a) ⊛ V;
a comes from Q and K through FFTs and an element-wise product (a
correlation).  The page prints no formula for a, so the oracle takes the
reading a[k] = (1/dh) Σ_c Σ_i Q[i, c] K[i ⊖ k, c] (the sum along each
wrapped 2-D diagonal of Q·K^T, averaged over the head's channels); the pins
below fix everything else and tie a to that reading through an explicit
Q·K^T, never through its own formula:

* h = 1 (or w = 1) reduces to the separately pinned 1-D CAT oracle;
* the explicit BCCB matrix (numpy) against the convolution;
* a against the diagonal sums of an explicit Q·K^T (numpy matmul);
* separable generators (outer products) against two 1-D convolutions;
* one-hot generators against a 2-D roll, uniform ones against the mean;
* the O(N²) definitions against numpy's 2-D FFT evaluation.
"""
import numpy as np
import pytest

import oracle
import synth


def _qkv(B, h, w, D, H, seed=0):
    N = h * w
    X, _, V = synth.make_inputs(B, N, D, H, "f32", seed)
    K = synth.make_grad(B, N, D, "f32", seed)
    return X.double().numpy(), K.double().numpy(), V.double().numpy()


@pytest.mark.parametrize("h,w", [(1, 9), (9, 1), (1, 16)])
def test_one_row_grid_is_1d_cat(h, w):
    """A 1 x N (or N x 1) grid is the 1-D circulant product and correlation."""
    B, D, H = 2, 6, 3
    Q, K, V = _qkv(B, h, w, D, H, seed=1)
    g = oracle.softmax(np.random.default_rng(0).standard_normal((B, H, h * w)))
    assert np.abs(oracle.circ2d_direct(g, V, h, w) - oracle.circ_direct(g, V)).max() <= 1e-14
    a = oracle.corr2d_direct(Q, K, H, h, w, scale=1.0)
    assert np.abs(a - oracle.corr_direct(Q, K, H)).max() <= 1e-12


@pytest.mark.parametrize("h,w", [(2, 3), (3, 4), (4, 4), (5, 2)])
def test_bccb_matrix_brute_force(h, w):
    B, D, H = 1, 4, 2
    _, _, V = _qkv(B, h, w, D, H, seed=h * w)
    g = oracle.softmax(np.random.default_rng(h).standard_normal((B, H, h * w)))
    O = oracle.circ2d_direct(g, V, h, w)
    Of = oracle.circ2d_fft(g, V, h, w)
    for c in range(D):
        M = oracle.bccb_matrix(g[0, c // (D // H)].reshape(h, w))
        ref = M @ V[0, :, c]
        assert np.abs(O[0, :, c] - ref).max() <= 1e-14
        assert np.abs(Of[0, :, c] - ref).max() <= 1e-13


def test_bccb_matrix_is_block_circulant_with_circulant_blocks():
    g = np.arange(12, dtype=np.float64).reshape(3, 4)
    M = oracle.bccb_matrix(g)
    h, w = g.shape
    blocks = [[M[i * w:(i + 1) * w, j * w:(j + 1) * w] for j in range(h)] for i in range(h)]
    for i in range(h):
        for j in range(h):
            assert np.array_equal(blocks[i][j], blocks[(i + 1) % h][(j + 1) % h])  # block circulant
            blk = blocks[i][j]
            for r in range(w):
                assert np.array_equal(np.roll(blk[r], 1), blk[(r + 1) % w])      # circulant blocks


@pytest.mark.parametrize("h,w", [(3, 5), (4, 4), (2, 7)])
def test_scores_are_diagonal_sums_of_qkt(h, w):
    """a[k] = (1/dh) Σ over token pairs (i, j) with i ⊖ j = k of (Q K^T)[i, j]."""
    B, D, H = 1, 6, 2
    dh = D // H
    Q, K, _ = _qkv(B, h, w, D, H, seed=3)
    a = oracle.corr2d_direct(Q, K, H, h, w)
    N = h * w
    n = np.arange(N)
    lag = ((n[:, None] // w - n[None, :] // w) % h) * w + (n[:, None] % w - n[None, :] % w) % w
    for hd in range(H):
        S = Q[0, :, hd * dh:(hd + 1) * dh] @ K[0, :, hd * dh:(hd + 1) * dh].T
        ref = np.array([S[lag == k].sum() for k in range(N)]) / dh
        assert np.abs(a[0, hd] - ref).max() <= 1e-12


def test_separable_generator():
    """g = u ⊗ v: the 2-D convolution is a 1-D convolution along y by u of
    a 1-D convolution along x by v."""
    h, w, D = 4, 6, 2
    rng = np.random.default_rng(5)
    u, v = rng.random(h), rng.random(w)
    g = np.outer(u, v).reshape(1, 1, h * w)
    V = rng.standard_normal((1, h * w, D))
    O = oracle.circ2d_direct(g, V, h, w)
    Vg = V.reshape(h, w, D)
    ref = np.zeros_like(Vg)
    for y in range(h):
        for x in range(w):
            for yy in range(h):
                for xx in range(w):
                    ref[y, x] += u[(y - yy) % h] * v[(x - xx) % w] * Vg[yy, xx]
    assert np.abs(O.reshape(h, w, D) - ref).max() <= 1e-13


@pytest.mark.parametrize("sy,sx", [(0, 0), (1, 2), (3, 0)])
def test_one_hot_generator_is_2d_shift(sy, sx):
    h, w, D = 4, 5, 3
    g = np.zeros((1, 1, h * w))
    g[0, 0, sy * w + sx] = 1.0
    V = np.random.default_rng(2).standard_normal((1, h * w, D))
    ref = np.roll(V.reshape(h, w, D), (sy, sx), axis=(0, 1)).reshape(1, h * w, D)
    assert np.array_equal(oracle.circ2d_direct(g, V, h, w), ref)
    assert np.abs(oracle.circ2d_fft(g, V, h, w) - ref).max() <= 1e-14


def test_uniform_generator_gives_mean():
    h, w, D = 3, 7, 4
    g = np.full((2, 2, h * w), 1.0 / (h * w))
    V = np.random.default_rng(3).standard_normal((2, h * w, D))
    O = oracle.circ2d_direct(g, V, h, w)
    assert np.abs(O - V.mean(axis=1, keepdims=True)).max() <= 1e-14


@pytest.mark.parametrize("h,w", [(14, 14), (7, 12), (8, 8), (5, 1), (6, 10)])
def test_direct_equals_fft(h, w):
    B, D, H = 2, 8, 2
    Q, K, V = _qkv(B, h, w, D, H, seed=h + w)
    O1, a1, z1 = oracle.forward2d(Q, K, V, H, h, w, "direct")
    O2, a2, z2 = oracle.forward2d(Q, K, V, H, h, w, "fft")
    assert np.abs(a1 - a2).max() <= 1e-12 * (1 + np.abs(a1).max())
    assert np.abs(O1 - O2).max() <= 1e-12 * (1 + np.abs(V).max())
    assert np.allclose(z1.sum(-1), 1.0, rtol=0, atol=1e-14)
    # a BCCB generator that sums to one keeps every column sum
    assert np.abs(O1.sum(axis=1) - V.sum(axis=1)).max() <= 1e-11 * h * w
