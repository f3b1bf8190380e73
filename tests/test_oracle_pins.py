"""Pins of the fp64 oracle against what the mathematics fixes (no GPU).

Each test ties the oracle to something other than itself: a hand-worked
example, a closed form, an invariant the CAT notes page states, a library
routine computing the same textbook quantity, or brute force.  Together they
are chosen so that a plausible mistake — a wrong shift direction, a missing
1/N, a transposed W_A, the softmax over the wrong axis, columns assigned to
the wrong head, a wrong twiddle sign — fails at least one of them.

Page cited throughout: "CAT: Circular-Convolutional Attention for
Sub-Quadratic Transformers", section 方法详解 (method), designs "circulant
attention matrix construction" and "FFT acceleration".
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = rest.strip()

    def num(tok):
        if tok.startswith("ln"):
            return math.log(float(tok[2:]))
        return float(Fraction(tok))

    def arr(s):
        rows = [r.split() for r in s.split(";")]
        return np.array([[num(t) for t in r] for r in rows], dtype=np.float64)

    return vals, arr


# --------------------------------------------------------------------------
# Worked example (hand-computed; see the fixture for the derivation)
# --------------------------------------------------------------------------

def test_worked_example_n4():
    vals, arr = _parse_golden("worked_example_n4.txt")
    X = arr(vals["X"])[None]          # [1, 4, 2]
    WA = arr(vals["W_A"])             # [2, 1]
    V = arr(vals["V"])[None]          # [1, 4, 2]
    zs_ref = arr(vals["Zstar"])       # [1, 4]
    O_ref = arr(vals["O"])            # [4, 2]
    for mode in ("direct", "fft"):
        O, zs = oracle.forward(X, WA, V, mode=mode)
        np.testing.assert_allclose(zs[0], zs_ref, rtol=0, atol=1e-15)
        np.testing.assert_allclose(O[0], O_ref, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# The DFT used by the FFT mode
# --------------------------------------------------------------------------

SIZES = [1, 2, 3, 4, 5, 6, 7, 8, 12, 15, 16, 49, 64, 196, 210, 256, 343, 1000,
         1024, 4096]


@pytest.mark.parametrize("N", SIZES)
def test_dft_matches_library_fft(N):
    """Same textbook quantity as numpy's pocketfft, forward and inverse."""
    rng = np.random.default_rng(N)
    x = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    scale = max(1.0, math.sqrt(N))
    np.testing.assert_allclose(oracle.dft(x), np.fft.fft(x), rtol=0,
                               atol=1e-12 * scale * math.log2(N + 1))
    np.testing.assert_allclose(oracle.dft(x, inverse=True), np.fft.ifft(x),
                               rtol=0, atol=1e-13 * math.log2(N + 1))


@pytest.mark.parametrize("N", [1, 2, 7, 12, 64, 196])
def test_dft_closed_forms(N):
    """DFT(delta_0) = 1; DFT(1) = N·delta_0; DFT(exp(+2πi m n/N)) = N·delta_m;
    a delayed delta gives exp(-2πi k s/N) (forward sign)."""
    n = np.arange(N)
    delta = np.zeros(N, complex)
    delta[0] = 1
    np.testing.assert_allclose(oracle.dft(delta), np.ones(N), atol=1e-14)
    ones = np.ones(N, complex)
    expect = np.zeros(N, complex)
    expect[0] = N
    np.testing.assert_allclose(oracle.dft(ones), expect, atol=1e-12 * N)
    m = (3 * N) // 4 if N > 1 else 0
    tone = np.exp(2j * np.pi * m * n / N)
    expect = np.zeros(N, complex)
    expect[m] = N
    np.testing.assert_allclose(oracle.dft(tone), expect, atol=1e-11 * N)
    s = N // 3
    shifted = np.zeros(N, complex)
    shifted[s] = 1
    k = np.arange(N)
    np.testing.assert_allclose(oracle.dft(shifted),
                               np.exp(-2j * np.pi * k * s / N), atol=1e-13)


def test_dft_roundtrip():
    rng = np.random.default_rng(5)
    for N in (196, 1024, 1 << 15):
        x = rng.standard_normal(N) + 1j * rng.standard_normal(N)
        np.testing.assert_allclose(oracle.dft(oracle.dft(x), inverse=True), x,
                                   atol=1e-12)


# --------------------------------------------------------------------------
# Score and softmax
# --------------------------------------------------------------------------

def test_scores_match_library_matmul():
    """z[b,h,n] = sum_d X[b,n,d] W_A[d,h], against numpy's einsum; H > 1 and
    D != H so that a transposed W_A index cannot pass."""
    X, WA, _ = synth.make_inputs(2, 33, 24, 3, "f32", seed=1)
    Xn, Wn = X.double().numpy(), WA.double().numpy()
    z = oracle.scores(Xn, Wn)
    assert z.shape == (2, 3, 33)
    np.testing.assert_allclose(z, np.einsum("bnd,dh->bhn", Xn, Wn),
                               rtol=1e-13, atol=1e-13)


def test_scores_one_hot_rows():
    """A one-hot token row picks a row of W_A."""
    D, H = 5, 3
    WA = np.arange(D * H, dtype=np.float64).reshape(D, H) - 7.0
    X = np.zeros((1, D, D))
    X[0, np.arange(D), np.arange(D)] = 1.0      # token n = e_n
    z = oracle.scores(X, WA)
    np.testing.assert_array_equal(z[0], WA.T)


def test_softmax_two_tokens_closed_form():
    """For two tokens z* = (1/(1+e^{b-a}), 1/(1+e^{a-b}))."""
    for a, b in [(0.0, 0.0), (1.5, -2.0), (-30.0, 40.0), (700.0, 0.0)]:
        zs = oracle.softmax(np.array([[a, b]]))
        np.testing.assert_allclose(
            zs[0], [1 / (1 + math.exp(min(b - a, 700))),
                    1 / (1 + math.exp(min(a - b, 700)))], rtol=1e-15, atol=1e-300)


def test_softmax_known_values_and_shift_invariance():
    z = np.log(np.array([[1.0, 2.0, 1.0, 4.0]]))
    np.testing.assert_allclose(oracle.softmax(z)[0], [1 / 8, 2 / 8, 1 / 8, 4 / 8],
                               atol=1e-16)
    rng = np.random.default_rng(2)
    z = rng.standard_normal((3, 50)) * 9
    np.testing.assert_allclose(oracle.softmax(z), oracle.softmax(z + 123.25),
                               rtol=1e-13)
    s = oracle.softmax(z)
    np.testing.assert_allclose(s.sum(-1), 1.0, atol=1e-14)
    assert (s > 0).all()


def test_softmax_axis_is_tokens():
    """Each (b, h) row is normalised over N, never across heads."""
    X, WA, _ = synth.make_inputs(2, 20, 8, 4, "f32", seed=3)
    zs = oracle.zstar(X, WA)
    assert zs.shape == (2, 4, 20)
    np.testing.assert_allclose(zs.sum(-1), 1.0, atol=1e-14)
    z = oracle.scores(X, WA)
    ref = np.exp(z - z.max(-1, keepdims=True))
    np.testing.assert_allclose(zs, ref / ref.sum(-1, keepdims=True), rtol=1e-13)


# --------------------------------------------------------------------------
# The circulant operator
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 13, 33, 64])
def test_softmax_commutes_with_circulant(N):
    """softmax(circ(z)) == circ(softmax(z)) entry-wise: the property stated in
    the circulant-construction design (each row of circ(z) permutes z)."""
    z = np.random.default_rng(N).standard_normal(N) * 4
    lhs = oracle.softmax(oracle.brute_circulant(z))
    rhs = oracle.brute_circulant(oracle.softmax(z[None])[0])
    np.testing.assert_allclose(lhs, rhs, rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("N", list(range(1, 17)))
def test_brute_force_small_n(N):
    """All three evaluations agree for every N <= 16 (primes included):
    the explicit N x N matrix times V, the O(N^2) sum, and the FFT path."""
    B, D, H = 2, 4, 2
    X, WA, V = synth.make_inputs(B, N, D, H, "f32", seed=N)
    zs = oracle.zstar(X, WA)
    Vn = V.double().numpy()
    dh = D // H
    ref = np.empty((B, N, D))
    for b in range(B):
        for c in range(D):
            ref[b, :, c] = oracle.brute_circulant(zs[b, c // dh]) @ Vn[b, :, c]
    np.testing.assert_allclose(oracle.circ_direct(zs, Vn), ref, rtol=0, atol=1e-14)
    np.testing.assert_allclose(oracle.circ_fft(zs, Vn), ref, rtol=0, atol=1e-13)


def test_rows_and_columns_of_circulant_sum_to_one():
    z = oracle.softmax(np.random.default_rng(9).standard_normal((1, 37)) * 3)[0]
    C = oracle.brute_circulant(z)
    np.testing.assert_allclose(C.sum(1), 1.0, atol=1e-15)
    np.testing.assert_allclose(C.sum(0), 1.0, atol=1e-15)
    # Every row is the previous row cyclically shifted by one place, and
    # column j is z* cyclically shifted by j (the orientation the convolution
    # theorem fixes: circ[i, j] = z*[(i - j) mod N]).
    for i in range(36):
        np.testing.assert_array_equal(C[i + 1], np.roll(C[i], 1))
    for j in range(37):
        np.testing.assert_array_equal(C[:, j], np.roll(z, j))


@pytest.mark.parametrize("mode", ["direct", "fft"])
def test_convex_combination_properties(mode):
    """Each output is a convex combination of its column: column sums are
    kept and every output lies within [min V, max V] of its column."""
    X, WA, V = synth.make_inputs(2, 48, 12, 3, "f32", seed=4, wa_scale=3.0)
    O, _ = oracle.forward(X, WA, V, mode=mode)
    Vn = V.double().numpy()
    np.testing.assert_allclose(O.sum(1), Vn.sum(1), atol=1e-12)
    assert (O <= Vn.max(1, keepdims=True) + 1e-12).all()
    assert (O >= Vn.min(1, keepdims=True) - 1e-12).all()


def test_spectrum_dc_and_bound():
    """Zf[0] = sum z* = 1 and |Zf[k]| <= 1 for a probability vector."""
    X, WA, _ = synth.make_inputs(2, 196, 16, 2, "f32", seed=6, wa_scale=4.0)
    zf = oracle.spectrum(oracle.zstar(X, WA))
    np.testing.assert_allclose(zf[..., 0], 1.0, atol=1e-14)
    assert (np.abs(zf) <= 1 + 1e-13).all()


def _one_hot_inputs(N, D, H, shifts, dtype="f32"):
    """X, W_A built so that z* of head h is exactly one-hot at shifts[h]:
    W_A[:, h] = e_h and X[n, h] = -100 except X[shifts[h], h] = +100."""
    _, _, V = synth.make_inputs(1, N, D, H, dtype, seed=11)
    X = np.zeros((1, N, D))
    WA = np.zeros((D, H))
    for h, s in enumerate(shifts):
        WA[h, h] = 1.0
        X[0, :, h] = -100.0
        X[0, s, h] = 100.0
    return X, WA, V.double().numpy()


@pytest.mark.parametrize("mode", ["direct", "fft"])
def test_one_hot_is_cyclic_shift(mode):
    """A one-hot z* = e_s gives O[i] = V[(i - s) mod N]: pins the shift
    direction, and (with a different s per head) the column-to-head map."""
    N, D, H = 40, 8, 4
    shifts = [0, 1, 7, 33]
    X, WA, V = _one_hot_inputs(N, D, H, shifts)
    O, zs = oracle.forward(X, WA, V, mode=mode)
    dh = D // H
    for h, s in enumerate(shifts):
        assert zs[0, h, s] == 1.0
        cols = slice(h * dh, (h + 1) * dh)
        np.testing.assert_allclose(O[0, :, cols], np.roll(V[0, :, cols], s, axis=0),
                                   atol=1e-13)


@pytest.mark.parametrize("mode", ["direct", "fft"])
def test_uniform_gives_column_mean(mode):
    """W_A = 0 makes z* uniform, so every output row is the column mean."""
    X, _, V = synth.make_inputs(3, 27, 6, 3, "f32", seed=12)
    WA = np.zeros((6, 3))
    O, zs = oracle.forward(X, WA, V, mode=mode)
    np.testing.assert_allclose(zs, 1 / 27, atol=1e-16)
    Vn = V.double().numpy()
    np.testing.assert_allclose(O, np.broadcast_to(Vn.mean(1, keepdims=True), O.shape),
                               atol=1e-14)


def test_shift_equivariance():
    """Rolling V by s rolls O by s; rolling X and V by s rolls O by 2s."""
    X, WA, V = synth.make_inputs(1, 30, 6, 2, "f32", seed=13)
    Xn, Vn = X.double().numpy(), V.double().numpy()
    O, _ = oracle.forward(Xn, WA, Vn, mode="direct")
    s = 7
    O1, _ = oracle.forward(Xn, WA, np.roll(Vn, s, axis=1), mode="direct")
    np.testing.assert_allclose(O1, np.roll(O, s, axis=1), atol=1e-13)
    O2, _ = oracle.forward(np.roll(Xn, s, axis=1), WA, np.roll(Vn, s, axis=1),
                           mode="fft")
    np.testing.assert_allclose(O2, np.roll(O, 2 * s, axis=1), atol=1e-13)


def test_linearity_in_v():
    X, WA, V1 = synth.make_inputs(1, 21, 4, 2, "f32", seed=14)
    _, _, V2 = synth.make_inputs(1, 21, 4, 2, "f32", seed=15)
    V1, V2 = V1.double().numpy(), V2.double().numpy()
    zs = oracle.zstar(X, WA)
    a, b = 1.75, -0.5
    np.testing.assert_allclose(
        oracle.circ_direct(zs, a * V1 + b * V2),
        a * oracle.circ_direct(zs, V1) + b * oracle.circ_direct(zs, V2), atol=1e-13)


# --------------------------------------------------------------------------
# Convolution theorem at the shapes of the workloads (reduced batch)
# --------------------------------------------------------------------------

CONV_CASES = [
    ("tiny", dict(B=1, N=256, D=64, H=2, dtype="f32")),
    ("vit196", dict(B=2, N=196, D=384, H=6, dtype="f32")),
    ("gpt2", dict(B=1, N=1024, D=96, H=12, dtype="bf16")),
    ("gpt2_peaked", dict(B=1, N=1024, D=96, H=12, dtype="f32", wa_scale=8.0)),
    ("long_slice", dict(B=1, N=4096, D=16, H=2, dtype="bf16")),
]


@pytest.mark.parametrize("name,cfg", CONV_CASES, ids=[c[0] for c in CONV_CASES])
def test_convolution_theorem(name, cfg):
    """The direct circulant product equals IFFT(FFT(z*) ⊙ FFT(V)) to fp64
    rounding (the "FFT acceleration" design calls the two exactly equal)."""
    cfg = dict(cfg)
    scale = cfg.pop("wa_scale", 1.0)
    X, WA, V = synth.make_inputs(wa_scale=scale, **cfg)
    zs = oracle.zstar(X, WA)
    Vn = V.double().numpy()
    Od = oracle.circ_direct(zs, Vn)
    Of, max_imag = oracle.circ_fft(zs, Vn, return_max_imag=True)
    vmax = np.abs(Vn).max()
    assert np.abs(Od - Of).max() <= 1e-12 * vmax
    assert max_imag <= 1e-12 * vmax


def test_direct_rows_match_full_direct():
    X, WA, V = synth.make_inputs(2, 64, 8, 2, "f32", seed=16)
    zs = oracle.zstar(X, WA)
    rows = [0, 5, 63, 31]
    full = oracle.circ_direct(zs, V)
    np.testing.assert_array_equal(oracle.circ_direct_rows(zs, V, rows), full[:, rows])


def test_peaked_softmax_is_finite_and_normalised():
    """W_A x 8 (near one-hot rows): no overflow, still sums to one."""
    X, WA, _ = synth.make_inputs(1, 1024, 768, 12, "bf16", wa_scale=8.0)
    zs = oracle.zstar(X, WA)
    assert np.isfinite(zs).all() and (zs >= 0).all()
    np.testing.assert_allclose(zs.sum(-1), 1.0, atol=1e-13)
    assert zs.max() > 0.5      # peaked


# --------------------------------------------------------------------------
# Value projection V = X · W_V (the fused-projection entry's first product)
# --------------------------------------------------------------------------

def test_projection_against_explicit_sums():
    """oracle.project against the sum written out term by term, and the
    identity and linearity it must have (section 整体框架: V = X·W_V)."""
    rng = np.random.default_rng(31)
    X = rng.standard_normal((2, 5, 6))
    W = rng.standard_normal((6, 4))
    V = oracle.project(X, W)
    for b in range(2):
        for n in range(5):
            for e in range(4):
                s = 0.0
                for d in range(6):
                    s += X[b, n, d] * W[d, e]
                assert abs(V[b, n, e] - s) <= 1e-13 * (1 + abs(s))
    np.testing.assert_array_equal(oracle.project(X, np.eye(6)), X)
    W2 = rng.standard_normal((6, 4))
    np.testing.assert_allclose(oracle.project(X, 2 * W - W2), 2 * V - oracle.project(X, W2),
                               atol=1e-12)
