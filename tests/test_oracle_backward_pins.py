"""Pins of the fp64 oracle's backward pass against what the mathematics fixes
(no GPU).

The page trains CAT layers with the usual losses and optimisers ("CAT:
Circular-Convolutional Attention for Sub-Quadratic Transformers", section
损失函数 / 训练策略, loss and training strategy) but prints no gradients, so
the backward is the chain rule through the forward definitions of section
方法详解 (designs "circulant attention matrix construction" and "FFT
acceleration").  The pins tie it to things other than its own formulas:

* exact symbolic derivatives (sympy) of the forward definition for tiny
  shapes, and central finite differences of the (separately pinned) forward
  oracle for the loss L = sum(O ⊙ G): every gradient, and dL/dz* with z*
  perturbed directly;
* the adjoint (dot-product) identity <circ(z*) V, G> = <V, circ(z*)^T G>;
* brute force: the explicit N x N circulant transposed, and numpy's roll;
* closed forms: the 2-token softmax, uniform and one-hot z*;
* library matmuls (numpy einsum) for the two dense contractions;
* agreement of the O(N^2) definitions with the FFT evaluations.

A plausible mistake — the transpose taken the wrong way round, the
correlation's lag reversed, the softmax Jacobian's mean term dropped, a
conjugate missing in a spectrum product, W_A read transposed — fails at
least one of them (test_oracle_mutants.py plants each and checks).
"""
import numpy as np
import pytest

import oracle
import synth


def _loss(X, WA, V, G):
    O, _ = oracle.forward(X, WA, V, mode="direct")
    return float(np.sum(O * G))


def _inputs(B, N, D, H, seed=0, wa_scale=1.0):
    X, WA, V = (t.double().numpy() for t in synth.make_inputs(B, N, D, H, "f32", seed, wa_scale))
    G = synth.make_grad(B, N, D, "f32", seed).double().numpy()
    return X, WA, V, G


def _fd(f, A, eps=1e-6):
    """Central differences of the scalar f() in every entry of array A."""
    out = np.empty_like(A)
    flat, g = A.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        keep = flat[i]
        flat[i] = keep + eps
        fp = f()
        flat[i] = keep - eps
        fm = f()
        flat[i] = keep
        g[i] = (fp - fm) / (2 * eps)
    return out


SHAPES = [(2, 6, 4, 2), (1, 5, 6, 3), (1, 7, 2, 1), (1, 9, 3, 1)]


@pytest.mark.parametrize("B,N,D,H", SHAPES)
@pytest.mark.parametrize("mode", ["direct", "fft"])
def test_gradients_match_finite_differences(B, N, D, H, mode):
    X, WA, V, G = _inputs(B, N, D, H, seed=3, wa_scale=2.0)
    g = oracle.backward(X, WA, V, G, mode)
    f = lambda: _loss(X, WA, V, G)
    for name, A in (("dX", X), ("dWA", WA), ("dV", V)):
        num = _fd(f, A)
        assert np.abs(g[name] - num).max() <= 1e-6 * (1 + np.abs(num).max()), name


@pytest.mark.parametrize("N", [4, 5, 8])
def test_dzstar_matches_finite_differences(N):
    """dL/dz*[k] with z* perturbed directly in the forward circulant product."""
    B, D, H = 2, 4, 2
    X, WA, V, G = _inputs(B, N, D, H, seed=5)
    zs = oracle.zstar(X, WA)
    f = lambda: float(np.sum(oracle.circ_direct(zs, V) * G))
    num = _fd(f, zs)
    for dzs in (oracle.corr_direct(G, V, H), oracle.corr_fft(G, V, H)):
        assert np.abs(dzs - num).max() <= 1e-7 * (1 + np.abs(num).max())


@pytest.mark.parametrize("N", [2, 3, 7])
def test_softmax_backward_matches_finite_differences(N):
    rng = np.random.default_rng(11)
    z = rng.standard_normal((3, N)) * 2
    g = rng.standard_normal((3, N))
    f = lambda: float(np.sum(oracle.softmax(z) * g))
    num = _fd(f, z)
    dz = oracle.softmax_backward(oracle.softmax(z), g)
    assert np.abs(dz - num).max() <= 1e-8


def test_softmax_backward_two_tokens_closed_form():
    """z = (a, b): z*_0 = p = 1/(1+e^{b-a});  dL/da = p(1-p)(g0-g1) = -dL/db."""
    a, b, g0, g1 = 0.3, -1.1, 2.0, -0.5
    p = 1.0 / (1.0 + np.exp(b - a))
    zs = np.array([[p, 1 - p]])
    dz = oracle.softmax_backward(zs, np.array([[g0, g1]]))
    ref = p * (1 - p) * (g0 - g1)
    assert np.allclose(dz[0], [ref, -ref], atol=1e-15)


def test_softmax_backward_is_orthogonal_to_constants():
    """softmax(z + c) = softmax(z), so every dL/dz row sums to zero."""
    rng = np.random.default_rng(2)
    zs = oracle.softmax(rng.standard_normal((4, 33)) * 3)
    dz = oracle.softmax_backward(zs, rng.standard_normal((4, 33)))
    assert np.abs(dz.sum(axis=1)).max() <= 1e-14


@pytest.mark.parametrize("N", [1, 2, 3, 8, 13, 16])
def test_transpose_brute_force(N):
    """dV = circ(z*)^T G with the N x N matrix built explicitly."""
    B, D, H = 1, 4, 2
    X, WA, V, G = _inputs(B, N, D, H, seed=N)
    zs = oracle.zstar(X, WA)
    dV = oracle.circ_transpose_direct(zs, G)
    dVf = oracle.circ_transpose_fft(zs, G)
    for c in range(D):
        M = oracle.brute_circulant(zs[0, c // (D // H)])
        ref = M.T @ G[0, :, c]
        assert np.abs(dV[0, :, c] - ref).max() <= 1e-14
        assert np.abs(dVf[0, :, c] - ref).max() <= 1e-12


@pytest.mark.parametrize("N", [1, 2, 6, 11, 16])
def test_correlation_by_roll(N):
    """dz*[k] = sum_c <G[:, c], roll(V[:, c], k)>, roll(v, k)[i] = v[i - k]."""
    B, D, H = 2, 6, 3
    _, _, V, G = _inputs(B, N, D, H, seed=7)
    dzs = oracle.corr_direct(G, V, H)
    dh = D // H
    for b in range(B):
        for h in range(H):
            for k in range(N):
                ref = sum(np.dot(G[b, :, c], np.roll(V[b, :, c], k))
                          for c in range(h * dh, (h + 1) * dh))
                assert abs(dzs[b, h, k] - ref) <= 1e-13 * (1 + abs(ref))


@pytest.mark.parametrize("N,mode", [(8, "direct"), (196, "fft"), (64, "fft")])
def test_adjoint_identity(N, mode):
    """<circ(z*) V, G> = <V, circ(z*)^T G> for every (b, head)."""
    B, D, H = 2, 8, 2
    X, WA, V, G = _inputs(B, N, D, H, seed=1)
    zs = oracle.zstar(X, WA)
    O = oracle.circ_direct(zs, V) if mode == "direct" else oracle.circ_fft(zs, V)
    dV = oracle.circ_transpose_direct(zs, G) if mode == "direct" else oracle.circ_transpose_fft(zs, G)
    lhs, rhs = np.sum(O * G), np.sum(V * dV)
    assert abs(lhs - rhs) <= 1e-12 * np.sum(np.abs(O * G))


def test_uniform_zstar_gives_column_mean():
    """W_A = 0 makes z* = 1/N, so dV[j, c] = mean_i G[i, c] for every j."""
    B, N, D, H = 2, 10, 4, 2
    X, WA, V, G = _inputs(B, N, D, H)
    WA[:] = 0
    for mode in ("direct", "fft"):
        g = oracle.backward(X, WA, V, G, mode)
        assert np.abs(g["dV"] - G.mean(axis=1, keepdims=True)).max() <= 1e-14


@pytest.mark.parametrize("s", [0, 1, 5])
def test_one_hot_zstar_is_reverse_shift(s):
    """z* = e_s: O[i] = V[i - s], so dV[j] = G[(j + s) mod N]."""
    N, D = 8, 4
    zs = np.zeros((1, 1, N))
    zs[0, 0, s] = 1.0
    G = synth.make_grad(1, N, D, "f32", 4).double().numpy()
    ref = np.roll(G, -s, axis=1)
    assert np.abs(oracle.circ_transpose_direct(zs, G) - ref).max() == 0
    assert np.abs(oracle.circ_transpose_fft(zs, G) - ref).max() <= 1e-14


def test_mean_term_equals_output_inner_product():
    """sum_m z*[m] dz*[m] = sum_{i, c in h} G[i, c] O[i, c] (both are dL along z*)."""
    B, N, D, H = 2, 12, 6, 3
    X, WA, V, G = _inputs(B, N, D, H, seed=9, wa_scale=3.0)
    g = oracle.backward(X, WA, V, G, "direct")
    O, zs = oracle.forward(X, WA, V, "direct")
    dh = D // H
    for b in range(B):
        for h in range(H):
            lhs = np.dot(zs[b, h], g["dzs"][b, h])
            rhs = np.sum(G[b, :, h * dh:(h + 1) * dh] * O[b, :, h * dh:(h + 1) * dh])
            assert abs(lhs - rhs) <= 1e-12 * (1 + abs(rhs))


def test_dense_contractions_match_library_matmul():
    B, N, D, H = 3, 10, 12, 4
    X, WA, _, _ = _inputs(B, N, D, H)
    dz = np.random.default_rng(0).standard_normal((B, H, N))
    assert np.allclose(oracle.grad_wa(X, dz), np.einsum("bnd,bhn->dh", X, dz), rtol=0, atol=1e-12)
    assert np.allclose(oracle.grad_x(dz, WA), np.einsum("bhn,dh->bnd", dz, WA), rtol=0, atol=1e-13)


@pytest.mark.parametrize("B,N,D,H", [(1, 196, 12, 2), (1, 256, 8, 2), (1, 1000, 4, 1), (2, 64, 6, 3)])
def test_direct_equals_fft(B, N, D, H):
    X, WA, V, G = _inputs(B, N, D, H, seed=2, wa_scale=4.0)
    a = oracle.backward(X, WA, V, G, "direct")
    b = oracle.backward(X, WA, V, G, "fft")
    for k in ("dV", "dzs", "dz", "dX", "dWA"):
        assert np.abs(a[k] - b[k]).max() <= 1e-12 * (1 + np.abs(a[k]).max()), k
    _, mi = oracle.corr_fft(G, V, H, return_max_imag=True)
    assert mi <= 1e-12 * (1 + np.abs(a["dzs"]).max())


def test_sampled_rows_and_bins_match_full():
    B, N, D, H = 2, 30, 6, 2
    X, WA, V, G = _inputs(B, N, D, H)
    zs = oracle.zstar(X, WA)
    rows = [0, 7, 29]
    assert np.array_equal(oracle.circ_transpose_direct_rows(zs, G, rows),
                          oracle.circ_transpose_direct(zs, G)[:, rows])
    assert np.array_equal(oracle.corr_direct_bins(G, V, H, rows),
                          oracle.corr_direct(G, V, H)[:, :, rows])


@pytest.mark.parametrize("N,D,H", [(3, 2, 1), (3, 2, 2), (4, 2, 1)])
def test_gradients_match_symbolic_differentiation(N, D, H):
    """Exact gradients: sympy differentiates the forward definition (scores,
    softmax over tokens, circulant product) of L = Σ O ⊙ G symbolically; the
    oracle's chain rule must agree to rounding."""
    sp = pytest.importorskip("sympy")
    rng = np.random.default_rng(N * 10 + D + H)
    dh = D // H
    Xn = np.round(rng.standard_normal((N, D)), 2)
    Wn = np.round(rng.standard_normal((D, H)), 2)
    Vn = np.round(rng.standard_normal((N, D)), 2)
    Gn = np.round(rng.standard_normal((N, D)), 2)
    X = sp.Matrix(N, D, lambda i, j: sp.Symbol("x_%d_%d" % (i, j)))
    W = sp.Matrix(D, H, lambda i, j: sp.Symbol("w_%d_%d" % (i, j)))
    V = sp.Matrix(N, D, lambda i, j: sp.Symbol("v_%d_%d" % (i, j)))
    L = 0
    for h in range(H):
        z = [sum(X[n, d] * W[d, h] for d in range(D)) for n in range(N)]
        e = [sp.exp(t) for t in z]
        s = sum(e)
        zs = [t / s for t in e]
        for i in range(N):
            for c in range(h * dh, (h + 1) * dh):
                O = sum(zs[(i - j) % N] * V[j, c] for j in range(N))
                L += O * sp.Rational(str(Gn[i, c]))
    subs = {X[i, j]: sp.Rational(str(Xn[i, j])) for i in range(N) for j in range(D)}
    subs.update({W[i, j]: sp.Rational(str(Wn[i, j])) for i in range(D) for j in range(H)})
    subs.update({V[i, j]: sp.Rational(str(Vn[i, j])) for i in range(N) for j in range(D)})
    g = oracle.backward(Xn[None], Wn, Vn[None], Gn[None], "direct")
    for name, M, shape in (("dX", X, (N, D)), ("dWA", W, (D, H)), ("dV", V, (N, D))):
        ref = np.array([[float(sp.N(sp.diff(L, M[i, j]).subs(subs), 30))
                         for j in range(shape[1])] for i in range(shape[0])])
        got = g[name][0] if name != "dWA" else g[name]
        assert np.abs(got - ref).max() <= 1e-12 * (1 + np.abs(ref).max()), name
