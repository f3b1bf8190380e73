"""fp64 CPU oracle for the CAT forward and backward passes — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its binding)
never does, and this package never imports the product.  It shares nothing
with the CUDA side except the seeded input generator in ``synth``.

What it computes (notes page "CAT: Circular-Convolutional Attention for
Sub-Quadratic Transformers", section 方法详解, designs "circulant attention
matrix construction" and "FFT acceleration"):

    z  = X · W_A              z[b, h, n]
    z* = softmax_n(z)         over the N tokens of each (b, h)
    O  = circ(z*) · V_h       circ(z*)[i, j] = z*[(i - j) mod N]
       = IFFT(FFT(z*) ⊙ FFT(V_h))   column by column

The backward pass (gradients of a loss L given G = dL/dO) follows from
these definitions by the chain rule; the page trains CAT layers with the
usual losses (section 损失函数 / 训练策略) but prints no gradient formulas:

    dV   = circ(z*)^T G                       dV[j, c] = sum_i z*[(i-j) mod N] G[i, c]
    dz*  = sum_{c in h} corr(G[:, c], V[:, c])  dz*[k] = sum_c sum_i G[i, c] V[(i-k) mod N, c]
    dz   = z* ⊙ (dz* - <z*, dz*>)             softmax Jacobian
    dW_A = X^T dz,   dX = dz W_A^T

All arithmetic is fp64 in ``cat_oracle.c``; this module only marshals numpy
arrays.  ``brute_circulant`` builds the N x N matrix explicitly (tiny N only)
and multiplies with numpy, so it is an independent third evaluation.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        L = ctypes.c_long
        lib.oracle_scores.argtypes = [dp, dp, L, L, L, L, dp]
        lib.oracle_scores.restype = None
        lib.oracle_softmax.argtypes = [dp, dp, L, L]
        lib.oracle_softmax.restype = None
        lib.oracle_circ_direct.argtypes = [dp, dp, L, L, L, L, dp]
        lib.oracle_circ_direct.restype = None
        lib.oracle_circ_direct_rows.argtypes = [dp, dp, L, L, L, L, lp, L, dp]
        lib.oracle_circ_direct_rows.restype = None
        lib.oracle_dft.argtypes = [dp, dp, L, ctypes.c_int]
        lib.oracle_dft.restype = ctypes.c_int
        lib.oracle_circ_fft.argtypes = [dp, dp, L, L, L, L, dp, dp]
        lib.oracle_circ_fft.restype = ctypes.c_int
        lib.oracle_spectrum.argtypes = [dp, L, L, dp]
        lib.oracle_spectrum.restype = ctypes.c_int
        lib.oracle_circ_transpose_direct.argtypes = [dp, dp, L, L, L, L, dp]
        lib.oracle_circ_transpose_direct.restype = None
        lib.oracle_circ_transpose_direct_rows.argtypes = [dp, dp, L, L, L, L, lp, L, dp]
        lib.oracle_circ_transpose_direct_rows.restype = None
        lib.oracle_corr_direct_bins.argtypes = [dp, dp, L, L, L, L, lp, L, dp]
        lib.oracle_corr_direct_bins.restype = None
        lib.oracle_softmax_backward.argtypes = [dp, dp, L, L, dp]
        lib.oracle_softmax_backward.restype = None
        lib.oracle_grad_wa.argtypes = [dp, dp, L, L, L, L, dp]
        lib.oracle_grad_wa.restype = None
        lib.oracle_grad_x.argtypes = [dp, dp, L, L, L, L, dp]
        lib.oracle_grad_x.restype = None
        lib.oracle_circ_transpose_fft.argtypes = [dp, dp, L, L, L, L, dp]
        lib.oracle_circ_transpose_fft.restype = ctypes.c_int
        lib.oracle_corr_fft.argtypes = [dp, dp, L, L, L, L, dp, dp]
        lib.oracle_corr_fft.restype = ctypes.c_int
        lib.oracle_corr2d_direct.argtypes = [dp, dp, L, L, L, L, L, ctypes.c_double, dp]
        lib.oracle_corr2d_direct.restype = None
        lib.oracle_circ2d_direct.argtypes = [dp, dp, L, L, L, L, L, dp]
        lib.oracle_circ2d_direct.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _LIB = lib
    return _LIB


def _f64(a):
    """Contiguous float64 numpy copy of a numpy array or a CPU torch tensor."""
    if hasattr(a, "detach"):  # torch tensor (any dtype, incl. bfloat16)
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Set the OpenMP threads later oracle calls use."""
    _lib().oracle_set_num_threads(int(n))


def scores(X, WA):
    """z[b, h, n] = sum_d X[b, n, d] W_A[d, h]."""
    X, WA = _f64(X), _f64(WA)
    B, N, D = X.shape
    H = WA.shape[1]
    assert WA.shape[0] == D
    z = np.empty((B, H, N), np.float64)
    _lib().oracle_scores(_p(X), _p(WA), B, N, D, H, _p(z))
    return z


def softmax(z):
    """Softmax over the last axis (the N tokens)."""
    z = _f64(z)
    N = z.shape[-1]
    out = np.empty_like(z)
    _lib().oracle_softmax(_p(z), _p(out), z.size // N if N else 0, N)
    return out


def project(X, W):
    """V = X · W per token (the value projection of a CAT layer), fp64:
    V[b, n, e] = sum_d X[b, n, d] W[d, e].  numpy's matmul is the step."""
    X, W = _f64(X), _f64(W)
    return X @ W


def zstar(X, WA):
    """z* = softmax_n(X · W_A), shape [B, H, N]."""
    return softmax(scores(X, WA))


def dft(x, inverse=False):
    """Complex DFT of a 1-D array (recursive radix-2 + naive odd-length DFT)."""
    x = np.asarray(x, dtype=np.complex128)
    re = np.ascontiguousarray(x.real, dtype=np.float64)
    im = np.ascontiguousarray(x.imag, dtype=np.float64)
    rc = _lib().oracle_dft(_p(re), _p(im), re.size, 1 if inverse else 0)
    if rc != 0:
        raise MemoryError("oracle_dft")
    return re + 1j * im


def spectrum(zs):
    """Zf[..., k] = sum_n z*[..., n] exp(-2πi kn/N) (complex128)."""
    zs = _f64(zs)
    N = zs.shape[-1]
    out = np.empty(zs.shape + (2,), np.float64)
    rc = _lib().oracle_spectrum(_p(zs), zs.size // N, N, _p(out))
    if rc != 0:
        raise MemoryError("oracle_spectrum")
    return out[..., 0] + 1j * out[..., 1]


def circ_direct(zs, V):
    """O = circ(z*) V by the O(N^2) definition.  zs [B,H,N], V [B,N,D]."""
    zs, V = _f64(zs), _f64(V)
    B, N, D = V.shape
    H = zs.shape[1]
    O = np.empty((B, N, D), np.float64)
    _lib().oracle_circ_direct(_p(zs), _p(V), B, N, D, H, _p(O))
    return O


def circ_direct_rows(zs, V, rows):
    """The O(N^2) definition at the listed output rows only: [B, len(rows), D]."""
    zs, V = _f64(zs), _f64(V)
    B, N, D = V.shape
    H = zs.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).astype(np.int_))
    O = np.empty((B, rows.size, D), np.float64)
    _lib().oracle_circ_direct_rows(
        _p(zs), _p(V), B, N, D, H,
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), rows.size, _p(O))
    return O


def circ_fft(zs, V, return_max_imag=False):
    """O = IFFT(FFT(z*) ⊙ FFT(V_h)) per column, fp64."""
    zs, V = _f64(zs), _f64(V)
    B, N, D = V.shape
    H = zs.shape[1]
    O = np.empty((B, N, D), np.float64)
    mi = ctypes.c_double(0.0)
    rc = _lib().oracle_circ_fft(_p(zs), _p(V), B, N, D, H, _p(O),
                                ctypes.pointer(mi))
    if rc != 0:
        raise MemoryError("oracle_circ_fft")
    return (O, mi.value) if return_max_imag else O


def brute_circulant(zs_row):
    """The explicit N x N matrix circ(z*)[i, j] = z*[(i - j) mod N]."""
    z = np.asarray(zs_row, dtype=np.float64)
    N = z.size
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return z[(i - j) % N]


def forward(X, WA, V, mode="auto"):
    """Whole forward: returns (O [B,N,D], z* [B,H,N]) in fp64.

    mode: "direct" (O(N^2) definition), "fft" (convolution theorem), or
    "auto" (direct while B·N²·D stays under ~2e9 multiply-adds, else fft).
    """
    X, WA, V = _f64(X), _f64(WA), _f64(V)
    B, N, D = V.shape
    zs = zstar(X, WA)
    if mode == "auto":
        mode = "direct" if B * N * N * D <= 2e9 else "fft"
    if mode == "direct":
        return circ_direct(zs, V), zs
    if mode == "fft":
        return circ_fft(zs, V), zs
    raise ValueError(mode)


# --------------------------------------------------------------------------
# Backward pass
# --------------------------------------------------------------------------

def _rows_arg(rows):
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).astype(np.int_))
    return rows, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long))


def circ_transpose_direct(zs, G):
    """dV = circ(z*)^T G by the O(N^2) definition.  zs [B,H,N], G [B,N,D]."""
    zs, G = _f64(zs), _f64(G)
    B, N, D = G.shape
    H = zs.shape[1]
    dV = np.empty((B, N, D), np.float64)
    _lib().oracle_circ_transpose_direct(_p(zs), _p(G), B, N, D, H, _p(dV))
    return dV


def circ_transpose_direct_rows(zs, G, rows):
    """dV by the definition at the listed rows only: [B, len(rows), D]."""
    zs, G = _f64(zs), _f64(G)
    B, N, D = G.shape
    H = zs.shape[1]
    rows, rp = _rows_arg(rows)
    out = np.empty((B, rows.size, D), np.float64)
    _lib().oracle_circ_transpose_direct_rows(_p(zs), _p(G), B, N, D, H, rp, rows.size, _p(out))
    return out


def circ_transpose_fft(zs, G):
    """dV = IFFT(conj(FFT(z*)) ⊙ FFT(G[:, c])) per column, fp64."""
    zs, G = _f64(zs), _f64(G)
    B, N, D = G.shape
    H = zs.shape[1]
    dV = np.empty((B, N, D), np.float64)
    if _lib().oracle_circ_transpose_fft(_p(zs), _p(G), B, N, D, H, _p(dV)) != 0:
        raise MemoryError("oracle_circ_transpose_fft")
    return dV


def corr_direct_bins(G, V, H, bins):
    """dz*[b, h, k] = sum_{c in h} sum_i G[b,i,c] V[b,(i-k) mod N,c] by the
    definition, at the listed bins k: [B, H, len(bins)]."""
    G, V = _f64(G), _f64(V)
    B, N, D = G.shape
    bins, bp = _rows_arg(bins)
    out = np.empty((B, H, bins.size), np.float64)
    _lib().oracle_corr_direct_bins(_p(G), _p(V), B, N, D, H, bp, bins.size, _p(out))
    return out


def corr_direct(G, V, H):
    """dz* at every bin by the definition, O(B·N^2·D): [B, H, N]."""
    N = np.shape(G)[1]
    return corr_direct_bins(G, V, H, np.arange(N))


def corr_fft(G, V, H, return_max_imag=False):
    """dz* = Re IFFT(sum_{c in h} FFT(G[:, c]) ⊙ conj(FFT(V[:, c]))), fp64."""
    G, V = _f64(G), _f64(V)
    B, N, D = G.shape
    out = np.empty((B, H, N), np.float64)
    mi = ctypes.c_double(0.0)
    if _lib().oracle_corr_fft(_p(G), _p(V), B, N, D, H, _p(out), ctypes.pointer(mi)) != 0:
        raise MemoryError("oracle_corr_fft")
    return (out, mi.value) if return_max_imag else out


def softmax_backward(zs, dzs):
    """dz = z* ⊙ (dz* - sum_m z*[m] dz*[m]) over the last axis."""
    zs, dzs = _f64(zs), _f64(dzs)
    N = zs.shape[-1]
    out = np.empty_like(zs)
    _lib().oracle_softmax_backward(_p(zs), _p(dzs), zs.size // N if N else 0, N, _p(out))
    return out


def grad_wa(X, dz):
    """dW_A[d, h] = sum_b sum_n X[b, n, d] dz[b, h, n]: [D, H]."""
    X, dz = _f64(X), _f64(dz)
    B, N, D = X.shape
    H = dz.shape[1]
    out = np.empty((D, H), np.float64)
    _lib().oracle_grad_wa(_p(X), _p(dz), B, N, D, H, _p(out))
    return out


def grad_x(dz, WA):
    """dX[b, n, d] = sum_h dz[b, h, n] W_A[d, h]: [B, N, D]."""
    dz, WA = _f64(dz), _f64(WA)
    B, H, N = dz.shape
    D = WA.shape[0]
    out = np.empty((B, N, D), np.float64)
    _lib().oracle_grad_x(_p(dz), _p(WA), B, N, D, H, _p(out))
    return out


def backward(X, WA, V, G, mode="auto"):
    """Whole backward for the upstream gradient G = dL/dO, fp64.

    Returns a dict with dX [B,N,D], dWA [D,H], dV [B,N,D], and the
    intermediates zs (z*), dzs (dL/dz*) and dz (dL/dz), each [B,H,N].
    mode: "direct" (O(N^2) definitions), "fft" (convolution and correlation
    theorems), or "auto" (direct while B·N²·D stays under ~2e9, else fft).
    """
    X, WA, V, G = _f64(X), _f64(WA), _f64(V), _f64(G)
    B, N, D = V.shape
    H = WA.shape[1]
    zs = zstar(X, WA)
    if mode == "auto":
        mode = "direct" if B * N * N * D <= 2e9 else "fft"
    if mode == "direct":
        dV = circ_transpose_direct(zs, G)
        dzs = corr_direct(G, V, H)
    elif mode == "fft":
        dV = circ_transpose_fft(zs, G)
        dzs = corr_fft(G, V, H)
    else:
        raise ValueError(mode)
    dz = softmax_backward(zs, dzs)
    return dict(dX=grad_x(dz, WA), dWA=grad_wa(X, dz), dV=dV, zs=zs, dzs=dzs, dz=dz)


# --------------------------------------------------------------------------
# 2-D circulant attention (page "Vision Transformers are Circulant Attention
# Learners"): tokens on an h x w grid (n = y·w + x), attention map a BCCB
# matrix with generator σ(a), O = σ(a) ⊛ V (2-D circular convolution).
# Reading for a (the page gives none): the channel-averaged 2-D circular
# cross-correlation of Q and K, a[k] = (1/dh) Σ_c Σ_i Q[i, c] K[i ⊖ k, c].
# --------------------------------------------------------------------------

def corr2d_direct(Q, K, H, h, w, scale=None):
    """a[b, hd, k] = scale · Σ_{c in hd} Σ_i Q[b,i,c] K[b, i ⊖ k, c] by the
    definition (scale defaults to 1/dh): [B, H, h·w]."""
    Q, K = _f64(Q), _f64(K)
    B, N, D = Q.shape
    assert N == h * w
    if scale is None:
        scale = 1.0 / (D // H)
    a = np.empty((B, H, N), np.float64)
    _lib().oracle_corr2d_direct(_p(Q), _p(K), B, h, w, D, H, float(scale), _p(a))
    return a


def corr2d_fft(Q, K, H, h, w, scale=None):
    """The same by the correlation theorem with numpy's 2-D FFT:
    a = scale · Re IFFT2( Σ_c FFT2(Q_c) ⊙ conj(FFT2(K_c)) )."""
    Q, K = _f64(Q), _f64(K)
    B, N, D = Q.shape
    dh = D // H
    if scale is None:
        scale = 1.0 / dh
    q = Q.reshape(B, h, w, H, dh)
    k = K.reshape(B, h, w, H, dh)
    spec = (np.fft.fft2(q, axes=(1, 2)) * np.conj(np.fft.fft2(k, axes=(1, 2)))).sum(axis=4)
    a = np.real(np.fft.ifft2(spec, axes=(1, 2)))          # [B, h, w, H]
    return scale * np.ascontiguousarray(a.transpose(0, 3, 1, 2).reshape(B, H, N))


def circ2d_direct(g, V, h, w):
    """O = BCCB(g) V by the definition: O[b,i,c] = Σ_j g[b,head(c), i ⊖ j] V[b,j,c]."""
    g, V = _f64(g), _f64(V)
    B, N, D = V.shape
    H = g.shape[1]
    assert N == h * w
    O = np.empty((B, N, D), np.float64)
    _lib().oracle_circ2d_direct(_p(g), _p(V), B, h, w, D, H, _p(O))
    return O


def circ2d_fft(g, V, h, w):
    """The same by the 2-D convolution theorem (numpy's 2-D FFT)."""
    g, V = _f64(g), _f64(V)
    B, N, D = V.shape
    H = g.shape[1]
    dh = D // H
    gf = np.fft.fft2(g.reshape(B, H, h, w), axes=(2, 3))            # [B, H, h, w]
    vf = np.fft.fft2(V.reshape(B, h, w, H, dh), axes=(1, 2))        # [B, h, w, H, dh]
    o = np.real(np.fft.ifft2(vf * gf.transpose(0, 2, 3, 1)[..., None], axes=(1, 2)))
    return np.ascontiguousarray(o.reshape(B, N, D))


def bccb_matrix(g2d):
    """The explicit N x N BCCB matrix of a generator g2d [h, w]."""
    g2d = np.asarray(g2d, dtype=np.float64)
    h, w = g2d.shape
    n = np.arange(h * w)
    yi, xi = (n // w)[:, None], (n % w)[:, None]
    yj, xj = (n // w)[None, :], (n % w)[None, :]
    return g2d[(yi - yj) % h, (xi - xj) % w]


def forward2d(Q, K, V, H, h, w, mode="auto"):
    """2-D circulant attention: returns (O [B,N,D], a [B,H,N], σ(a) [B,H,N])."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, N, D = V.shape
    if mode == "auto":
        mode = "direct" if B * N * N * D <= 2e9 else "fft"
    if mode == "direct":
        a = corr2d_direct(Q, K, H, h, w)
        zs = softmax(a)
        return circ2d_direct(zs, V, h, w), a, zs
    if mode == "fft":
        a = corr2d_fft(Q, K, H, h, w)
        zs = softmax(a)
        return circ2d_fft(zs, V, h, w), a, zs
    raise ValueError(mode)


__all__ = ["scores", "softmax", "zstar", "dft", "spectrum", "circ_direct",
           "circ_direct_rows", "circ_fft", "brute_circulant", "forward",
           "num_threads", "circ_transpose_direct", "circ_transpose_direct_rows",
           "circ_transpose_fft", "corr_direct", "corr_direct_bins", "corr_fft",
           "softmax_backward", "grad_wa", "grad_x", "backward", "corr2d_direct",
           "corr2d_fft", "circ2d_direct", "circ2d_fft", "bccb_matrix", "forward2d"]
