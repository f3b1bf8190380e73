"""The oracle's pins must catch plausible mistakes (no GPU).

Each case copies the oracle's C source to a temporary directory, plants one
mistake by a textual substitution, builds it there, and runs the pin that is
meant to catch it against the mutant.  The committed oracle is never
modified.
"""
import os
import shutil
import subprocess

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "cat_oracle.c")

MUTANTS = {
    # circulant orientation flipped (correlation instead of convolution)
    "shift_direction": ("long s = i - j;", "long s = j - i;"),
    # inverse transform without the 1/N factor
    "missing_inverse_scale": ("re[n] = inverse ? out[n] / (double)N : out[n];",
                              "re[n] = out[n];"),
    # W_A read transposed
    "transposed_wa": ("acc += x[d] * WA[d * H + h];", "acc += x[d] * WA[h * D + d];"),
    # columns interleaved across heads instead of contiguous blocks
    "head_map": ("return c / (D / H);", "return c % H;"),
    # twiddle with the wrong sign in the radix-2 combine
    "twiddle_sign": ("double ang = -2.0 * M_PI * (double)k / (double)N;",
                     "double ang = 2.0 * M_PI * (double)k / (double)N;"),
    # Hadamard product with a conjugated spectrum
    "conjugated_product": ("double pr = fr[k] * vr[k] - fi[k] * vi[k];",
                           "double pr = fr[k] * vr[k] + fi[k] * vi[k];"),
    # softmax without the normalisation
    "no_normalise": ("out[n] /= s;", "out[n] /= 1.0;"),
}

# Mistakes in the backward pass, caught by the backward pins.
BACKWARD_MUTANTS = {
    # correlation lag reversed (a convolution of G with V instead)
    "corr_lag": ("long s = i - k;", "long s = k - i;"),
    # softmax Jacobian without its mean term
    "softmax_bw_no_mean": ("dz[r * N + n] = p[n] * (g[n] - s);", "dz[r * N + n] = p[n] * g[n];"),
    # spectrum product without the conjugate on V (convolution theorem instead)
    "corr_fft_no_conj": ("ar[k] += gr[k] * vr[k] + gi[k] * vi[k];\n"
                         "          ai[k] += gi[k] * vr[k] - gr[k] * vi[k];",
                         "ar[k] += gr[k] * vr[k] - gi[k] * vi[k];\n"
                         "          ai[k] += gi[k] * vr[k] + gr[k] * vi[k];"),
    # transposed circulant's spectrum not conjugated
    "transpose_fft_no_conj": ("double pr = fr[k] * gr[k] + fi[k] * gi[k];\n"
                              "        double pi = fr[k] * gi[k] - fi[k] * gr[k];",
                              "double pr = fr[k] * gr[k] - fi[k] * gi[k];\n"
                              "        double pi = fr[k] * gi[k] + fi[k] * gr[k];"),
    # dX contracted with W_A read transposed
    "grad_x_transposed_wa": ("acc += dz[(b * H + h) * N + n] * WA[d * H + h];",
                             "acc += dz[(b * H + h) * N + n] * WA[h * D + d];"),
    # dW_A summed against the wrong token of dz
    "grad_wa_token": ("acc += X[(b * N + n) * D + d] * dz[(b * H + h) * N + n];",
                      "acc += X[(b * N + n) * D + d] * dz[(b * H + h) * N + (N - 1 - n)];"),
}

# Mistakes in the 2-D circulant attention, caught by the 2-D pins.
TWOD_MUTANTS = {
    # x offsets wrapped with the wrong period
    "wrap_period": ("if (x < 0) x += w;", "if (x < 0) x += h;"),
    # grid difference reversed along x only
    "x_direction": ("long y = yi - yk, x = xi - xk;", "long y = yi - yk, x = xk - xi;"),
    # correlation lag reversed (K[i ⊕ k] instead of K[i ⊖ k])
    "corr2d_lag": ("K[(b * N + grid_sub(i, k, h, w)) * D + c]",
                   "K[(b * N + grid_sub(k, i, h, w)) * D + c]"),
    # BCCB generator read transposed
    "bccb_transposed": ("acc += gr[grid_sub(i, j, h, w)] * V[(b * N + j) * D + c];",
                        "acc += gr[grid_sub(j, i, h, w)] * V[(b * N + j) * D + c];"),
}


def _build_mutant(tmp_path, name):
    table = {**MUTANTS, **BACKWARD_MUTANTS, **TWOD_MUTANTS}
    old, new = table[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    d = tmp_path / name
    d.mkdir()
    (d / "cat_oracle.c").write_text(src.replace(old, new))
    lib = d / "liboracle.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                    str(d / "cat_oracle.c"), "-o", str(lib), "-lm"], check=True)
    return str(lib)


def _with_lib(path):
    """Point the oracle module at another build of the same source."""
    saved = oracle._LIB
    oracle._LIB = None
    real_build = oracle._build.build
    oracle._build.build = lambda force=False: path
    try:
        oracle._lib()
    finally:
        oracle._build.build = real_build
    return saved


def _pins_fail():
    """Run the cheap pins; return True if any of them fails."""
    import test_oracle_pins as P
    checks = [
        P.test_worked_example_n4,
        lambda: P.test_dft_matches_library_fft(196),
        lambda: P.test_dft_matches_library_fft(64),
        P.test_scores_match_library_matmul,
        lambda: P.test_one_hot_is_cyclic_shift("direct"),
        lambda: P.test_one_hot_is_cyclic_shift("fft"),
        lambda: P.test_uniform_gives_column_mean("fft"),
        P.test_softmax_axis_is_tokens,
        lambda: P.test_brute_force_small_n(5),
        lambda: P.test_brute_force_small_n(12),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed > 0


def _backward_pins_fail():
    import test_oracle_backward_pins as P
    checks = [
        lambda: P.test_gradients_match_finite_differences(1, 5, 6, 3, "direct"),
        lambda: P.test_gradients_match_finite_differences(1, 5, 6, 3, "fft"),
        lambda: P.test_dzstar_matches_finite_differences(5),
        lambda: P.test_softmax_backward_matches_finite_differences(3),
        lambda: P.test_transpose_brute_force(8),
        lambda: P.test_correlation_by_roll(6),
        P.test_dense_contractions_match_library_matmul,
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed > 0


def _twod_pins_fail():
    import test_oracle_2d_pins as P
    checks = [
        lambda: P.test_one_row_grid_is_1d_cat(1, 9),
        lambda: P.test_bccb_matrix_brute_force(3, 4),
        lambda: P.test_scores_are_diagonal_sums_of_qkt(3, 5),
        lambda: P.test_one_hot_generator_is_2d_shift(1, 2),
        P.test_separable_generator,
        lambda: P.test_direct_equals_fft(7, 12),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed > 0


@pytest.mark.parametrize("name", sorted(TWOD_MUTANTS))
def test_twod_pins_catch_mutant(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = _build_mutant(tmp_path, name)
    saved = _with_lib(lib)
    try:
        assert _twod_pins_fail(), "mutant %s passed every 2-D pin" % name
    finally:
        oracle._LIB = saved


@pytest.mark.parametrize("name", sorted(BACKWARD_MUTANTS))
def test_backward_pins_catch_mutant(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = _build_mutant(tmp_path, name)
    saved = _with_lib(lib)
    try:
        assert _backward_pins_fail(), "mutant %s passed every backward pin" % name
    finally:
        oracle._LIB = saved


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = _build_mutant(tmp_path, name)
    saved = _with_lib(lib)
    try:
        assert _pins_fail(), "mutant %s passed every pin" % name
    finally:
        oracle._LIB = saved


def test_unmutated_copy_passes_pins(tmp_path):
    """Control: the same harness with the real source passes."""
    d = tmp_path / "clean"
    d.mkdir()
    shutil.copy(SRC, d / "cat_oracle.c")
    lib = d / "liboracle.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                    str(d / "cat_oracle.c"), "-o", str(lib), "-lm"], check=True)
    saved = _with_lib(str(lib))
    try:
        assert not _pins_fail()
        assert not _backward_pins_fail()
        assert not _twod_pins_fail()
    finally:
        oracle._LIB = saved
