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


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
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
    finally:
        oracle._LIB = saved
