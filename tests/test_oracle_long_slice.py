"""The fp64 FFT oracle against the plain definition at the full 131072-token
workload (B=1, N=2^17, D=1024, H=16, bf16 storage, seed 0).

The "FFT acceleration" design of the CAT notes page (section 关键设计) calls
IFFT(FFT(z*) ⊙ FFT(v)) exactly equal to the circulant product circ(z*)·v.
At N = 131072 the O(N^2) product cannot be evaluated at every row, so it is
evaluated on a slice of 4096 output rows, i = 32·r for r < 4096, and the FFT
oracle must agree with it there to fp64 rounding (1e-12·max|V|, the bound of
the shorter convolution-theorem pins).  The GPU parity test of this workload
compares its output at the same rows with the same definition.

Every column (all 16 heads) is checked on a host with at least 16 cores.
On fewer cores the check takes heads 0 and 15 only (128 of the 1024 value
columns: the first and the last head, whose W_A columns and value columns sit
at both ends of the arrays), so that the CPU suite stays within minutes.
"""
import os

import numpy as np

import oracle
import synth

N_ROWS, ROW_STEP = 4096, 32


def _heads_checked(H):
    return list(range(H)) if (os.cpu_count() or 1) >= 16 else [0, H - 1]


def test_fft_oracle_matches_definition_on_4096_row_slice_at_2e17():
    c = synth.CONFIGS["long128k"]
    B, N, D, H = c["B"], c["N"], c["D"], c["H"]
    assert N == N_ROWS * ROW_STEP
    X, WA, V = synth.make_inputs(B, N, D, H, c["dtype"], seed=0)
    zs = oracle.zstar(X, WA)                         # [1, 16, N], all heads from the full rows
    dh = D // H
    heads = _heads_checked(H)
    cols = np.concatenate([np.arange(h * dh, (h + 1) * dh) for h in heads])
    Vs = np.ascontiguousarray(V.double().numpy()[:, :, cols])
    zss = np.ascontiguousarray(zs[:, heads])
    rows = list(range(0, N, ROW_STEP))
    O_fft, max_imag = oracle.circ_fft(zss, Vs, return_max_imag=True)
    O_def = oracle.circ_direct_rows(zss, Vs, rows)
    vmax = float(np.abs(V.double().numpy()).max())
    err = float(np.abs(O_fft[:, rows] - O_def).max())
    print("N=%d: heads %s, %d rows x %d columns: max|FFT - definition| = %.3e "
          "(bound %.3e), max|Im| = %.3e" % (N, heads, len(rows), cols.size, err,
                                            1e-12 * vmax, max_imag))
    assert err <= 1e-12 * vmax
    assert max_imag <= 1e-12 * vmax
    # The slice is not trivially small: the outputs are O(1/sqrt(N_eff)).
    assert np.abs(O_def).max() > 1e-3
