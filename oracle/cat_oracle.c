/*
 * fp64 CPU oracle for the CAT forward pass (circular-convolutional attention)
 * and its backward pass (gradients by the chain rule, further below).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library: it is a plain restatement of the definitions, written to be
 * checked by eye.
 *
 * Source of every formula: the notes page "CAT: Circular-Convolutional
 * Attention for Sub-Quadratic Transformers" (NeurIPS 2025, arXiv 2504.06704),
 * section 方法详解 (method), sub-sections 整体框架 (overall framework) and
 * 关键设计 (key designs: "circulant attention matrix construction" and
 * "FFT acceleration").  In that notation, per head h:
 *
 *     Z      = X · W_A[:, h]                 (one score per token)
 *     Z*     = softmax(Z) over the N tokens
 *     circ(Z*)[i, j] = Z*[(i - j) mod N]     (row i = i-th cyclic shift)
 *     O_h    = circ(Z*) · V_h  =  IFFT( FFT(Z*) ⊙ FFT(V_h) )
 *
 * Readings taken where the page is open (each listed in the design notes):
 *   - W_A is D x H (one column per head), as the parameter count (D+H)·D
 *     requires, although the page prints D x 1;
 *   - "row softmax" of the N x 1 score vector is a softmax over the N tokens;
 *   - the shift direction is the one the convolution theorem in the "FFT
 *     acceleration" design fixes: circ[i, j] = z*[(i - j) mod N];
 *   - head h owns the contiguous value columns [h·D/H, (h+1)·D/H);
 *   - no temperature, bias, mask or output projection.
 *
 * Layouts (all row-major, fp64):
 *   X, V, O : [B, N, D]      W_A : [D, H]      z, z* : [B, H, N]
 *
 * Parallelism: OpenMP over independent output elements only; every sum is a
 * plain left-to-right loop in the order the definition writes it.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* Z = X · W_A  (整体框架 / circulant attention matrix construction).
 * z[b, h, n] = sum_d X[b, n, d] * W_A[d, h]. */
void oracle_scores(const double *X, const double *WA, long B, long N, long D,
                   long H, double *z) {
  long b, n;
#pragma omp parallel for collapse(2) schedule(static)
  for (b = 0; b < B; ++b) {
    for (n = 0; n < N; ++n) {
      const double *x = X + (b * N + n) * D;
      for (long h = 0; h < H; ++h) {
        double acc = 0.0;
        for (long d = 0; d < D; ++d) acc += x[d] * WA[d * H + h];
        z[(b * H + h) * N + n] = acc;
      }
    }
  }
}

/* Z* = softmax(Z) over the N entries of each of `rows` rows
 * (circulant attention matrix construction): subtract the row maximum,
 * exponentiate, divide by the sum. */
void oracle_softmax(const double *z, double *zs, long rows, long N) {
  long r;
#pragma omp parallel for schedule(static)
  for (r = 0; r < rows; ++r) {
    const double *zr = z + r * N;
    double *out = zs + r * N;
    double m = zr[0];
    for (long n = 1; n < N; ++n)
      if (zr[n] > m) m = zr[n];
    double s = 0.0;
    for (long n = 0; n < N; ++n) {
      out[n] = exp(zr[n] - m);
      s += out[n];
    }
    for (long n = 0; n < N; ++n) out[n] /= s;
  }
}

/* Index of the head that owns value column c. */
static long head_of(long c, long D, long H) { return c / (D / H); }

/* O = circ(Z*) · V by the plain definition, O(B·N²·D):
 * O[b, i, c] = sum_j z*[b, h(c), (i - j) mod N] * V[b, j, c]. */
void oracle_circ_direct(const double *zs, const double *V, long B, long N,
                        long D, long H, double *O) {
  long b, i;
#pragma omp parallel for collapse(2) schedule(static)
  for (b = 0; b < B; ++b) {
    for (i = 0; i < N; ++i) {
      for (long c = 0; c < D; ++c) {
        const double *w = zs + (b * H + head_of(c, D, H)) * N;
        double acc = 0.0;
        for (long j = 0; j < N; ++j) {
          long s = i - j;
          if (s < 0) s += N;
          acc += w[s] * V[(b * N + j) * D + c];
        }
        O[(b * N + i) * D + c] = acc;
      }
    }
  }
}

/* The same definition evaluated only at the output rows listed in `rows`
 * (nrows of them, each in [0, N)) for every batch and column:
 * Orows[b, r, c] = sum_j z*[b, h(c), (rows[r] - j) mod N] * V[b, j, c].
 * Every output is the same sum as in oracle_circ_direct, started at 0 and
 * taken over j in ascending order, so the two agree bit for bit.  Only the
 * order in which different outputs advance differs: the loop over j runs
 * outside the loops over a block of listed rows and the columns, so each
 * row V[b, j, :] is read once per block instead of once per output. */
void oracle_circ_direct_rows(const double *zs, const double *V, long B, long N,
                             long D, long H, const long *rows, long nrows,
                             double *Orows) {
  const long RB = 32; /* listed rows per block */
  const long dh = D / H;
  const long nblk = (nrows + RB - 1) / RB;
  long b, blk;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (b = 0; b < B; ++b) {
    for (blk = 0; blk < nblk; ++blk) {
      const long r0 = blk * RB;
      const long r1 = r0 + RB < nrows ? r0 + RB : nrows;
      double *acc = Orows + (b * nrows + r0) * D;
      for (long q = 0; q < (r1 - r0) * D; ++q) acc[q] = 0.0;
      for (long j = 0; j < N; ++j) {
        const double *v = V + (b * N + j) * D;
        for (long r = r0; r < r1; ++r) {
          long s = rows[r] - j;
          if (s < 0) s += N;
          double *o = acc + (r - r0) * D;
          for (long h = 0; h < H; ++h) {
            const double w = zs[(b * H + h) * N + s];
            for (long c = h * dh; c < (h + 1) * dh; ++c) o[c] += w * v[c];
          }
        }
      }
    }
  }
}

/* Textbook discrete Fourier transform, forward sign exp(-2πi kn/N), no
 * scaling.  Even lengths: one recursive radix-2 decimation-in-time split
 *     X[k]       = E[k] + w^k O[k]
 *     X[k + N/2] = E[k] - w^k O[k],   w = exp(-2πi/N),
 * with E, O the transforms of the even- and odd-indexed samples.  Odd
 * lengths: the naive O(N²) sum.  Twiddles come straight from cos/sin of the
 * exact angle (reduced mod N first), never from a recurrence. */
static void dft_rec(const double *re, const double *im, long N, long stride,
                    double *ore, double *oim, double *work) {
  if (N == 1) {
    ore[0] = re[0];
    oim[0] = im[0];
    return;
  }
  if (N % 2 == 1) {
    for (long k = 0; k < N; ++k) {
      double ar = 0.0, ai = 0.0;
      for (long n = 0; n < N; ++n) {
        long kn = (k * n) % N;
        double ang = -2.0 * M_PI * (double)kn / (double)N;
        double c = cos(ang), s = sin(ang);
        double xr = re[n * stride], xi = im[n * stride];
        ar += xr * c - xi * s;
        ai += xr * s + xi * c;
      }
      ore[k] = ar;
      oim[k] = ai;
    }
    return;
  }
  long h = N / 2;
  /* E into ore[0..h), O into ore[h..N); work gives the recursion scratch. */
  dft_rec(re, im, h, 2 * stride, ore, oim, work);
  dft_rec(re + stride, im + stride, h, 2 * stride, ore + h, oim + h, work);
  for (long k = 0; k < h; ++k) {
    double ang = -2.0 * M_PI * (double)k / (double)N;
    double c = cos(ang), s = sin(ang);
    double er = ore[k], ei = oim[k];
    double orr = ore[h + k], oi = oim[h + k];
    double tr = orr * c - oi * s;
    double ti = orr * s + oi * c;
    work[k] = er + tr;
    work[N + k] = ei + ti;
    work[h + k] = er - tr;
    work[N + h + k] = ei - ti;
  }
  memcpy(ore, work, (size_t)N * sizeof(double));
  memcpy(oim, work + N, (size_t)N * sizeof(double));
}

/* In-place DFT of one length-N complex signal (re, im).  inverse != 0 uses
 * exp(+2πi kn/N) and divides by N.  Returns 0, or -1 if memory ran out. */
int oracle_dft(double *re, double *im, long N, int inverse) {
  if (N <= 0) return 0;
  double *in = (double *)malloc(sizeof(double) * 2 * (size_t)N);
  double *out = (double *)malloc(sizeof(double) * 2 * (size_t)N);
  double *work = (double *)malloc(sizeof(double) * 2 * (size_t)N);
  if (!in || !out || !work) {
    free(in);
    free(out);
    free(work);
    return -1;
  }
  /* Inverse via conjugation: IDFT(x) = conj(DFT(conj(x))) / N. */
  double sgn = inverse ? -1.0 : 1.0;
  for (long n = 0; n < N; ++n) {
    in[n] = re[n];
    in[N + n] = sgn * im[n];
  }
  dft_rec(in, in + N, N, 1, out, out + N, work);
  for (long n = 0; n < N; ++n) {
    re[n] = inverse ? out[n] / (double)N : out[n];
    im[n] = inverse ? -out[N + n] / (double)N : out[N + n];
  }
  free(in);
  free(out);
  free(work);
  return 0;
}

/* O = IFFT(FFT(Z*) ⊙ FFT(V_h)) column by column (FFT acceleration design).
 * Each value column is transformed on its own as a real signal.  max_imag
 * receives max |Im| of the inverse transforms, which is zero in exact
 * arithmetic because both factors are real.  Returns 0 or -1 (memory). */
int oracle_circ_fft(const double *zs, const double *V, long B, long N, long D,
                    long H, double *O, double *max_imag) {
  long rows = B * H;
  double *zf = (double *)malloc(sizeof(double) * 2 * (size_t)(rows * N));
  if (!zf) return -1;
  int fail = 0;
  long r;
#pragma omp parallel for schedule(dynamic, 1)
  for (r = 0; r < rows; ++r) {
    double *fr = zf + 2 * r * N, *fi = fr + N;
    for (long n = 0; n < N; ++n) {
      fr[n] = zs[r * N + n];
      fi[n] = 0.0;
    }
    if (oracle_dft(fr, fi, N, 0) != 0) fail = 1;
  }
  double mi = 0.0;
  long b, c;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(max : mi)
  for (b = 0; b < B; ++b) {
    for (c = 0; c < D; ++c) {
      double *vr = (double *)malloc(sizeof(double) * 2 * (size_t)N);
      if (!vr) {
        fail = 1;
        continue;
      }
      double *vi = vr + N;
      for (long n = 0; n < N; ++n) {
        vr[n] = V[(b * N + n) * D + c];
        vi[n] = 0.0;
      }
      if (oracle_dft(vr, vi, N, 0) != 0) fail = 1;
      const double *fr = zf + 2 * (b * H + head_of(c, D, H)) * N;
      const double *fi = fr + N;
      for (long k = 0; k < N; ++k) { /* Hadamard product */
        double pr = fr[k] * vr[k] - fi[k] * vi[k];
        double pi = fr[k] * vi[k] + fi[k] * vr[k];
        vr[k] = pr;
        vi[k] = pi;
      }
      if (oracle_dft(vr, vi, N, 1) != 0) fail = 1;
      for (long n = 0; n < N; ++n) {
        O[(b * N + n) * D + c] = vr[n];
        if (fabs(vi[n]) > mi) mi = fabs(vi[n]);
      }
      free(vr);
    }
  }
  free(zf);
  if (max_imag) *max_imag = mi;
  return fail ? -1 : 0;
}

/* Spectrum of the softmax row: Zf[r, k] = sum_n z*[r, n] exp(-2πi kn/N),
 * stored as interleaved (re, im) pairs, rows x N x 2. */
int oracle_spectrum(const double *zs, long rows, long N, double *zf) {
  int fail = 0;
  long r;
#pragma omp parallel for schedule(dynamic, 1)
  for (r = 0; r < rows; ++r) {
    double *t = (double *)malloc(sizeof(double) * 2 * (size_t)N);
    if (!t) {
      fail = 1;
      continue;
    }
    for (long n = 0; n < N; ++n) {
      t[n] = zs[r * N + n];
      t[N + n] = 0.0;
    }
    if (oracle_dft(t, t + N, N, 0) != 0) fail = 1;
    for (long k = 0; k < N; ++k) {
      zf[2 * (r * N + k)] = t[k];
      zf[2 * (r * N + k) + 1] = t[N + k];
    }
    free(t);
  }
  return fail ? -1 : 0;
}

/* ------------------------------------------------------------------------
 * Backward pass.  The page trains CAT layers with the usual losses and
 * optimisers (section 损失函数 / 训练策略, loss and training strategy) but
 * prints no gradient formulas; these follow from the forward definitions
 * above by the chain rule.  With G = dL/dO [B, N, D] the upstream gradient:
 *
 *   O[i, c] = sum_j z*[(i - j) mod N] V[j, c]           (forward, head h(c))
 *   dV[j, c]   = sum_i z*[(i - j) mod N] G[i, c]        = (circ(z*)^T G)[j, c]
 *   dz*[h, k]  = sum_{c in h} sum_i G[i, c] V[(i - k) mod N, c]
 *   dz[h, n]   = z*[n] (dz*[n] - sum_m z*[m] dz*[m])     (softmax Jacobian)
 *   dW_A[d, h] = sum_b sum_n X[b, n, d] dz[b, h, n]
 *   dX[b, n, d] = sum_h dz[b, h, n] W_A[d, h]
 *
 * (∂O[i, c]/∂z*[k] = V[(i - k) mod N, c], because z*[k] multiplies V[j, c]
 * exactly where (i - j) mod N = k.)
 * ------------------------------------------------------------------------ */

/* dV = circ(z*)^T · G by the definition, O(B·N²·D). */
void oracle_circ_transpose_direct(const double *zs, const double *G, long B,
                                  long N, long D, long H, double *dV) {
  long b, j;
#pragma omp parallel for collapse(2) schedule(static)
  for (b = 0; b < B; ++b) {
    for (j = 0; j < N; ++j) {
      for (long c = 0; c < D; ++c) {
        const double *w = zs + (b * H + head_of(c, D, H)) * N;
        double acc = 0.0;
        for (long i = 0; i < N; ++i) {
          long s = i - j;
          if (s < 0) s += N;
          acc += w[s] * G[(b * N + i) * D + c];
        }
        dV[(b * N + j) * D + c] = acc;
      }
    }
  }
}

/* The same at the listed rows j only: dVrows[b, r, c]. */
void oracle_circ_transpose_direct_rows(const double *zs, const double *G,
                                       long B, long N, long D, long H,
                                       const long *rows, long nrows,
                                       double *dVrows) {
  long b, r;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (b = 0; b < B; ++b) {
    for (r = 0; r < nrows; ++r) {
      long j = rows[r];
      for (long c = 0; c < D; ++c) {
        const double *w = zs + (b * H + head_of(c, D, H)) * N;
        double acc = 0.0;
        for (long i = 0; i < N; ++i) {
          long s = i - j;
          if (s < 0) s += N;
          acc += w[s] * G[(b * N + i) * D + c];
        }
        dVrows[(b * nrows + r) * D + c] = acc;
      }
    }
  }
}

/* dz*[b, h, k] = sum_{c in head h} sum_i G[b, i, c] V[b, (i - k) mod N, c]
 * by the definition, at the listed bins k only (nbins of them; pass every
 * k for the whole row): out[b, h, r] for k = bins[r]. */
void oracle_corr_direct_bins(const double *G, const double *V, long B, long N,
                             long D, long H, const long *bins, long nbins,
                             double *out) {
  const long dh = D / H;
  long b, h;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (b = 0; b < B; ++b) {
    for (h = 0; h < H; ++h) {
      for (long r = 0; r < nbins; ++r) {
        long k = bins[r];
        double acc = 0.0;
        for (long c = h * dh; c < (h + 1) * dh; ++c) {
          for (long i = 0; i < N; ++i) {
            long s = i - k;
            if (s < 0) s += N;
            acc += G[(b * N + i) * D + c] * V[(b * N + s) * D + c];
          }
        }
        out[(b * H + h) * nbins + r] = acc;
      }
    }
  }
}

/* Softmax backward over each of `rows` rows of length N:
 * dz[n] = z*[n] · (dz*[n] - sum_m z*[m] dz*[m]). */
void oracle_softmax_backward(const double *zs, const double *dzs, long rows,
                             long N, double *dz) {
  long r;
#pragma omp parallel for schedule(static)
  for (r = 0; r < rows; ++r) {
    const double *p = zs + r * N, *g = dzs + r * N;
    double s = 0.0;
    for (long m = 0; m < N; ++m) s += p[m] * g[m];
    for (long n = 0; n < N; ++n) dz[r * N + n] = p[n] * (g[n] - s);
  }
}

/* dW_A[d, h] = sum_b sum_n X[b, n, d] · dz[b, h, n]. */
void oracle_grad_wa(const double *X, const double *dz, long B, long N, long D,
                    long H, double *dWA) {
  long d;
#pragma omp parallel for schedule(static)
  for (d = 0; d < D; ++d) {
    for (long h = 0; h < H; ++h) {
      double acc = 0.0;
      for (long b = 0; b < B; ++b)
        for (long n = 0; n < N; ++n)
          acc += X[(b * N + n) * D + d] * dz[(b * H + h) * N + n];
      dWA[d * H + h] = acc;
    }
  }
}

/* dX[b, n, d] = sum_h dz[b, h, n] · W_A[d, h]. */
void oracle_grad_x(const double *dz, const double *WA, long B, long N, long D,
                   long H, double *dX) {
  long b, n;
#pragma omp parallel for collapse(2) schedule(static)
  for (b = 0; b < B; ++b) {
    for (n = 0; n < N; ++n) {
      for (long d = 0; d < D; ++d) {
        double acc = 0.0;
        for (long h = 0; h < H; ++h) acc += dz[(b * H + h) * N + n] * WA[d * H + h];
        dX[(b * N + n) * D + d] = acc;
      }
    }
  }
}

/* dV by the convolution theorem: circ(z*)^T has the spectrum conj(FFT(z*))
 * (z* is real), so dV[:, c] = IFFT(conj(FFT(z*)) ⊙ FFT(G[:, c])), each
 * column transformed on its own.  Returns 0 or -1 (memory). */
int oracle_circ_transpose_fft(const double *zs, const double *G, long B, long N,
                              long D, long H, double *dV) {
  long rows = B * H;
  double *zf = (double *)malloc(sizeof(double) * 2 * (size_t)(rows * N));
  if (!zf) return -1;
  int fail = 0;
  long r;
#pragma omp parallel for schedule(dynamic, 1)
  for (r = 0; r < rows; ++r) {
    double *fr = zf + 2 * r * N, *fi = fr + N;
    for (long n = 0; n < N; ++n) {
      fr[n] = zs[r * N + n];
      fi[n] = 0.0;
    }
    if (oracle_dft(fr, fi, N, 0) != 0) fail = 1;
  }
  long b, c;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (b = 0; b < B; ++b) {
    for (c = 0; c < D; ++c) {
      double *gr = (double *)malloc(sizeof(double) * 2 * (size_t)N);
      if (!gr) {
        fail = 1;
        continue;
      }
      double *gi = gr + N;
      for (long n = 0; n < N; ++n) {
        gr[n] = G[(b * N + n) * D + c];
        gi[n] = 0.0;
      }
      if (oracle_dft(gr, gi, N, 0) != 0) fail = 1;
      const double *fr = zf + 2 * (b * H + head_of(c, D, H)) * N;
      const double *fi = fr + N;
      for (long k = 0; k < N; ++k) { /* conj(Zf) ⊙ Gf */
        double pr = fr[k] * gr[k] + fi[k] * gi[k];
        double pi = fr[k] * gi[k] - fi[k] * gr[k];
        gr[k] = pr;
        gi[k] = pi;
      }
      if (oracle_dft(gr, gi, N, 1) != 0) fail = 1;
      for (long n = 0; n < N; ++n) dV[(b * N + n) * D + c] = gr[n];
      free(gr);
    }
  }
  free(zf);
  return fail ? -1 : 0;
}

/* dz* by the correlation theorem: per (b, h),
 * dz* = IFFT( sum_{c in h} FFT(G[:, c]) ⊙ conj(FFT(V[:, c])) ), real part.
 * max_imag receives max |Im| of the inverse transforms (zero in exact
 * arithmetic).  Returns 0 or -1 (memory). */
int oracle_corr_fft(const double *G, const double *V, long B, long N, long D,
                    long H, double *dzs, double *max_imag) {
  const long dh = D / H;
  int fail = 0;
  double mi = 0.0;
  long b, h;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(max : mi)
  for (b = 0; b < B; ++b) {
    for (h = 0; h < H; ++h) {
      double *buf = (double *)malloc(sizeof(double) * 6 * (size_t)N);
      if (!buf) {
        fail = 1;
        continue;
      }
      double *ar = buf, *ai = buf + N;          /* accumulated spectrum */
      double *gr = buf + 2 * N, *gi = buf + 3 * N;
      double *vr = buf + 4 * N, *vi = buf + 5 * N;
      for (long k = 0; k < N; ++k) ar[k] = ai[k] = 0.0;
      for (long c = h * dh; c < (h + 1) * dh; ++c) {
        for (long n = 0; n < N; ++n) {
          gr[n] = G[(b * N + n) * D + c];
          gi[n] = 0.0;
          vr[n] = V[(b * N + n) * D + c];
          vi[n] = 0.0;
        }
        if (oracle_dft(gr, gi, N, 0) != 0 || oracle_dft(vr, vi, N, 0) != 0) fail = 1;
        for (long k = 0; k < N; ++k) { /* Gf ⊙ conj(Vf) */
          ar[k] += gr[k] * vr[k] + gi[k] * vi[k];
          ai[k] += gi[k] * vr[k] - gr[k] * vi[k];
        }
      }
      if (oracle_dft(ar, ai, N, 1) != 0) fail = 1;
      for (long n = 0; n < N; ++n) {
        dzs[(b * H + h) * N + n] = ar[n];
        if (fabs(ai[n]) > mi) mi = fabs(ai[n]);
      }
      free(buf);
    }
  }
  if (max_imag) *max_imag = mi;
  return fail ? -1 : 0;
}

/* ------------------------------------------------------------------------
 * 2-D circulant attention (the page "Vision Transformers are Circulant
 * Attention Learners", sections on the BCCB structure and "Circulant
 * Attention: 用FFT重构注意力"): tokens on an h x w grid, token n = y·w + x.
 * The attention map is a BCCB matrix (block circulant with circulant
 * blocks) with generator g over the grid,
 *     M[i, j] = g[(y_i - y_j) mod h, (x_i - x_j) mod w],
 * so M·v is the 2-D circular convolution of g with v: O = σ(a) ⊛ V.
 * Reading (the page prints no formula for a): a is the channel-averaged
 * 2-D circular cross-correlation of Q and K, the sum along each wrapped
 * 2-D diagonal of Q·K^T,
 *     a[b, hd, k] = scale · Σ_{c in head hd} Σ_i Q[b, i, c] · K[b, i ⊖ k, c],
 * with i ⊖ k the grid-wise difference mod (h, w) and scale = 1/dh.
 * ------------------------------------------------------------------------ */

/* Grid index of (y_i - y_k) mod h, (x_i - x_k) mod w for token indices. */
static long grid_sub(long i, long k, long h, long w) {
  long yi = i / w, xi = i % w, yk = k / w, xk = k % w;
  long y = yi - yk, x = xi - xk;
  if (y < 0) y += h;
  if (x < 0) x += w;
  return y * w + x;
}

/* a = scale · Σ_{c in head} Σ_i Q[i, c] K[i ⊖ k, c], every lag k. */
void oracle_corr2d_direct(const double *Q, const double *K, long B, long h,
                          long w, long D, long H, double scale, double *a) {
  const long N = h * w, dh = D / H;
  long b, hd;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (b = 0; b < B; ++b) {
    for (hd = 0; hd < H; ++hd) {
      for (long k = 0; k < N; ++k) {
        double acc = 0.0;
        for (long c = hd * dh; c < (hd + 1) * dh; ++c)
          for (long i = 0; i < N; ++i)
            acc += Q[(b * N + i) * D + c] * K[(b * N + grid_sub(i, k, h, w)) * D + c];
        a[(b * H + hd) * N + k] = scale * acc;
      }
    }
  }
}

/* O = BCCB(g) · V: O[b, i, c] = Σ_j g[b, head(c), i ⊖ j] · V[b, j, c]. */
void oracle_circ2d_direct(const double *g, const double *V, long B, long h,
                          long w, long D, long H, double *O) {
  const long N = h * w;
  long b, i;
#pragma omp parallel for collapse(2) schedule(static)
  for (b = 0; b < B; ++b) {
    for (i = 0; i < N; ++i) {
      for (long c = 0; c < D; ++c) {
        const double *gr = g + (b * H + head_of(c, D, H)) * N;
        double acc = 0.0;
        for (long j = 0; j < N; ++j)
          acc += gr[grid_sub(i, j, h, w)] * V[(b * N + j) * D + c];
        O[(b * N + i) * D + c] = acc;
      }
    }
  }
}

/* Number of OpenMP threads the oracle will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Set the number of OpenMP threads later calls use (no effect without
 * OpenMP); n < 1 is taken as 1. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  omp_set_num_threads(n < 1 ? 1 : n);
#else
  (void)n;
#endif
}
