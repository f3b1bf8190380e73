// 2-D circulant attention on square token grids of side M = 32·R (R = 2, 3,
// 4: sides 64, 96 and 128), after the page "Vision Transformers are
// Circulant Attention Learners" (section "Circulant Attention：用FFT重构注意力"):
// tokens on an M x M grid (token n = y·M + x), O = σ(a) ⊛ V, the 2-D
// circular convolution with the softmax of
//     a[b, h, k] = (1/dh) Σ_{c in head h} Σ_i Q[b, i, c] · K[b, i ⊖ k, c],
// the channel-averaged 2-D circular cross-correlation (the reading taken for
// the page's unprinted score formula).
//
// A 2-D DFT is separable: length-M DFTs along x over every grid row, then
// along y over every column.  A grid of 96 x 96 has too few (b, h) rows and
// too long a side for a register transform per column, so the work runs as
// five passes, each over many independent grid rows or columns, with the
// intermediate spectra in a scratch that stays in L2:
//   1. rows:    x-DFT of every channel-pair signal of Q, K (and V);
//   2. columns: y-DFT of Q and K, the pair sum of Q̂·conj(K̂) (a fixed
//               order), the inverse y-DFT of that sum;
//   3. rows:    inverse x-DFT, giving a; per grid row the max and the sum of
//               exp(a − max); the x-DFT of exp(a − row max);
//   4. columns: the softmax's scale for every grid row (max and sum over the
//               rows), the y-DFT of the column of σ, divided by N; the y-DFT
//               of V's columns, the product with it, the inverse y-DFT;
//   5. rows:    inverse x-DFT of V's rows, stored as O.
// Pairs of channels (2g, 2g + 1) travel as one complex signal; for the
// correlation Re(IDFT(X̂·conj(Ŷ))) of two such signals is the sum of the two
// channels' real correlations.
//
// Inside a CTA, a length-M DFT (M = P·Q: 64 = 8·8, 96 = 12·8, 128 = 16·8)
// of S signals is two stages: a register DFT-P over each stride-Q
// subsequence, times w_M^{e1·k2}, then a DFT-Q over adjacent slots, with the
// signals in shared memory (stride M + 1, odd, so that column accesses hit
// distinct banks) between them.  The first stage of a pass reads its input
// straight from global memory and the last writes its output there, a
// warp's lanes on consecutive channel pairs.  With n = e1 + Q·e2 and
// k = k2 + P·k1,
//     X[k2 + P·k1] = Σ_e1 w_Q^{e1·k1} · w_M^{e1·k2} · Σ_e2 w_P^{e2·k2} x[e1 + Q·e2],
// so the spectrum lands in the slot order k ↦ k1 + Q·k2.  The inverse runs
// the stages in reverse, from that order back to natural order.  Spectra
// are only ever multiplied with spectra of the same order, or inverted.
#include <cuda_bf16.h>

#include <cmath>

#include "../../include/cat.h"
#include "cat_internal.h"
#include "elem.cuh"
#include "fft_device.cuh"
#include "fft_reg.cuh"

namespace cat {

constexpr int kGpMaxThreads = 512;
constexpr int kGpRowsPerCta = 8;          // pass 3: one warp per grid row

// i / d for 0 <= i with i + d < 2^22, given r = 1.0f / d: the quotient's
// fractional part stays at least 0.5/d away from an integer, farther than
// the error of the float product, so the truncation is exact.
__device__ __forceinline__ int fdiv(int i, float r) { return (int)(((float)i + 0.5f) * r); }

// Elements i = 0 .. count-1 moved by the CTA's threads from ld(i) to st(i, ·),
// U loads in flight a thread before the first store (a loop that stored each
// value before the next load would wait a full memory latency per element).
template <int U, class V, class Ld, class St>
__device__ __forceinline__ void batched(int count, Ld ld, St st) {
  for (int i0 = threadIdx.x; i0 < count; i0 += U * blockDim.x) {
    V v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < count) v[u] = ld(i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < count) st(i, v[u]);
    }
  }
}

// The split of a grid side M = 32·R into the two stages of its DFT,
// M = P·Q: a register DFT of length P over stride-Q subsequences, then a
// DFT of length Q over adjacent slots.  Short register transforms (12 or
// 16 points, not 32) keep a thread's registers near 60, so that more warps
// fit an SM.
template <int R> struct Split;
template <> struct Split<2> { static constexpr int P = 8, Q = 8; };
template <> struct Split<3> { static constexpr int P = 12, Q = 8; };
template <> struct Split<4> { static constexpr int P = 16, Q = 8; };

// The two stages of a length-M DFT of S signals.  Element n of signal sig
// comes from ld(sig, n) and goes to st(sig, n, value), so a stage reads from
// or writes to global memory or shared memory as the pass needs.  Tasks run
// signal-fastest, so that the lanes of a warp touch consecutive signals:
// consecutive channel pairs in global memory, rows M + 1 apart (an odd
// stride: distinct banks) in shared memory.  twm: w_M^m, m < M.
//
// Stage A, forward: task (sig, e1), e1 < Q, transforms x[e1 + Q·e2] over
// e2 < P (a register DFT-P) and writes slot e1 + Q·k2 times w_M^{e1·k2}.
template <int R, class Ld, class St>
__device__ __forceinline__ void stage_a_fwd(int S, const float2* __restrict__ twm, Ld ld, St st) {
  constexpr int P = Split<R>::P, Q = Split<R>::Q;
  const float rS = 1.0f / (float)S;
  for (int t = threadIdx.x; t < S * Q; t += blockDim.x) {
    const int e1 = fdiv(t, rS), sig = t - e1 * S;
    float2 a[P];
#pragma unroll
    for (int e2 = 0; e2 < P; ++e2) a[e2] = ld(sig, e1 + Q * e2);
    dft<P, false>(a);
#pragma unroll
    for (int k2 = 0; k2 < P; ++k2) st(sig, e1 + Q * k2, cmul(a[k2], __ldg(&twm[e1 * k2])));
  }
}
// Stage A, inverse: slot e1 + Q·k2 times conj w_M^{e1·k2}, the inverse
// DFT-P over k2, written to element e1 + Q·e2.
template <int R, class Ld, class St>
__device__ __forceinline__ void stage_a_inv(int S, const float2* __restrict__ twm, Ld ld, St st) {
  constexpr int P = Split<R>::P, Q = Split<R>::Q;
  const float rS = 1.0f / (float)S;
  for (int t = threadIdx.x; t < S * Q; t += blockDim.x) {
    const int e1 = fdiv(t, rS), sig = t - e1 * S;
    float2 a[P];
#pragma unroll
    for (int k2 = 0; k2 < P; ++k2) a[k2] = cmulc(ld(sig, e1 + Q * k2), __ldg(&twm[e1 * k2]));
    dft<P, true>(a);
#pragma unroll
    for (int e2 = 0; e2 < P; ++e2) st(sig, e1 + Q * e2, a[e2]);
  }
}
// Stage B: task (sig, k2), k2 < P, applies the DFT-Q (inverse: its
// conjugate) to the Q adjacent slots Q·k2 .. Q·k2 + Q - 1.
template <int R, bool INV, class Ld, class St>
__device__ __forceinline__ void stage_b(int S, Ld ld, St st) {
  constexpr int P = Split<R>::P, Q = Split<R>::Q;
  const float rS = 1.0f / (float)S;
  for (int t = threadIdx.x; t < S * P; t += blockDim.x) {
    const int k2 = fdiv(t, rS), sig = t - k2 * S;
    float2 a[Q];
#pragma unroll
    for (int j = 0; j < Q; ++j) a[j] = ld(sig, Q * k2 + j);
    dft_small<Q, INV>(a);
#pragma unroll
    for (int j = 0; j < Q; ++j) st(sig, Q * k2 + j, a[j]);
  }
}

// Shared-memory signals: signal sig at buf + sig·(M + 1).
template <int R>
struct Smem {
  static constexpr int LS = 32 * R + 1;
  float2* buf;
  __device__ __forceinline__ float2 operator()(int sig, int e) const { return buf[sig * LS + e]; }
  __device__ __forceinline__ void operator()(int sig, int e, float2 v) const {
    buf[sig * LS + e] = v;
  }
};

// Channels (c, c + 1) of a row as one complex value; c + 1 past the head
// width reads as 0.  `aligned`: c even in an even-width row (pair access).
template <typename T>
__device__ __forceinline__ float2 ld_chan_pair(const T* p, bool pair, bool aligned) {
  if (pair && aligned) return ld_pair(p);
  return make_float2(ld_elem(p), pair ? ld_elem(p + 1) : 0.f);
}
template <typename T>
__device__ __forceinline__ void st_chan_pair(T* p, float2 v, bool pair, bool aligned) {
  if (pair && aligned) {
    st_pair(p, v);
  } else {
    st_elem(p, v.x);
    if (pair) st_elem(p + 1, v.y);
  }
}

// Pass 1: grid row y of (b, h) = bh0 + blockIdx.y, tensor blockIdx.z (Q, K,
// V): the x-DFT of its npair signals into xs[z][bhl][y][slot][g]; stage A
// reads the row's channel pairs, stage B writes the scratch.
template <typename T, int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_rows_fwd(const T* __restrict__ X0, const T* __restrict__ X1, const T* __restrict__ X2,
            float2* __restrict__ xs, size_t tstride, const float2* __restrict__ twm, int D,
            int H, int dh, int np, int bh0) {
  pdl_trigger();   // the next pass may launch; it waits for this one
  constexpr int M = 32 * R;
  extern __shared__ float4 smem4[];
  const Smem<R> sm{reinterpret_cast<float2*>(smem4)};
  const int y = blockIdx.x, bhl = blockIdx.y, z = blockIdx.z;
  const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
  const T* X = z == 0 ? X0 : (z == 1 ? X1 : X2);
  const bool aligned = ((h * dh) % 2) == 0 && (D % 2) == 0;
  const T* row = X + ((size_t)b * M * M + (size_t)y * M) * D + (size_t)h * dh;
  // Whole pairs at even offsets (the common case) load without a branch, so
  // that all of a task's loads issue before its transform.
  if (aligned && (dh % 2) == 0)
    stage_a_fwd<R>(np, twm, [&](int g, int x) { return ld_pair(row + (size_t)x * D + 2 * g); },
                   sm);
  else
    stage_a_fwd<R>(
        np, twm,
        [&](int g, int x) {
          return ld_chan_pair(row + (size_t)x * D + 2 * g, 2 * g + 1 < dh, aligned);
        },
        sm);
  __syncthreads();
  float2* dst = xs + z * tstride + ((size_t)bhl * M + y) * M * np;
  stage_b<R, false>(np, sm, [&](int g, int s, float2 v) { dst[(size_t)s * np + g] = v; });
}

// Pass 2: column slot kx = blockIdx.x of (b, h) row bhl = blockIdx.y: the
// y-DFT of Q's and K's npair signals (stage A reads the scratch column),
// Σ_g Q̂_g·conj(K̂_g) in the order g = 0, 1, …, and its inverse y-DFT into
// tsc[bhl][y][kx].
template <int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_cols_scores(const float2* qs, const float2* ks,
               float2* __restrict__ tsc, const float2* __restrict__ twm, int np) {
  pdl_trigger();
  pdl_wait();      // launched as the previous pass's programmatic dependent
  constexpr int M = 32 * R, LS = M + 1;
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);   // Q's signals, then K's
  const Smem<R> sm{buf};
  const Smem<R> sum{buf + 2 * np * LS};
  const int kx = blockIdx.x, bhl = blockIdx.y;
  const size_t base = (size_t)bhl * M * M * np + (size_t)kx * np;
  stage_a_fwd<R>(
      2 * np, twm,
      [&](int sig, int y) {
        const int q = sig >= np;
        return (q ? ks : qs)[base + (size_t)y * M * np + (sig - q * np)];
      },
      sm);
  __syncthreads();
  stage_b<R, false>(2 * np, sm, sm);
  __syncthreads();
  for (int s = threadIdx.x; s < M; s += blockDim.x) {
    float2 acc = make_float2(0.f, 0.f);
    for (int g = 0; g < np; ++g) {
      const float2 q = buf[g * LS + s], k = buf[(np + g) * LS + s];
      acc.x = fmaf(q.x, k.x, fmaf(q.y, k.y, acc.x));
      acc.y = fmaf(q.y, k.x, fmaf(-q.x, k.y, acc.y));
    }
    sum(0, s, acc);
  }
  __syncthreads();
  stage_b<R, true>(1, sum, sum);
  __syncthreads();
  float2* dst = tsc + (size_t)bhl * M * M + kx;
  stage_a_inv<R>(1, twm, sum, [&](int, int yy, float2 v) { dst[(size_t)yy * M] = v; });
}

// Pass 3: grid rows y0 .. y0 + 7 (one warp each) of (b, h) row bhl: the
// inverse x-DFT gives a (× scale = 1/(dh·N)), written to aout[bh][y·M + x]
// when given; with esp, the row's max m and sum s of exp(a − m) go to
// stats[bhl][y] and the x-DFT of exp(a − m) to esp[bhl][y][slot].
template <int R>
__global__ void __launch_bounds__(32 * kGpRowsPerCta)
gp_rows_scores(const float2* tsc, float2* __restrict__ esp,
               float2* __restrict__ stats, float* __restrict__ aout,
               const float2* __restrict__ twm, int bh0, float scale) {
  pdl_trigger();
  pdl_wait();      // launched as the previous pass's programmatic dependent
  constexpr int M = 32 * R, LS = M + 1, RB = kGpRowsPerCta;
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  const Smem<R> sm{buf};
  const int bhl = blockIdx.y, bh = bh0 + bhl, y0 = blockIdx.x * RB;
  const float2* src = tsc + ((size_t)bhl * M + y0) * M;
  stage_b<R, true>(RB, [&](int r, int s) { return src[r * M + s]; }, sm);
  __syncthreads();
  stage_a_inv<R>(RB, twm, sm, sm);
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, y = y0 + w;
  float v[R];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    v[j] = buf[w * LS + lane + 32 * j].x * scale;
    m = fmaxf(m, v[j]);
  }
  if (aout) {
#pragma unroll
    for (int j = 0; j < R; ++j) aout[(size_t)bh * M * M + (size_t)y * M + lane + 32 * j] = v[j];
  }
  if (!esp) return;
  m = warp_max(m);
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const float e = expf(v[j] - m);
    s += e;
    buf[w * LS + lane + 32 * j] = make_float2(e, 0.f);
  }
  s = warp_sum(s);
  if (lane == 0) stats[(size_t)bhl * M + y] = make_float2(m, s);
  __syncthreads();
  stage_a_fwd<R>(RB, twm, sm, sm);
  __syncthreads();
  float2* dst = esp + ((size_t)bhl * M + y0) * M;
  stage_b<R, false>(RB, sm, [&](int r, int sl, float2 val) { dst[r * M + sl] = val; });
}

// Pass 4: column slot kx of (b, h) row bhl.  The softmax's scale of grid
// row y is c_y = exp(m_y − m) / Σ_y' s_y'·exp(m_y' − m), m = max_y m_y, the
// same in every CTA of the row; the column of σ's x-spectrum times c_y / N
// is y-transformed together with V's npair columns, V's spectra are
// multiplied by it and inverse y-transformed back into vs.
template <int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_cols_conv(float2* vs, const float2* esp,
             const float2* stats, const float2* __restrict__ twm, int np,
             float invN) {
  pdl_trigger();
  pdl_wait();      // launched as the previous pass's programmatic dependent
  constexpr int M = 32 * R, LS = M + 1;
  extern __shared__ float4 smem4[];
  float2* sbuf = reinterpret_cast<float2*>(smem4);   // σ's column, then V's npair columns
  const Smem<R> all{sbuf};
  const Smem<R> vb{sbuf + LS};
  float* cy = reinterpret_cast<float*>(sbuf + (np + 1) * LS);
  const int kx = blockIdx.x, bhl = blockIdx.y;
  // σ's column and (warp 0) the row statistics, fetched first.
  float2 ev[2], st[R];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int y = threadIdx.x + u * blockDim.x;
    if (y < M) ev[u] = esp[((size_t)bhl * M + y) * M + kx];
  }
  if (threadIdx.x < 32) {
#pragma unroll
    for (int j = 0; j < R; ++j) st[j] = stats[(size_t)bhl * M + threadIdx.x + 32 * j];
  }
  float2* col = vs + (size_t)bhl * M * M * np + (size_t)kx * np;
  auto gcol_ld = [&](int g, int y) { return col[(size_t)y * M * np + g]; };
  auto gcol_st = [&](int g, int y, float2 v) { col[(size_t)y * M * np + g] = v; };
  stage_a_fwd<R>(np, twm, gcol_ld, vb);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float mm = -INFINITY;
#pragma unroll
    for (int j = 0; j < R; ++j) mm = fmaxf(mm, st[j].x);
    mm = warp_max(mm);
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < R; ++j) ss += st[j].y * expf(st[j].x - mm);
    ss = warp_sum(ss);
    const float inv = invN / ss;
#pragma unroll
    for (int j = 0; j < R; ++j) cy[lane + 32 * j] = expf(st[j].x - mm) * inv;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int y = threadIdx.x + u * blockDim.x;
    if (y < M) sbuf[y] = cscale(ev[u], cy[y]);
  }
  __syncthreads();
  stage_a_fwd<R>(1, twm, all, all);
  __syncthreads();
  stage_b<R, false>(np + 1, all, all);
  __syncthreads();
  const float rM = 1.0f / (float)M;
  for (int i = threadIdx.x; i < M * np; i += blockDim.x) {
    const int g = fdiv(i, rM), s = i - g * M;
    vb(g, s, cmul(vb(g, s), sbuf[s]));
  }
  __syncthreads();
  stage_b<R, true>(np, vb, vb);
  __syncthreads();
  stage_a_inv<R>(np, twm, vb, gcol_st);
}

// Pass 5: grid row y of (b, h) row bhl: the inverse x-DFT of V's npair
// signals (stage B reads the scratch row), stored as O's channels
// (2g, 2g + 1) by stage A.
template <typename T, int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_rows_out(const float2* vs, T* __restrict__ O, const float2* __restrict__ twm,
            int D, int H, int dh, int np, int bh0) {
  pdl_trigger();
  pdl_wait();      // launched as the previous pass's programmatic dependent
  constexpr int M = 32 * R;
  extern __shared__ float4 smem4[];
  const Smem<R> sm{reinterpret_cast<float2*>(smem4)};
  const int y = blockIdx.x, bhl = blockIdx.y;
  const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
  const float2* src = vs + ((size_t)bhl * M + y) * M * np;
  stage_b<R, true>(np, [&](int g, int s) { return src[(size_t)s * np + g]; }, sm);
  __syncthreads();
  const bool aligned = ((h * dh) % 2) == 0 && (D % 2) == 0;
  T* row = O + ((size_t)b * M * M + (size_t)y * M) * D + (size_t)h * dh;
  if (aligned && (dh % 2) == 0)
    stage_a_inv<R>(np, twm, sm,
                   [&](int g, int x, float2 v) { st_pair(row + (size_t)x * D + 2 * g, v); });
  else
    stage_a_inv<R>(np, twm, sm, [&](int g, int x, float2 v) {
      st_chan_pair(row + (size_t)x * D + 2 * g, v, 2 * g + 1 < dh, aligned);
    });
}

// ---------------------------------------------------------------------------
// Host side.

namespace {

// Threads of a CTA whose stage A has `tasks` tasks: whole warps, 128 .. 512.
int gp_threads(int tasks) {
  int t = (tasks + 31) / 32 * 32;
  return t < 128 ? 128 : (t > kGpMaxThreads ? kGpMaxThreads : t);
}

size_t sig_bytes(int M, int nsig) { return (size_t)nsig * (M + 1) * sizeof(float2); }
size_t smem_rows(int M, int np) { return sig_bytes(M, np); }
size_t smem_cols_scores(int M, int np) { return sig_bytes(M, 2 * np + 1); }
size_t smem_rows_scores(int M) { return sig_bytes(M, kGpRowsPerCta); }
size_t smem_cols_conv(int M, int np) { return sig_bytes(M, np + 1) + (size_t)M * sizeof(float); }

// Complex values of scratch per (b, h) row: Q, K, V after pass 1 (M²·npair
// each), the correlation after pass 2 and σ's x-spectrum (M² each), and the
// per-row softmax statistics (M).
size_t per_bh(int M, int np) { return ((size_t)3 * np + 2) * M * M + M; }

constexpr size_t kGpScratchBudget = (size_t)64 << 20;

template <typename T, int R>
cudaError_t setup_r() {
  cudaError_t e = allow_max_smem(gp_rows_fwd<T, R>);
  if (e == cudaSuccess) e = allow_max_smem(gp_cols_scores<R>);
  if (e == cudaSuccess) e = allow_max_smem(gp_rows_scores<R>);
  if (e == cudaSuccess) e = allow_max_smem(gp_cols_conv<R>);
  if (e == cudaSuccess) e = allow_max_smem(gp_rows_out<T, R>);
  return e;
}

// Scratch layout: the M twiddles w_M^m, then per chunk of (b, h) rows the
// pass-1 spectra of Q, K, V, the correlation, σ's x-spectrum and the row
// statistics.
struct Bufs {
  float2* twm;     // [M]
  float2* xs;      // [3][chunk][M][M][np]
  size_t tstride;  // chunk·M²·np
  float2* tsc;     // [chunk][M][M]
  float2* esp;     // [chunk][M][M]
  float2* stats;   // [chunk][M]
};

Bufs bufs(const cat_plan_s* p) {
  const int M = p->gp.M, np = p->npair, c = p->gp.chunk;
  Bufs b;
  b.twm = p->scratch;
  b.xs = p->scratch + M;
  b.tstride = (size_t)c * M * M * np;
  b.tsc = b.xs + 3 * b.tstride;
  b.esp = b.tsc + (size_t)c * M * M;
  b.stats = b.esp + (size_t)c * M * M;
  return b;
}

// One chunk of (b, h) rows [bh0, bh0 + nb): passes 1-3 (scores into aout
// when given), and with V and O passes 4-5.
template <typename T, int R>
cudaError_t run_chunk(const cat_plan_s* p, const T* Q, const T* K, const T* V, T* O, float* aout,
                      int bh0, int nb) {
  constexpr int M = 32 * R;
  const int np = p->npair;
  const Bufs bf = bufs(p);
  cudaStream_t st = p->stream;
  const bool fwd = V != nullptr;
  const int ntens = fwd ? 3 : 2;
  gp_rows_fwd<T, R><<<dim3(M, nb, ntens), gp_threads(np * Split<R>::Q), smem_rows(M, np), st>>>(
      Q, K, V, bf.xs, bf.tstride, bf.twm, p->D, p->H, p->dh, np, bh0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // Passes 2-5 launch as programmatic dependents (each waits for the pass
  // ahead at its start), which hides the launch gaps.
  e = launch_dependent(gp_cols_scores<R>, dim3(M, nb), dim3(gp_threads(2 * np * Split<R>::Q)),
                       smem_cols_scores(M, np), st, (const float2*)bf.xs,
                       (const float2*)(bf.xs + bf.tstride), bf.tsc, (const float2*)bf.twm, np);
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / ((float)p->dh * (float)(M * M));
  e = launch_dependent(gp_rows_scores<R>, dim3(M / kGpRowsPerCta, nb), dim3(32 * kGpRowsPerCta),
                       smem_rows_scores(M), st, (const float2*)bf.tsc,
                       fwd ? bf.esp : (float2*)nullptr, bf.stats, aout, (const float2*)bf.twm,
                       bh0, scale);
  if (e != cudaSuccess || !fwd) return e;
  e = launch_dependent(gp_cols_conv<R>, dim3(M, nb), dim3(gp_threads(np * Split<R>::Q)),
                       smem_cols_conv(M, np), st, bf.xs + 2 * bf.tstride,
                       (const float2*)bf.esp, (const float2*)bf.stats, (const float2*)bf.twm, np,
                       1.0f / (float)(M * M));
  if (e != cudaSuccess) return e;
  return launch_dependent(gp_rows_out<T, R>, dim3(M, nb), dim3(gp_threads(np * Split<R>::Q)),
                          smem_rows(M, np), st, (const float2*)(bf.xs + 2 * bf.tstride), O,
                          (const float2*)bf.twm, p->D, p->H, p->dh, np, bh0);
}

template <typename T>
cudaError_t run_all(const cat_plan_s* p, const void* Q, const void* K, const void* V, void* O,
                    float* aout) {
  const int rows = p->B * p->H;
  for (int bh0 = 0; bh0 < rows; bh0 += p->gp.chunk) {
    const int nb = rows - bh0 < p->gp.chunk ? rows - bh0 : p->gp.chunk;
    const T* q = (const T*)Q;
    const T* k = (const T*)K;
    const T* v = (const T*)V;
    T* o = (T*)O;
    cudaError_t e;
    switch (p->gp.R) {
      case 2: e = run_chunk<T, 2>(p, q, k, v, o, aout, bh0, nb); break;
      case 3: e = run_chunk<T, 3>(p, q, k, v, o, aout, bh0, nb); break;
      case 4: e = run_chunk<T, 4>(p, q, k, v, o, aout, bh0, nb); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool grid_pass_supported(int h, int w, int dh) {
  if (h != w || (h != 64 && h != 96 && h != 128)) return false;
  const int np = (dh + 1) / 2;
  // Pass 2 holds Q's and K's columns of one slot in shared memory.
  return smem_cols_scores(h, np) <= (size_t)200 * 1024;
}

int configure_grid_pass(cat_plan_s* p) {
  const int M = p->grid_w, np = p->npair;
  GridPassCfg& g = p->gp;
  g.M = M;
  g.R = M / 32;
  const size_t one = per_bh(M, np) * sizeof(float2);
  const int rows = p->B * p->H;
  long long c = (long long)(kGpScratchBudget / one);
  if (c < 1) c = 1;
  if (c > rows) c = rows;
  g.chunk = rows > 0 ? (int)c : 1;
  g.scratch_bytes = (size_t)M * sizeof(float2) + (size_t)g.chunk * one;
  return CAT_OK;
}

// Kernel attributes, and the M twiddles w_M^m = exp(-2πi m/M) (evaluated in
// fp64, rounded once) at the start of the scratch.
cudaError_t setup_grid_pass(const cat_plan_s* p) {
  cudaError_t e = p->dtype == 1 ? setup_r<__nv_bfloat16, 2>() : setup_r<float, 2>();
  if (e == cudaSuccess) e = p->dtype == 1 ? setup_r<__nv_bfloat16, 3>() : setup_r<float, 3>();
  if (e == cudaSuccess) e = p->dtype == 1 ? setup_r<__nv_bfloat16, 4>() : setup_r<float, 4>();
  if (e != cudaSuccess) return e;
  const int M = p->gp.M;
  float2 host[128];
  const double two_pi = 6.283185307179586476925286766559;
  for (int m = 0; m < M; ++m) {
    const double a = -two_pi * (double)m / (double)M;
    host[m] = make_float2((float)std::cos(a), (float)std::sin(a));
  }
  return cudaMemcpy(p->scratch, host, (size_t)M * sizeof(float2), cudaMemcpyHostToDevice);
}

cudaError_t launch_grid_pass(const cat_plan_s* p, const void* Q, const void* K, const void* V,
                             void* O, float* aout) {
  if (p->B == 0) return cudaSuccess;
  return p->dtype == 1 ? run_all<__nv_bfloat16>(p, Q, K, V, O, aout)
                       : run_all<float>(p, Q, K, V, O, aout);
}

}  // namespace cat
