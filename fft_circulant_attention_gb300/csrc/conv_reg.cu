// Circulant product for square lengths N = M·M (M in {8, 14, 16, 32}, i.e.
// N = 64, 196, 256, 1024) with the whole transform in registers and one
// shared-memory exchange per direction — the "FFT acceleration" design of
// the notes page "CAT: Circular-Convolutional Attention for Sub-Quadratic
// Transformers" (section 关键设计):
//     O_h[:, c] = IFFT( FFT(z*_h) ⊙ FFT(V_h[:, c]) ),
// for value column pairs packed as complex signals (see conv_smem.cu).
//
// With n = n1 + M·n2 and k = k2 + M·k1:
//     FFT(v)[k2 + M k1] = sum_n1 w_M^{n1 k1} · w_N^{n1 k2} · sum_n2 w_M^{n2 k2} v[n1 + M n2].
// A CTA owns P pairs of one (b, h); thread (i, p) (p fastest) is pair p and
//   step 1: n1 = i — loads its M rows n1 + M·n2, DFT over n2, twiddle
//           w_N^{n1·k2}, stores [k2][n1][p];
//   step 2: k2 = i — DFT over n1 (bins k2 + M·k1), product with FFT(z*)/N,
//           inverse DFT over k1, conjugate twiddle, stores back in place;
//   step 3: n1 = i — inverse DFT over k2, stores the output rows.
// Every shared-memory access has the pair index fastest, so it is free of
// bank conflicts; the twiddles w_N^{n1·k2} and the (b, h) row of FFT(z*)/N
// sit in shared memory.
#include <cuda_bf16.h>

#include "cat_internal.h"
#include "elem.cuh"
#include "fft_reg.cuh"
#include "tc.cuh"

namespace cat {

// A column pair (c, c+1), or the lone last column of an odd head width
// (imaginary part zero).  Pairs at odd columns (odd head width, odd head)
// move element by element.
template <typename T>
__device__ __forceinline__ float2 ld_col_pair(const T* p, bool pair, bool aligned) {
  if (pair && aligned) return ld_pair(p);
  return make_float2(ld_elem(p), pair ? ld_elem(p + 1) : 0.f);
}

// The M rows r0 + step·n2 (n2 < M) of a column pair.  On the common path
// (whole pair, aligned) every load is issued before any value is widened,
// so all M are in flight at once.
template <typename T, int M>
__device__ __forceinline__ void ld_rows(float2* a, const T* base, size_t step, size_t r0,
                                        bool active, bool pair, bool aligned) {
  if (active && pair && aligned) {
    if constexpr (sizeof(T) == 2) {
      unsigned int raw[M];
#pragma unroll
      for (int n2 = 0; n2 < M; ++n2)
        raw[n2] = __ldg(reinterpret_cast<const unsigned int*>(base + r0 + step * n2));
#pragma unroll
      for (int n2 = 0; n2 < M; ++n2)
        a[n2] = make_float2(__uint_as_float(raw[n2] << 16), __uint_as_float(raw[n2] & 0xffff0000u));
    } else {
#pragma unroll
      for (int n2 = 0; n2 < M; ++n2) a[n2] = ld_pair(base + r0 + step * n2);
    }
  } else {
#pragma unroll
    for (int n2 = 0; n2 < M; ++n2)
      a[n2] = active ? ld_col_pair(base + r0 + step * n2, pair, aligned) : make_float2(0.f, 0.f);
  }
}

template <typename T>
__device__ __forceinline__ void st_col_pair(T* p, float2 v, bool pair, bool aligned) {
  if (pair && aligned) {
    st_pair(p, v);
  } else {
    st_elem(p, v.x);
    if (pair) st_elem(p + 1, v.y);
  }
}

// Shared layout of the product kernel: the [M][M][P] signal block with a
// row (first index) stride of M·P + 8 when P = 8 (a warp then spans four
// rows in step 2; rows M·P = 256 apart would share banks), and the twiddle
// table with a row stride of M + 1 for M = 32 (step 1 reads a column).
// (conv_reg_pairs gives P = 8 exactly when M = 32, so the product kernel
// takes both strides as compile-time constants there.)
__host__ __device__ inline int reg_rs(int M, int P) { return M * P + (P == 8 ? 8 : 0); }
__host__ __device__ constexpr int reg_tws(int M) { return M == 32 ? M + 1 : M; }

// TW = false: no twiddle between the two steps, i.e. the 2-D DFT of an
// M x M token grid (n1 = x, n2 = y): the 2-D circular convolution of the
// second page's circulant attention.
// Below M = 32 a CTA is M·16 threads (16 pairs) and three should share an
// SM (short transforms need few registers); at M = 32 it is the plain
// 512-thread bound (128 registers a thread).
#define CAT_REG_BOUNDS(M) __launch_bounds__((M) == 32 ? 512 : (M) * 16, (M) == 32 ? 0 : 3)

template <typename T, int M, bool TW = true>
__global__ void CAT_REG_BOUNDS(M)
conv_reg_kernel(const T* __restrict__ V, T* __restrict__ O, const float2* zf,
                const float2* __restrict__ W, int D, int H, int dh, int npair, int P,
                int groups, int conj) {
  constexpr int N = M * M, TWS = reg_tws(M);
  if (M == 32) P = 8;
  const int RS = reg_rs(M, P);
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);   // [M][M][P], rows RS apart
  float2* tw = buf + M * RS;                         // tw[n1·TWS + k2] = w_N^{n1·k2}
  float2* zs = tw + M * TWS;                         // FFT(z*)/N of this (b, h)
  const int bh = blockIdx.x / groups, grp = blockIdx.x - (blockIdx.x / groups) * groups;
  const int b = bh / H, h = bh - b * H;
  const int p = threadIdx.x % P, i = threadIdx.x / P;
  // Twiddles to shared memory, four loads in flight per thread (one round
  // trip for N = 32² with 256 threads).  The spectrum follows the first
  // transform: it is the kernel ahead's output (see pdl_wait).
  constexpr int kPro = 4;
  if (TW) {
    for (int e0 = threadIdx.x; e0 < N; e0 += kPro * blockDim.x) {
      float2 tv[kPro];
#pragma unroll
      for (int u = 0; u < kPro; ++u) {
        const int e = e0 + u * blockDim.x;
        if (e < N) tv[u] = __ldg(&W[(e / M) * (e % M)]);
      }
#pragma unroll
      for (int u = 0; u < kPro; ++u) {
        const int e = e0 + u * blockDim.x;
        if (e < N) tw[(e / M) * TWS + e % M] = tv[u];
      }
    }
  }

  const int g = grp * P + p;
  const bool active = g < npair;
  const bool pair = 2 * g + 1 < dh;
  const int col = h * dh + 2 * (active ? g : 0);
  // Pair accesses need the pair's first element at an even offset in every
  // row: an even column and an even row length.
  const bool aligned = (col & 1) == 0 && (D & 1) == 0;
  const size_t base = (size_t)b * N * D + col;

  float2 a[M];
  ld_rows<T, M>(a, V + base, (size_t)M * D, (size_t)i * D, active, pair, aligned);
  dft<M, false, CxPaired>(a);
  // V's loads and first transform may overlap the spectrum kernel ahead
  // (launched as its programmatic dependent); its output is read only now.
  pdl_wait();
  for (int e0 = threadIdx.x; e0 < N; e0 += kPro * blockDim.x) {
    float2 zv[kPro];
#pragma unroll
    for (int u = 0; u < kPro; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < N) zv[u] = ld_dep(&zf[(size_t)bh * N + e]);
    }
#pragma unroll
    for (int u = 0; u < kPro; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < N) zs[e] = conj ? make_float2(zv[u].x, -zv[u].y) : zv[u];
    }
  }
  __syncthreads();   // twiddles and spectrum ready
#pragma unroll
  for (int k2 = 0; k2 < M; ++k2) buf[k2 * RS + i * P + p] = TW ? cmul(a[k2], tw[i * TWS + k2]) : a[k2];
  __syncthreads();

  // Step 2: k2 = i.  Each thread reads and rewrites only its own M slots.
#pragma unroll
  for (int n1 = 0; n1 < M; ++n1) a[n1] = buf[i * RS + n1 * P + p];
  dft<M, false, CxPaired>(a);
#pragma unroll
  for (int k1 = 0; k1 < M; ++k1) a[k1] = cmul(a[k1], zs[i + M * k1]);
  dft<M, true, CxPaired>(a);
#pragma unroll
  for (int n1 = 0; n1 < M; ++n1) buf[i * RS + n1 * P + p] = TW ? cmulc(a[n1], tw[n1 * TWS + i]) : a[n1];
  __syncthreads();

  // Step 3: n1 = i.
#pragma unroll
  for (int k2 = 0; k2 < M; ++k2) a[k2] = buf[k2 * RS + i * P + p];
  dft<M, true, CxPaired>(a);
  if (active) {
#pragma unroll
    for (int n2 = 0; n2 < M; ++n2)
      st_col_pair(O + base + (size_t)(i + M * n2) * D, a[n2], pair, aligned);
  }
}

// Correlation of pair-packed column signals summed over a head, by the
// register transform of N = M·M (n = n1 + M·n2, k = k2 + M·k1), for two
// uses:
//  - TW = false, the 2-D scores of the second page's circulant attention
//    ("Vision Transformers are Circulant Attention Learners": a from Q and K
//    by FFTs and an element-wise product) on an M x M grid (n1 = x, n2 = y),
//    read as the channel-averaged 2-D circular cross-correlation
//        a[b, h, k] = (1/dh) Σ_{c in head h} Σ_i Q[b, i, c] · K[b, i ⊖ k, c];
//  - TW = true, the backward pass's dz*[b, h, k] = Σ_{c in h} Σ_i dO[b, i, c]
//    · V[b, (i - k) mod N, c] (the derivative of the CAT output with respect
//    to z*), a 1-D correlation of length N.
// Both are Re IFFT( Σ_pairs FFT(q) · conj(FFT(kk)) ) times `scale`, with
// q = A[:, c] + i·A[:, c+1] and kk likewise from B (the imaginary parts of
// the pair products transform to purely imaginary signals, so the real part
// of the inverse is the two columns' sum).  One CTA per (b, h): thread
// (i, p) transforms pair p of A and of B as the circulant product's first
// two steps do, the products are summed over the head's pairs in a fixed
// order, and M threads run the inverse of the sum.  Writes out (fp32) and,
// if z2 is given, (value, 0) into it.
template <typename T, int M, bool TW>
__global__ void CAT_REG_BOUNDS(M)
corr_reg_kernel(const T* __restrict__ Q, const T* __restrict__ K, float2* __restrict__ z2,
                float* __restrict__ out, const float2* __restrict__ W, int D, int H, int dh,
                int npair, int P, float scale, float2* __restrict__ part, int G) {
  constexpr int N = M * M, TWS = reg_tws(M);
  const int RS = reg_rs(M, P);
  extern __shared__ float4 smem4[];
  float2* bq = reinterpret_cast<float2*>(smem4);   // [M][M][P] Q pairs, then products (rows RS apart)
  float2* bk = bq + M * RS;                         // [M][M][P] K pairs
  float2* S = bk + M * RS;                          // [k2][k1] running sum
  float2* tw = S + N;                               // TW: tw[n1·TWS + k2] = w_N^{n1·k2}
  // With part (G > 1), CTA gi of the (b, h) row takes its share of the
  // pairs (whole groups of P) and leaves its partial sum S in part instead
  // of inverting it; a finishing kernel adds the G partials in order.
  const int bh = blockIdx.x / G, gi = blockIdx.x - bh * G;
  const int b = bh / H, h = bh - b * H;
  const int share = (npair + P * G - 1) / (P * G) * P;
  const int pbeg = gi * share, pend = min(npair, pbeg + share);
  const int p = threadIdx.x % P, i = threadIdx.x / P;
  // Twiddles: eight loads a thread in flight before any is stored.
  for (int e0 = threadIdx.x; e0 < N; e0 += 8 * blockDim.x) {
    float2 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * blockDim.x;
      if (TW && e < N) w[u] = __ldg(&W[(e / M) * (e % M)]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < N) {
        S[e] = make_float2(0.f, 0.f);
        if (TW) tw[(e / M) * TWS + e % M] = w[u];
      }
    }
  }
  for (int g0 = pbeg; g0 < pend; g0 += P) {
    const int g = g0 + p;
    const bool active = g < pend;
    const bool pair = 2 * g + 1 < dh;
    const int col = h * dh + 2 * (active ? g : 0);
    const bool aligned = (col & 1) == 0 && (D & 1) == 0;
    const size_t base = (size_t)b * N * D + col;
    // One signal's M values in registers at a time: Q's transforms go back
    // to shared memory and K's product reads them there.
    float2 a[M];
    ld_rows<T, M>(a, Q + base, (size_t)M * D, (size_t)i * D, active, pair, aligned);
    dft<M, false, CxPaired>(a);
    __syncthreads();   // the previous pass's sums have read bq; twiddles ready
#pragma unroll
    for (int k2 = 0; k2 < M; ++k2) bq[k2 * RS + i * P + p] = TW ? cmul(a[k2], tw[i * TWS + k2]) : a[k2];
    ld_rows<T, M>(a, K + base, (size_t)M * D, (size_t)i * D, active, pair, aligned);
    dft<M, false, CxPaired>(a);
#pragma unroll
    for (int k2 = 0; k2 < M; ++k2) bk[k2 * RS + i * P + p] = TW ? cmul(a[k2], tw[i * TWS + k2]) : a[k2];
    __syncthreads();
    // Step 2 (k2 = i): each thread reads and rewrites only its own slots.
#pragma unroll
    for (int n1 = 0; n1 < M; ++n1) a[n1] = bq[i * RS + n1 * P + p];
    dft<M, false, CxPaired>(a);
#pragma unroll
    for (int k1 = 0; k1 < M; ++k1) bq[i * RS + k1 * P + p] = a[k1];
#pragma unroll
    for (int n1 = 0; n1 < M; ++n1) a[n1] = bk[i * RS + n1 * P + p];
    dft<M, false, CxPaired>(a);
#pragma unroll
    for (int k1 = 0; k1 < M; ++k1)
      bq[i * RS + k1 * P + p] = cmulc(bq[i * RS + k1 * P + p], a[k1]);
    __syncthreads();
    // Sum over the pairs, element e starting at pair e mod P (P a power of
    // two): consecutive lanes' rows of P slots would otherwise share banks.
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
      float2 s = S[e];
      const float2* pr = bq + (e / M) * RS + (e % M) * P;   // S[k2][k1]: row k2, slot k1
      for (int q = 0; q < P; ++q) s = cadd(s, pr[(q + e) & (P - 1)]);
      S[e] = s;
    }
  }
  __syncthreads();
  if (part) {
    float2* dst = part + (size_t)blockIdx.x * N;   // [k2][k1], as S
    for (int e = threadIdx.x; e < N; e += blockDim.x) dst[e] = S[e];
    return;
  }
  // The inverse of the one summed signal, on threads t < M.
  const int t = threadIdx.x;
  float2 a[M];
  if (t < M) {   // k2 = t: inverse over k1, to [n1][k2]
#pragma unroll
    for (int k1 = 0; k1 < M; ++k1) a[k1] = S[t * M + k1];
    dft<M, true, CxPaired>(a);
#pragma unroll
    for (int n1 = 0; n1 < M; ++n1) bk[n1 * M + t] = TW ? cmulc(a[n1], tw[n1 * TWS + t]) : a[n1];
  }
  __syncthreads();
  if (t < M) {   // n1 = t: inverse over k2
#pragma unroll
    for (int k2 = 0; k2 < M; ++k2) a[k2] = bk[t * M + k2];
    dft<M, true, CxPaired>(a);
#pragma unroll
    for (int n2 = 0; n2 < M; ++n2) {
      const float v = a[n2].x * scale;
      if (z2) z2[(size_t)bh * N + t + M * n2] = make_float2(v, 0.f);
      if (out) out[(size_t)bh * N + t + M * n2] = v;
    }
  }
}

// The split correlation at N = 32² (the backward's dz*, partial spectra of
// G CTAs a row as corr_reg_kernel leaves them) through one exchange block
// instead of two: after Q's two forward steps, each thread's 32 bins
// (k2 = i, k1 = 0..31 of its pair) wait in tensor memory while K takes the
// same shared block, and K's second step multiplies by them as it reads
// them back.  A CTA then needs 84 KB of shared memory instead of 152 KB, and
// two CTAs (16 warps) share an SM instead of one.  Tensor memory: 128
// columns a CTA, two CTAs 256 of the SM's 512; warp w keeps its threads'
// 64 floats in lanes 32·(w mod 4) + lane, columns 64·(w / 4) ...
constexpr int kCorrTmCols = 128;
constexpr int kCorrTmP = 8;   // pairs a CTA, as conv_reg_pairs(32)
constexpr size_t kSmemCorrTm =
    ((size_t)32 * (32 * kCorrTmP + 8) + 1024 + 32 * 33) * sizeof(float2) + 16;

template <typename T>
__global__ void __launch_bounds__(32 * kCorrTmP, 2)
corr_reg_tm_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                   const float2* __restrict__ W, int D, int H, int dh, int npair,
                   float2* __restrict__ part, int G) {
  constexpr int M = 32, N = M * M, P = kCorrTmP, TWS = reg_tws(M), RS = M * P + 8;
  static_assert(RS == M * P + (P == 8 ? 8 : 0), "row stride as reg_rs(32, 8)");
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);   // [M][M][P], rows RS apart
  float2* S = buf + M * RS;                         // [k2][k1] running sum
  float2* tw = S + N;                               // tw[n1·TWS + k2] = w_N^{n1·k2}
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tw + M * TWS);
  const int warp = threadIdx.x >> 5;
  if (warp == 0) tmem_alloc(tslot, kCorrTmCols);
  const int bh = blockIdx.x / G, gi = blockIdx.x - bh * G;
  const int b = bh / H, h = bh - b * H;
  const int share = (npair + P * G - 1) / (P * G) * P;
  const int pbeg = gi * share, pend = min(npair, pbeg + share);
  const int p = threadIdx.x % P, i = threadIdx.x / P;
  for (int e0 = threadIdx.x; e0 < N; e0 += 8 * blockDim.x) {
    float2 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < N) w[u] = __ldg(&W[(e / M) * (e % M)]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < N) {
        S[e] = make_float2(0.f, 0.f);
        tw[(e / M) * TWS + e % M] = w[u];
      }
    }
  }
  tc_fence_before();
  __syncthreads();   // tensor-memory address, twiddles and sums ready
  tc_fence_after();
  const uint32_t tq = *tslot + ((uint32_t)(32 * (warp & 3)) << 16) + 64u * (uint32_t)(warp >> 2);
  for (int g0 = pbeg; g0 < pend; g0 += P) {
    const int g = g0 + p;
    const bool active = g < pend;
    const bool pair = 2 * g + 1 < dh;
    const int col = h * dh + 2 * (active ? g : 0);
    const bool aligned = (col & 1) == 0 && (D & 1) == 0;
    const size_t base = (size_t)b * N * D + col;
    float2 a[M];
    // Q: step 1 (n1 = i) into the block, step 2 (k2 = i) out of it.
    ld_rows<T, M>(a, Q + base, (size_t)M * D, (size_t)i * D, active, pair, aligned);
    dft<M, false, CxPaired>(a);
    __syncthreads();   // the previous pass's sums have read the block
#pragma unroll
    for (int k2 = 0; k2 < M; ++k2) buf[k2 * RS + i * P + p] = cmul(a[k2], tw[i * TWS + k2]);
    __syncthreads();
#pragma unroll
    for (int n1 = 0; n1 < M; ++n1) a[n1] = buf[i * RS + n1 * P + p];
    dft<M, false, CxPaired>(a);
#pragma unroll
    for (int c = 0; c < 4; ++c) tc_st8c(tq + 16 * c, a + 8 * c);
    tc_wait_st();
    // K: the same two steps through the same block.
    ld_rows<T, M>(a, K + base, (size_t)M * D, (size_t)i * D, active, pair, aligned);
    dft<M, false, CxPaired>(a);
    __syncthreads();   // every thread has read its Q slots
#pragma unroll
    for (int k2 = 0; k2 < M; ++k2) buf[k2 * RS + i * P + p] = cmul(a[k2], tw[i * TWS + k2]);
    __syncthreads();
#pragma unroll
    for (int n1 = 0; n1 < M; ++n1) a[n1] = buf[i * RS + n1 * P + p];
    dft<M, false, CxPaired>(a);
    // FFT(q)·conj(FFT(k)) into the thread's own slots.
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float qv[16];
      tc_ld16(tq + 16 * c, qv);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        buf[i * RS + (8 * c + j) * P + p] = cmulc(make_float2(qv[2 * j], qv[2 * j + 1]), a[8 * c + j]);
    }
    __syncthreads();
    // Sum over the pairs, element e starting at pair e mod P: the lanes of
    // a warp (consecutive k1, 16 words apart) then read distinct banks.
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
      float2 s = S[e];
      const float2* pr = buf + (e / M) * RS + (e % M) * P;   // S[k2][k1]: row k2, slot k1
#pragma unroll
      for (int q = 0; q < P; ++q) s = cadd(s, pr[(q + e) & (P - 1)]);
      S[e] = s;
    }
  }
  __syncthreads();
  float2* dst = part + (size_t)blockIdx.x * N;   // [k2][k1], as S
  for (int e = threadIdx.x; e < N; e += blockDim.x) dst[e] = S[e];
  tc_fence_before();
  __syncthreads();   // every tensor-memory access of the CTA is done
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tslot, kCorrTmCols);
  }
}

size_t corr_reg_smem(int M, int P) {
  return ((size_t)2 * M * reg_rs(M, P) + (size_t)M * M + (size_t)M * reg_tws(M)) *
         sizeof(float2);
}

template <typename T, bool TW>
static cudaError_t corr_t(const cat_plan_s* p, const T* A, const T* Bm, float2* z2, float* out,
                          float scale, float2* part = nullptr, int G = 1) {
  const int M = p->sm.reg_m, P = p->sm.G;
  const size_t smem = corr_reg_smem(M, P);
  switch (M) {
#define CAT_M(m)                                                                              \
  case m:                                                                                     \
    corr_reg_kernel<T, m, TW><<<p->B * p->H * G, m * P, smem, p->stream>>>(                    \
        A, Bm, z2, out, p->tw, p->D, p->H, p->dh, p->npair, P, scale, part, G);               \
    break;
    CAT_M(8) CAT_M(14) CAT_M(16) CAT_M(32)
#undef CAT_M
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_scores2d_reg(const cat_plan_s* p, const void* Q, const void* K, float* out) {
  if (p->B * p->H == 0) return cudaSuccess;
  const float scale = 1.0f / ((float)p->dh * (float)p->N);
  if (p->dtype == 1)
    return corr_t<__nv_bfloat16, false>(p, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K,
                                        p->z2, out, scale);
  return corr_t<float, false>(p, (const float*)Q, (const float*)K, p->z2, out, scale);
}

cudaError_t launch_corr_reg(const cat_plan_s* p, const void* G, const void* V, float* dzs) {
  if (p->B * p->H == 0) return cudaSuccess;
  const float scale = 1.0f / (float)p->N;
  if (p->dtype == 1)
    return corr_t<__nv_bfloat16, true>(p, (const __nv_bfloat16*)G, (const __nv_bfloat16*)V,
                                       nullptr, dzs, scale);
  return corr_t<float, true>(p, (const float*)G, (const float*)V, nullptr, dzs, scale);
}

// Softmax and spectrum of z* for N = M² in registers: a group of GL lanes
// (M rounded up to a power of two; lanes >= M idle) owns one (b, h) row, so
// the row maximum and Σ exp(z - m) are lane-group shuffles.  Lane i holds
// z[i + M·n2] (n1 = i); it writes z* there, takes the DFT over n2, the
// twiddle w_N^{n1·k2}, and exchanges through the row's shared-memory block
// (row stride M + 1); then lane i (k2 = i) takes the DFT over n1 and writes
// FFT(z*)/N at the natural bins k2 + M·k1.  The exact difference z - m comes
// from the double-float score (exp_shifted), as in the block kernel.
constexpr int kSpecRegThreads = 256;

template <int M, bool TW = true>
__global__ void __launch_bounds__(kSpecRegThreads)
softmax_spectrum_reg(const float2* z, float* __restrict__ zs,
                     float2* __restrict__ zf, const float2* __restrict__ W, int rows) {
  constexpr int N = M * M;
  constexpr int GL = M <= 8 ? 8 : (M <= 16 ? 16 : 32);
  constexpr int RS = M + 1;                  // shared row of one k2 (complex)
  extern __shared__ float4 smem4[];
  float2* xb = reinterpret_cast<float2*>(smem4);   // one block of M·RS per row
  // Rows are independent (a row's lanes are one warp's): the CTA holds
  // blockDim.x / GL of them, whole warps, sized by the launch to the row
  // count.  Lane i reads its twiddles w_N^{i·k2} straight from the table.
  const int i = threadIdx.x % GL, r = threadIdx.x / GL;
  const int row = blockIdx.x * (blockDim.x / GL) + r;
  // Let the product kernel behind (its programmatic dependent) launch, then
  // wait for the scores (a no-op after an ordinary launch).
  pdl_trigger();
  pdl_wait();
  const bool act = i < M && row < rows;
  const float2* src = z + (size_t)(row < rows ? row : 0) * N;
  float2 v[M];
#pragma unroll
  for (int n2 = 0; n2 < M; ++n2) v[n2] = act ? ld_dep(src + i + M * n2) : make_float2(-INFINITY, 0.f);
  float m = -INFINITY;
#pragma unroll
  for (int n2 = 0; n2 < M; ++n2) m = fmaxf(m, v[n2].x);
#pragma unroll
  for (int o = GL / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
  float2 a[M];
#pragma unroll
  for (int n2 = 0; n2 < M; ++n2) {
    const float e = act ? exp_shifted(v[n2], m) : 0.f;
    a[n2] = make_float2(e, 0.f);
    sum += e;
  }
#pragma unroll
  for (int o = GL / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.0f / sum;
  float* out = zs + (size_t)row * N;
#pragma unroll
  for (int n2 = 0; n2 < M; ++n2) {
    a[n2].x *= inv;
    if (act) out[i + M * n2] = a[n2].x;
  }
  dft<M, false, CxPaired>(a);
  float2* xr = xb + r * M * RS;
  if (i < M) {
#pragma unroll
    for (int k2 = 0; k2 < M; ++k2) xr[k2 * RS + i] = TW ? cmul(a[k2], __ldg(&W[i * k2])) : a[k2];
  }
  __syncwarp();      // a row's lanes are one warp's
  if (i < M) {
#pragma unroll
    for (int n1 = 0; n1 < M; ++n1) a[n1] = xr[i * RS + n1];
  }
  dft<M, false, CxPaired>(a);
  if (act) {
    const float invN = 1.0f / (float)N;
    float2* spec = zf + (size_t)row * N + i;
#pragma unroll
    for (int k1 = 0; k1 < M; ++k1) spec[M * k1] = cscale(a[k1], invN);
  }
}

// Rows per CTA: whole warps, at most kSpecRegThreads threads, and no more
// rows than keep two CTAs on every SM when the row count is small.
static int spectrum_reg_rows(int M, int rows, int sms) {
  const int GL = M <= 8 ? 8 : (M <= 16 ? 16 : 32);
  const int unit = 32 / GL, most = kSpecRegThreads / GL;
  int per = rows / (2 * (sms > 0 ? sms : 1));
  per = per < unit ? unit : (per > most ? most : per);
  return per / unit * unit;
}

size_t spectrum_reg_smem(int M) {
  const int GL = M <= 8 ? 8 : (M <= 16 ? 16 : 32);
  return (size_t)(kSpecRegThreads / GL) * M * (M + 1) * sizeof(float2);
}

// The same softmax and spectrum for N = 32², one (b, h) row per CTA of 128
// threads: each 32-point DFT of the two steps is split over 4 threads
// (n2 = q + 4m, k2 = ka + 8kb: thread q takes the DFT-8 over m, times
// w_32^{q·ka}; the DFT-4 over q runs after a hand-over through shared
// memory, thread q taking ka = 2q, 2q + 1), so that a row's serial chain is
// about a quarter of the one-warp kernel's.  The softmax is spread over the
// 128 threads.  Output as softmax_spectrum_reg: z* in natural order, the
// spectrum at index k2 + 32·k1.
constexpr int kSpecQ4Threads = 128;
// CTAs per (b, h) row of the split register correlation (N = 32²).
constexpr int kCorrSplitG = 4;

// Column of element (row, col) in the q4 kernels' [32][36] arrays: the low
// two bits of col flipped by bits 2-3 of row, so that a warp writing one
// column of 32 rows (the transposed store of σ) hits distinct banks, while
// the step's reads (four rows a half-warp, four columns each) stay
// conflict-free.
__device__ __forceinline__ int q4_col(int row, int col) { return col ^ ((row >> 2) & 3); }

// One 32-point DFT (INV: its unscaled inverse) of column g of `in` ([g][n]
// with row stride 36, columns placed by q4_col), split over the 4 threads q
// of the column; thread q ends with bins 2q + h + 8kb in out[4h + kb].
// W: the length-1024 table.
template <bool INV>
__device__ __forceinline__ void spec_q4_step(const float2* __restrict__ in, float2* ex,
                                             const float2* __restrict__ W, int g, int q,
                                             float2 (&out)[8]) {
  constexpr int LD = 36;
  float2 a[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) a[m] = in[g * LD + q4_col(g, q + 4 * m)];
  dft<8, INV, CxPaired>(a);
  float2* mine = ex + g * 33;
#pragma unroll
  for (int ka = 0; ka < 8; ++ka)
    mine[q * 8 + ka] = ka == 0 || q == 0 ? a[ka] : twr<INV>(a[ka], W[32 * q * ka]);
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int ka = 2 * q + h;
    float2 c[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) c[r] = mine[r * 8 + ka];
    dft_small<4, INV>(c);
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) out[4 * h + kb] = c[kb];   // bin ka + 8·kb
  }
}

template <bool TW>
__global__ void __launch_bounds__(kSpecQ4Threads)
softmax_spectrum_q4(const float2* z, float* __restrict__ zs, float2* __restrict__ zf,
                    const float2* __restrict__ W) {
  constexpr int N = 1024, LD = 36;
  __shared__ float2 sa[32 * LD];   // σ as [n1][n2], then the spectrum
  __shared__ float2 sb[32 * LD];   // step 1's output as [k2][n1]
  __shared__ float2 ex[32 * 33];   // the 4-thread hand-over, one block per column
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int t = threadIdx.x, row = blockIdx.x;
  const float2* src = z + (size_t)row * N;
  float2 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = ld_dep(src + t + kSpecQ4Threads * j);
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, v[j].x);
  m = block_reduce<true>(m, red);
  float e[8], sum = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    e[j] = exp_shifted(v[j], m);
    sum += e[j];
  }
  sum = block_reduce<false>(sum, red);
  const float inv = 1.0f / sum;
  float* out = zs + (size_t)row * N;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int n = t + kSpecQ4Threads * j;
    const float sg = e[j] * inv;
    out[n] = sg;
    sa[(n & 31) * LD + q4_col(n & 31, n >> 5)] = make_float2(sg, 0.f);
  }
  __syncthreads();
  const int g = t >> 2, q = t & 3;
  float2 y[8];
  spec_q4_step<false>(sa, ex, W, g, q, y);   // column n1 = g: bins k2 = 2q + h + 8kb
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      const int k2 = 2 * q + h + 8 * kb;
      const float2 w = y[4 * h + kb];
      sb[k2 * LD + q4_col(k2, g)] = TW ? cmul(w, W[g * k2]) : w;
    }
  __syncthreads();
  spec_q4_step<false>(sb, ex, W, g, q, y);   // k2 = g: bins k1 = 2q + h + 8kb
  const float invN = 1.0f / (float)N;
  float2* so = sa;                         // step 1 is done with sa
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) so[g + 32 * (2 * q + h + 8 * kb)] = cscale(y[4 * h + kb], invN);
  __syncthreads();
  float2* spec = zf + (size_t)row * N;
#pragma unroll
  for (int j = 0; j < 8; ++j) spec[t + kSpecQ4Threads * j] = so[t + kSpecQ4Threads * j];
}

// The backward's correlation at N = 32², finished: the G partial spectra
// of a (b, h) row (S[k2][k1], from corr_reg_kernel's partial mode) added in
// the order g = 0, 1, …; the inverse DFT (over k1, conjugate twiddle
// w_N^{-n1·k2}, over k2; each 32-point DFT split over 4 threads as in
// softmax_spectrum_q4); dz* = Re/N; then the softmax backward
// dz = z*⊙(dz* − ⟨z*, dz*⟩), the threads' fp32 partial sums added in fp64 in
// a fixed order.  One row per CTA of 128 threads.
__global__ void __launch_bounds__(kSpecQ4Threads)
corr_finish_q4(const float2* __restrict__ part, int G, const float* __restrict__ zs,
               float* __restrict__ dzs, float* __restrict__ dz,
               const float2* __restrict__ W) {
  constexpr int N = 1024, LD = 36;
  __shared__ float2 sa[32 * LD];   // S as [k2][k1], then dz* in natural order
  __shared__ float2 sb[32 * LD];   // step 1's output as [n1][k2]
  __shared__ float2 ex[32 * 33];
  __shared__ double red[kSpecQ4Threads / 32];
  __shared__ float total;
  const int t = threadIdx.x, row = blockIdx.x;
  const float2* src = part + (size_t)row * G * N;
  float2 acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = make_float2(0.f, 0.f);
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = cadd(acc[j], src[(size_t)g * N + t + kSpecQ4Threads * j]);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = t + kSpecQ4Threads * j;   // e = k2·32 + k1
    sa[(e >> 5) * LD + q4_col(e >> 5, e & 31)] = acc[j];
  }
  __syncthreads();
  const int g = t >> 2, q = t & 3;
  float2 y[8];
  spec_q4_step<true>(sa, ex, W, g, q, y);   // k2 = g: bins n1 = 2q + h + 8kb
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      const int n1 = 2 * q + h + 8 * kb;
      sb[n1 * LD + q4_col(n1, g)] = cmulc(y[4 * h + kb], W[n1 * g]);
    }
  __syncthreads();
  spec_q4_step<true>(sb, ex, W, g, q, y);   // n1 = g: bins n2 = 2q + h + 8kb
  float* flat = reinterpret_cast<float*>(sa);   // dz*[n1 + 32·n2]
  const float invN = 1.0f / (float)N;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) flat[g + 32 * (2 * q + h + 8 * kb)] = y[4 * h + kb].x * invN;
  __syncthreads();
  const size_t off = (size_t)row * N;
  float d[8], zv[8], pt = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int n = t + kSpecQ4Threads * j;
    d[j] = flat[n];
    zv[j] = zs[off + n];
    dzs[off + n] = d[j];
    pt = fmaf(zv[j], d[j], pt);
  }
  double sd = pt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sd += __shfl_xor_sync(0xffffffffu, sd, o);
  if ((t & 31) == 0) red[t >> 5] = sd;
  __syncthreads();
  if (t == 0) {
    double tot = 0.0;
    for (int w = 0; w < kSpecQ4Threads / 32; ++w) tot += red[w];
    total = (float)tot;
  }
  __syncthreads();
  const float sf = total;
#pragma unroll
  for (int j = 0; j < 8; ++j) dz[off + t + kSpecQ4Threads * j] = zv[j] * (d[j] - sf);
}

bool corr_reg_split_fits(const cat_plan_s* p) {
  return p->sm.reg_m == 32 && !p->twod &&
         (size_t)p->B * p->H * kCorrSplitG * p->N * sizeof(float2) <= p->bw.scratch_bytes;
}

cudaError_t launch_corr_reg_split(const cat_plan_s* p, const void* G, const void* V) {
  const int rows = p->B * p->H;
  if (rows == 0) return cudaSuccess;
  float2* part = p->bw_scr;
  const dim3 grid(rows * kCorrSplitG), block(32 * kCorrTmP);
  if (p->dtype == 1)
    corr_reg_tm_kernel<__nv_bfloat16><<<grid, block, kSmemCorrTm, p->stream>>>(
        (const __nv_bfloat16*)G, (const __nv_bfloat16*)V, p->tw, p->D, p->H, p->dh, p->npair,
        part, kCorrSplitG);
  else
    corr_reg_tm_kernel<float><<<grid, block, kSmemCorrTm, p->stream>>>(
        (const float*)G, (const float*)V, p->tw, p->D, p->H, p->dh, p->npair, part, kCorrSplitG);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  corr_finish_q4<<<rows, kSpecQ4Threads, 0, p->stream>>>(part, kCorrSplitG, p->zs, p->bw_dzs,
                                                         p->bw_dz, p->tw);
  return cudaGetLastError();
}

// An ordinary launch, or (dep) one as the programmatic dependent of the
// kernel ahead on the stream.
template <typename... KArgs, typename... Args>
static cudaError_t spec_launch(bool dep, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                               size_t smem, cudaStream_t st, Args... args) {
  if (dep) return launch_dependent(kernel, grid, block, smem, st, args...);
  kernel<<<grid, block, smem, st>>>(args...);
  return cudaGetLastError();
}

// The spectrum kernel follows the scores; the product kernel behind it is
// its programmatic dependent.  After the 1-D score it is an ordinary
// launch: as the score's dependent it let the product kernel start while
// the score still ran, and the product's value loads and first transforms
// then slowed the score, which every later step waits for (per forward,
// vit196 30.1 -> 26.7 us, gpt2_f32 66.1 -> 61.8 us, gpt2_bf16 47.8 ->
// 43.1 us once it waits).  After the 2-D scores (few long CTAs) the
// dependent launch still pays (ca_vit196 39.0 against 41.0 us).
template <bool TW>
static cudaError_t spectrum_reg_t(const cat_plan_s* p) {
  const int rows = p->B * p->H;
  if (rows == 0) return cudaSuccess;
  const int M = p->sm.reg_m;
  const bool dep = !TW;
  if (M == 32)
    return spec_launch(dep, softmax_spectrum_q4<TW>, dim3(rows), dim3(kSpecQ4Threads), 0,
                       p->stream, (const float2*)p->z2, p->zs, p->zf, (const float2*)p->tw);
  const int GL = M <= 8 ? 8 : (M <= 16 ? 16 : 32);
  const int per = spectrum_reg_rows(M, rows, p->sms);
  const int ctas = (rows + per - 1) / per;
  const size_t smem = (size_t)per * M * (M + 1) * sizeof(float2);
  switch (M) {
#define CAT_M(m)                                                                         \
  case m:                                                                                \
    return spec_launch(dep, softmax_spectrum_reg<m, TW>, dim3(ctas), dim3(per * GL), smem,  \
                       p->stream, (const float2*)p->z2, p->zs, p->zf, (const float2*)p->tw, \
                       rows);
    CAT_M(8) CAT_M(14) CAT_M(16) CAT_M(32)
#undef CAT_M
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_softmax_spectrum_reg(const cat_plan_s* p) {
  return p->twod ? spectrum_reg_t<false>(p) : spectrum_reg_t<true>(p);
}

// Pairs per CTA and the CTA shape for side M: 16 pairs (8 for M = 32, so
// that a CTA of 256 threads and 74 KB of shared memory leaves room for more).
int conv_reg_pairs(int M) { return M == 32 ? 8 : 16; }

size_t conv_reg_smem(int M, int P) {
  return ((size_t)M * reg_rs(M, P) + (size_t)M * reg_tws(M) + (size_t)M * M) * sizeof(float2);
}

template <typename T, bool TW>
static cudaError_t setup_tw() {
  cudaError_t e = allow_max_smem(softmax_spectrum_reg<8, TW>);
  if (e == cudaSuccess) e = allow_max_smem(softmax_spectrum_reg<14, TW>);
  if (e == cudaSuccess) e = allow_max_smem(softmax_spectrum_reg<16, TW>);
  if (e == cudaSuccess) e = allow_max_smem(softmax_spectrum_reg<32, TW>);
  if (e == cudaSuccess) e = allow_max_smem(conv_reg_kernel<T, 8, TW>);
  if (e == cudaSuccess) e = allow_max_smem(conv_reg_kernel<T, 14, TW>);
  if (e == cudaSuccess) e = allow_max_smem(conv_reg_kernel<T, 16, TW>);
  if (e == cudaSuccess) e = allow_max_smem(conv_reg_kernel<T, 32, TW>);
  return e;
}

template <typename T>
static cudaError_t setup_t() {
  cudaError_t e = setup_tw<T, true>();
  if (e == cudaSuccess) e = setup_tw<T, false>();
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 8, false>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 14, false>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 16, false>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 32, false>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 8, true>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 14, true>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 16, true>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_kernel<T, 32, true>);
  if (e == cudaSuccess) e = allow_max_smem(corr_reg_tm_kernel<T>);
  return e;
}

cudaError_t setup_conv_reg(const cat_plan_s* p) {
  return p->dtype == 1 ? setup_t<__nv_bfloat16>() : setup_t<float>();
}

template <typename T, bool TW>
static cudaError_t launch_tw(const cat_plan_s* p, const T* V, T* O, bool conj) {
  const int M = p->sm.reg_m, P = p->sm.G, groups = p->sm.groups;
  const int ctas = p->B * p->H * groups;
  const dim3 block(M * P);
  const size_t smem = p->sm.smem;
  switch (M) {
#define CAT_M(m)                                                                             \
  case m:                                                                                    \
    return launch_dependent(conv_reg_kernel<T, m, TW>, dim3(ctas), block, smem, p->stream, V, \
                            O, (const float2*)p->zf, (const float2*)p->tw, p->D, p->H, p->dh, \
                            p->npair, P, groups, (int)conj);
    CAT_M(8) CAT_M(14) CAT_M(16) CAT_M(32)
#undef CAT_M
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t launch_t(const cat_plan_s* p, const T* V, T* O, bool conj) {
  return p->twod ? launch_tw<T, false>(p, V, O, conj) : launch_tw<T, true>(p, V, O, conj);
}

cudaError_t launch_conv_reg(const cat_plan_s* p, const void* V, void* O, bool conj) {
  if (p->B == 0) return cudaSuccess;
  if (p->dtype == 1) return launch_t(p, (const __nv_bfloat16*)V, (__nv_bfloat16*)O, conj);
  return launch_t(p, (const float*)V, (float*)O, conj);
}

}  // namespace cat
