// Backward pass of CAT.  The notes page "CAT: Circular-Convolutional
// Attention for Sub-Quadratic Transformers" trains CAT layers with the usual
// losses and optimisers (section 损失函数 / 训练策略) but gives no gradient
// formulas; these follow from the forward definitions of section 方法详解
// by the chain rule.  With G = dL/dO the upstream gradient:
//
//   dV   = circ(z*)^T G                  (the forward's circulant product with
//                                         the scores reversed, see below)
//   dz*[h, k] = sum_{c in h} sum_i G[i, c] V[(i - k) mod N, c]
//             = Re IFFT( sum_{c in h} FFT(G[:, c]) ⊙ conj(FFT(V[:, c])) )
//   dz   = z* ⊙ (dz* - <z*, dz*>)         (softmax Jacobian)
//   dW_A = X^T dz,   dX = dz W_A^T
//
// Correlation.  Columns (c, c+1) are packed as complex signals g = G_c +
// i G_{c+1} and v = V_c + i V_{c+1}.  Then FFT(g)·conj(FFT(v)) = Y_c + Y_{c+1}
// + i (FFT(G_{c+1})conj(FFT(V_c)) - FFT(G_c)conj(FFT(V_{c+1}))), where Y_c is
// the spectrum of column c's (real) correlation; the bracket is the spectrum
// of a real signal too, so after the inverse transform the cross terms are
// purely imaginary and the real part is the sum of both columns'
// correlations.  The sum over a head's pairs is taken on the spectra, so each
// (b, h) needs one inverse transform.
//
// The transforms use the four-step split N = N1·N2 (n = n1 + N1·n2,
// k = N2·k1 + k2) of the long-sequence forward path, or N1 = N, N2 = 1 for
// short rows (on the fast path's shapes, its own pass A and the register
// kernel fsf_corr_b take passes A and B, and pass C below runs on their
// one-signal result):
//   pass A (per n1): length-N2 DFTs of every G and V pair, twiddle
//     w_N^{n1 k2}, into scratch [bh][k2][n1][q] (q < npair: G pairs,
//     q >= npair: V pairs);
//   pass B (per k2): length-N1 DFTs give both spectra at bins N2 k1 + k2;
//     sum over pairs of FFT(g)·conj(FFT(v)); inverse DFT over k1; conjugate
//     twiddle; into scratch signal 0;
//   pass C (per n1): inverse DFT over k2; real part / N is dz*.
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "cat_internal.h"
#include "elem.cuh"

namespace cat {

// ---------------------------------------------------------------------------
// dV: circ(z*)^T = circ(r) with r[n] = z*[(-n) mod N].  The softmax commutes
// with any permutation of the tokens, so reversing the scores
// z[n] -> z[(-n) mod N] makes the forward's spectrum and product kernels
// compute circ(z*)^T·G.  In place: entries n and N - n swap, 1 <= n < N - n.
// ---------------------------------------------------------------------------
__global__ void reverse_scores_kernel(float2* __restrict__ z, int N, long long items) {
  const int half = (N - 1) / 2;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < items;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / half;
    const int n = 1 + (int)(i - row * half);
    float2* r = z + row * (long long)N;
    const float2 a = r[n], b = r[N - n];
    r[n] = b;
    r[N - n] = a;
  }
}

// ---------------------------------------------------------------------------
// Correlation pass A.  blockIdx.x = (bhl · (N1/TA) + tile) · groups + grp.
// Shared layout: signal (t, s) at buf[(t·S + s)·N2], S = 2·gc; s < gc are
// G pairs g0 + s, s >= gc the V pairs g0 + s - gc.
// ---------------------------------------------------------------------------
template <typename T, bool TW>
__global__ void __launch_bounds__(1024)
corr_pass_a(const T* __restrict__ G, const T* __restrict__ V, float2* __restrict__ scr,
            const float2* __restrict__ W, RadixPlan rp2, int N, int N1, int D, int H, int dh,
            int npair, int GA, int groups, int TA, int Q, int bh0, unsigned int* status) {
  extern __shared__ float2 buf[];
  const int N2 = rp2.L;
  const int ntile = N1 / TA;
  int r = blockIdx.x;
  const int grp = r % groups; r /= groups;
  const int tile = r % ntile;
  const int bhl = r / ntile;
  const int bh = bh0 + bhl;
  const int b = bh / H, h = bh - b * H;
  const int g0 = grp * GA;
  const int gc = min(GA, npair - g0);
  if (gc <= 0) return;
  const int S = 2 * gc;
  const int count = TA * S;
  if (count * N2 > vals_capacity(rp2) * (int)blockDim.x) {
    report(status, 0x601);
    return;
  }
  const int n1_0 = tile * TA;
  const int col0 = h * dh + 2 * g0;
  const bool full_pairs = (2 * (g0 + gc) <= dh);
  const bool aligned = ((col0 & 1) == 0) && ((D & 1) == 0);   // even column, even row length
  const size_t boff = (size_t)b * N * D;

  // Load: s fastest (a row's G pairs, then its V pairs), then t, then n2.
  const int total = count * N2;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int s = idx % S, q = idx / S;
    const int t = q % TA, n2 = q / TA;
    const int n = n1_0 + t + N1 * n2;
    const bool isv = s >= gc;
    const int g = isv ? s - gc : s;
    const T* src = (isv ? V : G) + boff + (size_t)n * D + col0 + 2 * g;
    float2 v;
    if (full_pairs && aligned) {
      v = ld_pair(src);
    } else {
      v.x = ld_elem(src);
      v.y = (2 * (g0 + g) + 1 < dh) ? ld_elem(src + 1) : 0.f;
    }
    buf[(t * S + s) * N2 + n2] = v;
  }
  __syncthreads();
  block_fft<false>(buf, rp2, count, N2, W, N1);

  float2* srow = scr + (size_t)bhl * N * Q;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int s = idx % S, q = idx / S;
    const int t = q % TA, k2 = q / TA;
    const int n1 = n1_0 + t;
    float2 v = buf[(t * S + s) * N2 + k2];
    if (TW) v = cmul(v, __ldg(&W[(size_t)n1 * k2]));
    const int qi = s < gc ? g0 + s : npair + g0 + (s - gc);
    srow[((size_t)k2 * N1 + n1) * Q + qi] = v;
  }
}

// ---------------------------------------------------------------------------
// Correlation pass B.  blockIdx.x = bhl · (N2/TB) + tile.  The head's pairs
// go through in chunks of GB: signal (t, s) of a chunk at buf[(t·S + s)·N1]
// (S = 2·gc: G pairs, then V pairs); the running sum of FFT(g)·conj(FFT(v))
// for k2-slot t at acc[t·N1 + k1], after the chunk buffer.
// ---------------------------------------------------------------------------
template <bool TW>
__global__ void __launch_bounds__(1024)
corr_pass_b(float2* __restrict__ scr, const float2* __restrict__ W, RadixPlan rp1, int N,
            int N2, int npair, int GB, int TB, int Q, unsigned int* status) {
  extern __shared__ float2 buf[];
  const int N1 = rp1.L;
  const int ntile = N2 / TB;
  const int tile = blockIdx.x % ntile;
  const int bhl = blockIdx.x / ntile;
  const int k2_0 = tile * TB;
  if (TB * 2 * GB * N1 > vals_capacity(rp1) * (int)blockDim.x ||
      TB * N1 > vals_capacity(rp1) * (int)blockDim.x) {
    report(status, 0x602);
    return;
  }
  float2* acc = buf + (size_t)TB * 2 * GB * N1;
  float2* srow = scr + (size_t)bhl * N * Q;
  const int npts = TB * N1;
  for (int i = threadIdx.x; i < npts; i += blockDim.x) acc[i] = make_float2(0.f, 0.f);

  for (int c0 = 0; c0 < npair; c0 += GB) {
    const int gc = min(GB, npair - c0);
    const int S = 2 * gc;
    const int total = TB * S * N1;
    __syncthreads();   // the previous chunk's reads of buf are done
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
      const int s = idx % S, q = idx / S;
      const int n1 = q % N1, t = q / N1;
      const int k2 = k2_0 + t;
      const int qi = s < gc ? c0 + s : npair + c0 + (s - gc);
      buf[(t * S + s) * N1 + n1] = srow[((size_t)k2 * N1 + n1) * Q + qi];
    }
    __syncthreads();
    block_fft<false>(buf, rp1, TB * S, N1, W, N2);
    for (int idx = threadIdx.x; idx < npts; idx += blockDim.x) {
      const int k1 = idx % N1, t = idx / N1;
      float2 a = acc[idx];
      for (int s = 0; s < gc; ++s)
        a = cadd(a, cmulc(buf[(t * S + s) * N1 + k1], buf[(t * S + gc + s) * N1 + k1]));
      acc[idx] = a;
    }
  }
  __syncthreads();
  block_fft<true>(acc, rp1, TB, N1, W, N2);

  // Conjugate twiddle w_N^{-n1 k2}; the result goes to scratch signal 0
  // (this CTA's k2 slots have been read in full).
  for (int idx = threadIdx.x; idx < npts; idx += blockDim.x) {
    const int n1 = idx % N1, t = idx / N1;
    const int k2 = k2_0 + t;
    srow[((size_t)k2 * N1 + n1) * Q] = TW ? cmulc(acc[idx], __ldg(&W[(size_t)n1 * k2])) : acc[idx];
  }
}

// ---------------------------------------------------------------------------
// Correlation pass C.  blockIdx.x = bhl · (N1/TC) + tile.  Inverse DFT over
// k2 of scratch signal 0 for TC values of n1; dz*[n1 + N1 n2] = Re / N.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
corr_pass_c(const float2* __restrict__ scr, float* __restrict__ dzs,
            const float2* __restrict__ W, RadixPlan rp2, int N, int N1, int TC, int Q, int bh0,
            unsigned int* status) {
  extern __shared__ float2 buf[];
  const int N2 = rp2.L;
  const int ntile = N1 / TC;
  const int tile = blockIdx.x % ntile;
  const int bhl = blockIdx.x / ntile;
  if (TC * N2 > vals_capacity(rp2) * (int)blockDim.x) {
    report(status, 0x603);
    return;
  }
  const int n1_0 = tile * TC;
  const float2* srow = scr + (size_t)bhl * N * Q;
  const int total = TC * N2;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int t = idx % TC, k2 = idx / TC;
    buf[t * N2 + k2] = srow[((size_t)k2 * N1 + n1_0 + t) * Q];
  }
  __syncthreads();
  block_fft<true>(buf, rp2, TC, N2, W, N1);
  const float invN = 1.0f / (float)N;
  float* out = dzs + (size_t)(bh0 + bhl) * N;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int t = idx % TC, n2 = idx / TC;
    out[n1_0 + t + (size_t)N1 * n2] = buf[t * N2 + n2].x * invN;
  }
}

// ---------------------------------------------------------------------------
// Softmax backward, one CTA per (b, h) row: s = sum_m z*[m] dz*[m] (fp32 per
// thread, the threads' partial sums added in fp64 in a fixed order), then
// dz[n] = z*[n] (dz*[n] - s).
// ---------------------------------------------------------------------------
constexpr int kSmBwThreads = 1024;

__global__ void __launch_bounds__(kSmBwThreads)
softmax_bw_kernel(const float* __restrict__ zs, const float* __restrict__ dzs,
                  float* __restrict__ dz, int N) {
  __shared__ double red[kSmBwThreads / 32];
  __shared__ float total;
  const size_t off = (size_t)blockIdx.x * N;
  const int bd = blockDim.x;
  // Each thread's terms in order n = t, t + bd, ...; eight of each operand
  // loaded before they are used.
  float part = 0.f;
  int n = threadIdx.x;
  for (; n + 7 * bd < N; n += 8 * bd) {
    float a[8], c[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      a[u] = zs[off + n + u * bd];
      c[u] = dzs[off + n + u * bd];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) part = fmaf(a[u], c[u], part);
  }
  for (; n < N; n += bd) part = fmaf(zs[off + n], dzs[off + n], part);
  double s = part;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  if (lane == 0) red[warp] = s;
  __syncthreads();
  // One thread adds the warps' sums in order (fp64 is a slow pipe on this
  // GPU: the sum is done once, not by every thread), then shares it.
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < nw; ++w) tot += red[w];
    total = (float)tot;
  }
  __syncthreads();
  const float sf = total;
  n = threadIdx.x;
  for (; n + 7 * bd < N; n += 8 * bd) {
    float a[8], c[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      a[u] = zs[off + n + u * bd];
      c[u] = dzs[off + n + u * bd];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) dz[off + n + u * bd] = a[u] * (c[u] - sf);
  }
  for (; n < N; n += bd) dz[off + n] = zs[off + n] * (dzs[off + n] - sf);
}

// ---------------------------------------------------------------------------
// dW_A[d, h] = sum over tokens of X[t, d] dz[h, t]: each CTA takes a range of
// tokens (split), 512 columns d (2 consecutive per thread) and 16 heads,
// and writes its partial sums to part[split][h][d]; dwa_reduce adds the
// splits in order.
// ---------------------------------------------------------------------------
constexpr int kDwThreads = 256, kDwDpt = 2, kDwH = 16, kDwTok = 32, kDwPre = 16;
static_assert(kDwTok % kDwPre == 0, "token tile is whole groups of preloads");

// Two consecutive elements from column d0 (d0 even); `left` columns remain;
// vec: the row length is even, so the two are one aligned pair.
__device__ __forceinline__ void ld2(const float* p, int left, bool vec, float* x) {
  if (vec) {
    const float2 v = __ldg(reinterpret_cast<const float2*>(p));
    x[0] = v.x; x[1] = v.y;
  } else {
    x[0] = __ldg(p);
    x[1] = left > 1 ? __ldg(p + 1) : 0.f;
  }
}
__device__ __forceinline__ void ld2(const __nv_bfloat16* p, int left, bool vec, float* x) {
  if (vec) {
    const float2 v = ld_pair(p);
    x[0] = v.x; x[1] = v.y;
  } else {
    x[0] = ld_elem(p);
    x[1] = left > 1 ? ld_elem(p + 1) : 0.f;
  }
}
__device__ __forceinline__ void st2(float* p, int left, bool vec, const float* x) {
  if (vec) {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  } else {
    p[0] = x[0];
    if (left > 1) p[1] = x[1];
  }
}
__device__ __forceinline__ void st2(__nv_bfloat16* p, int left, bool vec, const float* x) {
  if (vec) {
    st_pair(p, make_float2(x[0], x[1]));
  } else {
    st_elem(p, x[0]);
    if (left > 1) st_elem(p + 1, x[1]);
  }
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kDwThreads, 2)
dwa_partial_kernel(const T* __restrict__ X, const float* __restrict__ dz, float* __restrict__ part,
                   int N, int D, int H, long long tokens, long long tps) {
  __shared__ __align__(16) float dzs[kDwTok][kDwH];
  const int split = blockIdx.x;
  const int d0 = (blockIdx.y * kDwThreads + threadIdx.x) * kDwDpt;
  const int h0 = blockIdx.z * kDwH;
  const int hc = min(kDwH, H - h0);
  const long long t_begin = (long long)split * tps;
  const long long t_end = min(tokens, t_begin + tps);
  constexpr bool vec = VEC;   // even row length: column pairs are aligned
  float acc[kDwDpt][kDwH];
#pragma unroll
  for (int j = 0; j < kDwDpt; ++j)
#pragma unroll
    for (int q = 0; q < kDwH; ++q) acc[j][q] = 0.f;

  for (long long t0 = t_begin; t0 < t_end; t0 += kDwTok) {
    __syncthreads();
    for (int i = threadIdx.x; i < kDwTok * kDwH; i += kDwThreads) {
      const int tl = i % kDwTok, hl = i / kDwTok;
      const long long t = t0 + tl;
      float v = 0.f;
      if (t < t_end && hl < hc) {
        const long long b = t / N, n = t - b * N;
        v = dz[((size_t)b * H + h0 + hl) * N + n];
      }
      dzs[tl][hl] = v;
    }
    __syncthreads();
    const int nt = (int)min((long long)kDwTok, t_end - t0);
    if (d0 < D) {
      // Sixteen tokens' loads in flight before their products.
      // The loads take no branch: a token past the tile reads the last
      // valid row instead (its dzs entry is zero, so it adds nothing).
      for (int tb = 0; tb < nt; tb += kDwPre) {
        float x[kDwPre][kDwDpt];
#pragma unroll
        for (int u = 0; u < kDwPre; ++u) {
          const long long t = min(t0 + tb + u, tokens - 1);
          ld2(X + (size_t)t * D + d0, D - d0, vec, x[u]);
        }
#pragma unroll
        for (int u = 0; u < kDwPre; ++u) {
          const float4* zr = reinterpret_cast<const float4*>(&dzs[(tb + u) & (kDwTok - 1)][0]);
#pragma unroll
          for (int q = 0; q < kDwH / 4; ++q) {
            const float4 z = zr[q];
#pragma unroll
            for (int j = 0; j < kDwDpt; ++j) {
              acc[j][4 * q + 0] = fmaf(x[u][j], z.x, acc[j][4 * q + 0]);
              acc[j][4 * q + 1] = fmaf(x[u][j], z.y, acc[j][4 * q + 1]);
              acc[j][4 * q + 2] = fmaf(x[u][j], z.z, acc[j][4 * q + 2]);
              acc[j][4 * q + 3] = fmaf(x[u][j], z.w, acc[j][4 * q + 3]);
            }
          }
        }
      }
    }
  }
  if (d0 >= D) return;
#pragma unroll
  for (int q = 0; q < kDwH; ++q) {
    if (q < hc) {
      float v[kDwDpt];
#pragma unroll
      for (int j = 0; j < kDwDpt; ++j) v[j] = acc[j][q];
      st2(part + ((size_t)split * H + h0 + q) * D + d0, D - d0, vec, v);
    }
  }
}

template <typename T>
__global__ void dwa_reduce_kernel(const float* __restrict__ part, T* __restrict__ dWA, int nsplit,
                                  int D, int H) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;   // i = h·D + d
  if (i >= D * H) return;
  // Splits added in order k = 0, 1, ...; sixteen loads in flight at a time.
  float s = 0.f;
  int k = 0;
  for (; k + 16 <= nsplit; k += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) v[u] = part[(size_t)(k + u) * H * D + i];
#pragma unroll
    for (int u = 0; u < 16; ++u) s += v[u];
  }
  for (; k < nsplit; ++k) s += part[(size_t)k * H * D + i];
  const int h = i / D, d = i - h * D;
  st_elem(dWA + (size_t)d * H + h, s);
}

// ---------------------------------------------------------------------------
// dX[t, d] = sum_h dz[h, t] W_A[d, h]: a CTA owns 512 columns (2
// consecutive per thread) and walks tiles of 16 tokens; heads go 16 at a
// time, W_A's slice staged once in shared memory as fp32 [h][d] and held in
// registers (re-staged per tile only when there are more than 16 heads),
// dz's slice of the tile in shared memory.
// ---------------------------------------------------------------------------
constexpr int kDxThreads = 256, kDxDpt = 2, kDxTok = 16, kDxH = 16;
constexpr int kDxCols = kDxThreads * kDxDpt;
constexpr size_t kDxSmem = (size_t)(kDxH * kDxCols + kDxTok * kDxH) * sizeof(float);

template <typename T>
__global__ void __launch_bounds__(kDxThreads, 2)
dx_kernel(const float* __restrict__ dz, const T* __restrict__ WA, T* __restrict__ dX, int N, int D,
          int H, long long tokens, long long ntiles) {
  extern __shared__ float4 dxsm[];
  float* Ws = reinterpret_cast<float*>(dxsm);     // [kDxH][kDxCols]
  float* dzs = Ws + kDxH * kDxCols;                // [kDxTok][kDxH]
  const int dbase = blockIdx.y * kDxCols;
  const int d0 = dbase + threadIdx.x * kDxDpt;
  const bool vec = (D & 1) == 0;
  const int nchunks = (H + kDxH - 1) / kDxH;
  float w[kDxDpt][kDxH];
  auto stage_w = [&](int h0) {
    const int hc = min(kDxH, H - h0);
    for (int i = threadIdx.x; i < kDxH * kDxCols; i += kDxThreads) {
      const int hl = i / kDxCols, d = dbase + (i - hl * kDxCols);
      Ws[i] = (hl < hc && d < D) ? ld_elem(WA + (size_t)d * H + h0 + hl) : 0.f;
    }
  };
  auto load_w = [&]() {
#pragma unroll
    for (int q = 0; q < kDxH; ++q) {
      const float2 v = *reinterpret_cast<const float2*>(Ws + q * kDxCols + threadIdx.x * kDxDpt);
      w[0][q] = v.x; w[1][q] = v.y;
    }
  };
  // dz element (token tl, head h0 + hl) of a tile, zero outside the tile.
  auto ld_dz = [&](long long t0, int h0, int i) {
    const int tl = i % kDxTok, hl = i / kDxTok;
    const int hc = min(kDxH, H - h0);
    const long long t = t0 + tl;
    if (t >= tokens || hl >= hc) return 0.f;
    const long long b = t / N, n = t - b * N;
    return dz[((size_t)b * H + h0 + hl) * N + n];
  };
  static_assert(kDxTok * kDxH == kDxThreads, "one dz element per thread and tile");
  float pre = 0.f;   // the next tile's element (one head chunk only)
  if (nchunks == 1) {
    stage_w(0);
    __syncthreads();
    load_w();
    if (blockIdx.x < ntiles) pre = ld_dz((long long)blockIdx.x * kDxTok, 0, threadIdx.x);
  }
  for (long long tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const long long t0 = tile * kDxTok;
    const int nt = (int)min((long long)kDxTok, tokens - t0);
    float acc[kDxTok][kDxDpt];
#pragma unroll
    for (int t = 0; t < kDxTok; ++t)
#pragma unroll
      for (int j = 0; j < kDxDpt; ++j) acc[t][j] = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const int h0 = c * kDxH;
      __syncthreads();   // the previous tile's (or chunk's) reads are done
      // Thread i holds token i mod 16, head i / 16 of the tile (ld_dz).
      float* slot = dzs + (threadIdx.x % kDxTok) * kDxH + threadIdx.x / kDxTok;
      if (nchunks > 1) {
        stage_w(h0);
        *slot = ld_dz(t0, h0, threadIdx.x);
      } else {
        *slot = pre;
      }
      __syncthreads();
      // Issue the next tile's load now; it completes during the products.
      if (nchunks == 1 && tile + gridDim.x < ntiles)
        pre = ld_dz((tile + gridDim.x) * kDxTok, 0, threadIdx.x);
      if (nchunks > 1) load_w();
      if (d0 < D) {
#pragma unroll
        for (int tl = 0; tl < kDxTok; ++tl) {
          const float4* zr = reinterpret_cast<const float4*>(dzs + tl * kDxH);
#pragma unroll
          for (int q = 0; q < kDxH / 4; ++q) {
            const float4 z = zr[q];
#pragma unroll
            for (int j = 0; j < kDxDpt; ++j) {
              float a = acc[tl][j];
              a = fmaf(w[j][4 * q + 0], z.x, a);
              a = fmaf(w[j][4 * q + 1], z.y, a);
              a = fmaf(w[j][4 * q + 2], z.z, a);
              a = fmaf(w[j][4 * q + 3], z.w, a);
              acc[tl][j] = a;
            }
          }
        }
      }
    }
    if (d0 < D) {
#pragma unroll
      for (int tl = 0; tl < kDxTok; ++tl)
        if (tl < nt) st2(dX + (size_t)(t0 + tl) * D + d0, D - d0, vec, acc[tl]);
    }
  }
}

// ---------------------------------------------------------------------------
// Host launchers (plan's stream).
// ---------------------------------------------------------------------------
cudaError_t setup_backward_kernels(const cat_plan_s* p) {
  cudaError_t e = p->dtype == 1 ? allow_max_smem(dx_kernel<__nv_bfloat16>)
                                : allow_max_smem(dx_kernel<float>);
  const bool tw = !p->twod;
  if (e == cudaSuccess) e = tw ? allow_max_smem(corr_pass_b<true>) : allow_max_smem(corr_pass_b<false>);
  if (e == cudaSuccess) e = allow_max_smem(corr_pass_c);
  if (e == cudaSuccess)
    e = p->dtype == 1 ? (tw ? allow_max_smem(corr_pass_a<__nv_bfloat16, true>)
                            : allow_max_smem(corr_pass_a<__nv_bfloat16, false>))
                      : (tw ? allow_max_smem(corr_pass_a<float, true>)
                            : allow_max_smem(corr_pass_a<float, false>));
  if (e == cudaSuccess && p->dtype == 1) e = setup_dense_mma();
  return e;
}

cudaError_t launch_reverse_scores(const cat_plan_s* p) {
  const int half = (p->N - 1) / 2;
  const long long items = (long long)p->B * p->H * half;
  if (items == 0) return cudaSuccess;
  long long blocks = (items + 255) / 256;
  if (blocks > 8 * (long long)p->sms) blocks = 8 * (long long)p->sms;
  reverse_scores_kernel<<<(int)blocks, 256, 0, p->stream>>>(p->z2, p->N, items);
  return cudaGetLastError();
}

template <typename T, bool TW>
static cudaError_t corr_t(const cat_plan_s* p, const T* G, const T* V) {
  const BwCfg& w = p->bw;
  const int rows = p->B * p->H;
  for (int bh0 = 0; bh0 < rows; bh0 += w.chunk_bh) {
    const int nb = rows - bh0 < w.chunk_bh ? rows - bh0 : w.chunk_bh;
    corr_pass_a<T, TW><<<nb * (w.N1 / w.TA) * w.groupsA, w.threadsA, w.smemA, p->stream>>>(
        G, V, p->bw_scr, p->tw, w.rp2, p->N, w.N1, p->D, p->H, p->dh, p->npair, w.GA, w.groupsA,
        w.TA, w.Q, bh0, p->status);
    corr_pass_b<TW><<<nb * (w.N2 / w.TB), w.threadsB, w.smemB, p->stream>>>(
        p->bw_scr, p->tw, w.rp1, p->N, w.N2, p->npair, w.GB, w.TB, w.Q, p->status);
    corr_pass_c<<<nb * (w.N1 / w.TC), w.threadsC, w.smemC, p->stream>>>(
        p->bw_scr, p->bw_dzs, p->tw, w.rp2, p->N, w.N1, w.TC, w.Q, bh0, p->status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Fast path: its own pass A on dO and on V, fsf_corr_b into the one-signal
// buffer bw_scr ([bhl][k2][n1]), then pass C (in registers for N2 = 32, else
// pass C above with Q = 1).
// With the forward's chunks of 8 rows (N2 = 32) the correlation runs chunks
// of 4 rows alternately on the plan's two internal streams: chunk c uses the
// half c mod 2 of both scratch slots (dO's and V's spectra) and of the
// one-signal buffer y, so two chunks are in flight in the same 64 MB.
// With dV given, each chunk then runs the forward's passes B and C on dO's
// transform, still in its half slot, with the spectrum of z* conjugated
// (that of z* reversed): dV = circ(z*)^T dO without transforming dO a
// second time.  The plan's stream then waits only for the streams'
// correlation work (event ev_front[k] after each chunk's), so that the last
// chunks' dV passes run beside pass C, the softmax backward and dW_A, dX;
// backward_join_dv joins the streams at the end.
static cudaError_t corr_fast_overlapped(const cat_plan_s* p, const void* G, const void* V,
                                        void* dV) {
  const int rows = p->B * p->H;
  const int cb = p->fs.chunk_bh / 2;
  const size_t half = p->scratch_bytes / 4 / sizeof(float2);   // a half slot
  cudaError_t e = cudaEventRecord(p->ev_fork, p->stream);
  for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
    e = cudaStreamWaitEvent(p->side[k], p->ev_fork, 0);
    if (e == cudaSuccess && dV) e = cudaEventRecord(p->ev_front[k], p->side[k]);
  }
  for (int bh0 = 0, c = 0; bh0 < rows && e == cudaSuccess; bh0 += cb, ++c) {
    const int nb = rows - bh0 < cb ? rows - bh0 : cb;
    const int k = c & 1;
    float2* s0 = p->scratch + (size_t)k * half;
    float2* s1 = p->scratch + 2 * half + (size_t)k * half;
    // Each chunk's y at its own rows: pass C runs once for all rows below.
    e = launch_fast_corr(p, G, V, p->bw_scr + (size_t)bh0 * p->N, bh0, nb, p->side[k], s0, s1);
    if (e == cudaSuccess && dV) e = cudaEventRecord(p->ev_front[k], p->side[k]);
    if (e == cudaSuccess && dV) e = launch_fast_bc32(p, s0, dV, bh0, nb, k * cb, p->side[k]);
  }
  for (int k = 0; k < 2; ++k) {
    cudaError_t e2 = cudaEventRecord(p->ev_join[k], p->side[k]);
    if (e2 == cudaSuccess)
      e2 = cudaStreamWaitEvent(p->stream, dV ? p->ev_front[k] : p->ev_join[k], 0);
    if (e == cudaSuccess) e = e2;
  }
  if (e == cudaSuccess) e = launch_fast_corr_c32(p, p->bw_scr, p->bw_dzs, 0, rows, p->stream);
  return e;
}

cudaError_t backward_join_dv(const cat_plan_s* p) {
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < 2 && e == cudaSuccess; ++k) e = cudaStreamWaitEvent(p->stream, p->ev_join[k], 0);
  return e;
}

static bool corr_overlapped(const cat_plan_s* p) {
  return p->bw.fast && p->bw.N2 == 32 && p->fs.chunk_bh >= 2 && p->fs.chunk_bh % 2 == 0;
}

static cudaError_t corr_fast(const cat_plan_s* p, const void* G, const void* V, void* dV) {
  const BwCfg& w = p->bw;
  const int rows = p->B * p->H;
  if (corr_overlapped(p)) return corr_fast_overlapped(p, G, V, dV);
  for (int bh0 = 0; bh0 < rows; bh0 += w.chunk_bh) {
    const int nb = rows - bh0 < w.chunk_bh ? rows - bh0 : w.chunk_bh;
    cudaError_t e = launch_fast_corr(p, G, V, p->bw_scr, bh0, nb, p->stream);
    if (e != cudaSuccess) return e;
    if (w.N2 == 32) {
      e = launch_fast_corr_c32(p, p->bw_scr, p->bw_dzs, bh0, nb, p->stream);
    } else {
      corr_pass_c<<<nb * (w.N1 / w.TC), w.threadsC, w.smemC, p->stream>>>(
          p->bw_scr, p->bw_dzs, p->tw, w.rp2, p->N, w.N1, w.TC, 1, bh0, p->status);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool backward_dv_in_corr(const cat_plan_s* p) {
  const char* e = std::getenv("CAT_BW_DV_CORR");
  return corr_overlapped(p) && !(e && e[0] == '0');
}

cudaError_t launch_backward_dz(const cat_plan_s* p, const void* G, const void* V, void* dV) {
  const int rows = p->B * p->H;
  if (rows == 0) return cudaSuccess;
  if (dV && !backward_dv_in_corr(p)) return cudaErrorInvalidValue;
  // Square lengths with a register transform (N = 8², 14², 16², 32²) take
  // the register correlation kernel; CAT_BW_REG=0 keeps the block passes.
  const char* env = std::getenv("CAT_BW_REG");
  const bool reg = !p->bw.fast && !p->twod && p->path == PATH_SMEM && p->sm.reg_m > 0 &&
                   !(env && std::strcmp(env, "0") == 0);
  if (reg && corr_reg_split_fits(p)) return launch_corr_reg_split(p, G, V);
  const cudaError_t e = p->bw.fast ? corr_fast(p, G, V, dV)
      : reg           ? launch_corr_reg(p, G, V, p->bw_dzs)
      : p->dtype == 1 ? corr_t<__nv_bfloat16, true>(p, (const __nv_bfloat16*)G, (const __nv_bfloat16*)V)
                      : corr_t<float, true>(p, (const float*)G, (const float*)V);
  if (e != cudaSuccess) return e;
  softmax_bw_kernel<<<rows, kSmBwThreads, 0, p->stream>>>(p->zs, p->bw_dzs, p->bw_dz, p->N);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// 2-D circulant attention scores (page "Vision Transformers are Circulant
// Attention Learners"): a = scale · Σ_{c in head} corr2d(Q_c, K_c), the
// correlation passes above without their twiddles over the h x w grid
// (N1 = w, N2 = h), then a stored as the softmax's scores (hi = a, lo = 0).
// ---------------------------------------------------------------------------
__global__ void scores_from_corr_kernel(const float* __restrict__ a, float2* __restrict__ z2,
                                        float* __restrict__ out, float scale, long long count) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
       i += (long long)gridDim.x * blockDim.x) {
    const float v = a[i] * scale;
    z2[i] = make_float2(v, 0.f);
    if (out) out[i] = v;
  }
}

cudaError_t launch_scores2d(const cat_plan_s* p, const void* Q, const void* K, float* out) {
  const int rows = p->B * p->H;
  if (rows == 0) return cudaSuccess;
  cudaError_t e = p->dtype == 1
      ? corr_t<__nv_bfloat16, false>(p, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K)
      : corr_t<float, false>(p, (const float*)Q, (const float*)K);
  if (e != cudaSuccess) return e;
  const long long count = (long long)rows * p->N;
  long long blocks = (count + 255) / 256;
  if (blocks > 8ll * p->sms) blocks = 8ll * p->sms;
  scores_from_corr_kernel<<<(int)blocks, 256, 0, p->stream>>>(p->bw_dzs, p->z2, out,
                                                              1.0f / (float)p->dh, count);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t dense_t(const cat_plan_s* p, const T* X, const T* WA, T* dX, T* dWA) {
  const BwCfg& w = p->bw;
  const long long tokens = (long long)p->B * p->N;
  if (dense_mma_ok(p, X, dX)) {
    const int ns = dwa_mma_splits(p, w.wsplit);
    cudaError_t e = launch_dwa_mma(p, X, p->bw_wpart, ns);
    if (e != cudaSuccess) return e;
    dwa_reduce_kernel<T><<<(p->D * p->H + 255) / 256, 256, 0, p->stream>>>(p->bw_wpart, dWA, ns,
                                                                          p->D, p->H);
    e = cudaGetLastError();
    return e == cudaSuccess ? launch_dx_mma(p, WA, dX) : e;
  }
  const int dchunks = (p->D + kDwThreads * kDwDpt - 1) / (kDwThreads * kDwDpt);
  const int hchunks = (p->H + kDwH - 1) / kDwH;
  const long long tps = (tokens + w.wsplit - 1) / w.wsplit;
  dim3 gw(w.wsplit, dchunks, hchunks);
  if ((p->D & 1) == 0)
    dwa_partial_kernel<T, true><<<gw, kDwThreads, 0, p->stream>>>(X, p->bw_dz, p->bw_wpart, p->N,
                                                                  p->D, p->H, tokens, tps);
  else
    dwa_partial_kernel<T, false><<<gw, kDwThreads, 0, p->stream>>>(X, p->bw_dz, p->bw_wpart, p->N,
                                                                   p->D, p->H, tokens, tps);
  const int dh_items = p->D * p->H;
  dwa_reduce_kernel<T><<<(dh_items + 255) / 256, 256, 0, p->stream>>>(p->bw_wpart, dWA, w.wsplit,
                                                                      p->D, p->H);
  const long long ntiles = (tokens + kDxTok - 1) / kDxTok;
  const int dxc = (p->D + kDxCols - 1) / kDxCols;
  long long gxx = 2ll * p->sms / dxc;
  if (gxx < 1) gxx = 1;
  if (gxx > ntiles) gxx = ntiles;
  dim3 gx((unsigned)gxx, dxc);
  dx_kernel<T><<<gx, kDxThreads, kDxSmem, p->stream>>>(p->bw_dz, WA, dX, p->N, p->D, p->H, tokens,
                                                       ntiles);
  return cudaGetLastError();
}

cudaError_t launch_backward_dense(const cat_plan_s* p, const void* X, const void* WA, void* dX,
                                  void* dWA) {
  if (p->B == 0) return cudaSuccess;
  if (p->dtype == 1)
    return dense_t(p, (const __nv_bfloat16*)X, (const __nv_bfloat16*)WA, (__nv_bfloat16*)dX,
                   (__nv_bfloat16*)dWA);
  return dense_t(p, (const float*)X, (const float*)WA, (float*)dX, (float*)dWA);
}

int backward_wsplit(long long tokens, int D, int H, int sms) {
  const int dchunks = (D + kDwThreads * kDwDpt - 1) / (kDwThreads * kDwDpt);
  const int hchunks = (H + kDwH - 1) / kDwH;
  long long s = 2ll * sms / ((long long)dchunks * hchunks);
  const long long most = (tokens + kDwTok - 1) / kDwTok;
  if (s > most) s = most;
  if (s < 1) s = 1;
  return (int)s;
}

}  // namespace cat
