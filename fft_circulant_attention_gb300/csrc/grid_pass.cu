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
// Inside a CTA, a length-M DFT of S signals held in shared memory (stride
// M + 1, odd, so that column accesses hit distinct banks) is two in-place
// stages: a register DFT-32 over each stride-R subsequence, times
// w_M^{e1·k2}, then a DFT-R over adjacent slots.  With n = e1 + R·e2 and
// k = k2 + 32·k1,
//     X[k2 + 32·k1] = Σ_e1 w_R^{e1·k1} · w_M^{e1·k2} · Σ_e2 w_32^{e2·k2} x[e1 + R·e2],
// so the spectrum lands in the slot order k ↦ k1 + R·k2.  The inverse runs
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

// The M twiddles w_M^m of a CTA (blocks of at least 64 threads, M <= 128:
// at most two a thread), fetched into registers at the start and put in
// shared memory after the CTA's main loads, so that no thread waits on them
// before issuing those.  The plan's table holds w_N^j for N = M², and
// w_M^m = w_N^{M·m}.
template <int R>
struct Twm {
  static constexpr int M = 32 * R;
  float2 v[2];
  __device__ __forceinline__ void fetch(const float2* __restrict__ tw) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int m = threadIdx.x + u * blockDim.x;
      if (m < M) v[u] = __ldg(&tw[(size_t)M * m]);
    }
  }
  __device__ __forceinline__ void put(float2* twm) const {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int m = threadIdx.x + u * blockDim.x;
      if (m < M) twm[m] = v[u];
    }
  }
};

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

// A 16-byte chunk of a token's channels as PV (channel 2j, 2j + 1) pairs.
template <typename T> struct Chunk16;
template <> struct Chunk16<float> {
  static constexpr int PV = 2;
  static __device__ __forceinline__ void unpack(uint4 u, float2* v) {
    v[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    v[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
  static __device__ __forceinline__ uint4 pack(const float2* v) {
    return make_uint4(__float_as_uint(v[0].x), __float_as_uint(v[0].y), __float_as_uint(v[1].x),
                      __float_as_uint(v[1].y));
  }
};
template <> struct Chunk16<__nv_bfloat16> {
  static constexpr int PV = 4;
  static __device__ __forceinline__ float2 word(unsigned int w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ unsigned int bits(float2 v) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<const unsigned int*>(&b);
  }
  static __device__ __forceinline__ void unpack(uint4 u, float2* v) {
    v[0] = word(u.x);
    v[1] = word(u.y);
    v[2] = word(u.z);
    v[3] = word(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float2* v) {
    return make_uint4(bits(v[0]), bits(v[1]), bits(v[2]), bits(v[3]));
  }
};

// Length-M DFT of S signals in shared memory (signal s at buf + s·(M + 1)),
// in place, all threads of the CTA.  Forward: natural order in, slot order
// k1 + R·k2 out.  Inverse (unscaled): slot order in, natural order out.
// Callers synchronise before; the routine ends with a barrier.
template <int R, bool INV>
__device__ __forceinline__ void dft_m(float2* buf, int S, const float2* twm) {
  constexpr int M = 32 * R, LS = M + 1;
  const float rS = 1.0f / (float)S;
  auto stage_a = [&]() {
    for (int t = threadIdx.x; t < S * R; t += blockDim.x) {
      const int e1 = fdiv(t, rS), sig = t - e1 * S;
      float2* s = buf + sig * LS + e1;
      float2 a[32];
      if constexpr (!INV) {
#pragma unroll
        for (int e2 = 0; e2 < 32; ++e2) a[e2] = s[R * e2];
        dft<32, false>(a);
#pragma unroll
        for (int k2 = 0; k2 < 32; ++k2) s[R * k2] = cmul(a[k2], twm[e1 * k2]);
      } else {
#pragma unroll
        for (int k2 = 0; k2 < 32; ++k2) a[k2] = cmulc(s[R * k2], twm[e1 * k2]);
        dft<32, true>(a);
#pragma unroll
        for (int e2 = 0; e2 < 32; ++e2) s[R * e2] = a[e2];
      }
    }
    __syncthreads();
  };
  auto stage_b = [&]() {
    for (int t = threadIdx.x; t < S * 32; t += blockDim.x) {
      const int k2 = fdiv(t, rS), sig = t - k2 * S;
      float2* s = buf + sig * LS + R * k2;
      float2 a[R];
#pragma unroll
      for (int j = 0; j < R; ++j) a[j] = s[j];
      dft_small<R, INV>(a);
#pragma unroll
      for (int j = 0; j < R; ++j) s[j] = a[j];
    }
    __syncthreads();
  };
  if constexpr (!INV) {
    stage_a();
    stage_b();
  } else {
    stage_b();
    stage_a();
  }
}

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

// Scratch rows [y][slot][g] of npair complex values: the M·np values of
// one grid row (or the strided column entries) to and from shared-memory
// signals buf[g·LS + e].  Two pairs (16 bytes) an access when npair is even.
// Load: element e of the signals from src + e·estride + g.
template <int R>
__device__ __forceinline__ void scr_load(float2* buf, int sigoff, const float2* __restrict__ src,
                                         size_t estride, int np) {
  constexpr int M = 32 * R, LS = M + 1;
  if ((np & 1) == 0) {
    const int h2 = np / 2;
    const float r2 = 1.0f / (float)h2;
    batched<8, float4>(
        M * h2,
        [&](int i) {
          const int e = fdiv(i, r2), g2 = i - e * h2;
          return __ldg(reinterpret_cast<const float4*>(src + (size_t)e * estride) + g2);
        },
        [&](int i, float4 v) {
          const int e = fdiv(i, r2), g = 2 * (i - e * h2);
          buf[(sigoff + g) * LS + e] = make_float2(v.x, v.y);
          buf[(sigoff + g + 1) * LS + e] = make_float2(v.z, v.w);
        });
  } else {
    const float r = 1.0f / (float)np;
    batched<16, float2>(
        M * np,
        [&](int i) {
          const int e = fdiv(i, r), g = i - e * np;
          return src[(size_t)e * estride + g];
        },
        [&](int i, float2 v) {
          const int e = fdiv(i, r), g = i - e * np;
          buf[(sigoff + g) * LS + e] = v;
        });
  }
}
template <int R>
__device__ __forceinline__ void scr_store(const float2* buf, float2* __restrict__ dst,
                                          size_t estride, int np) {
  constexpr int M = 32 * R, LS = M + 1;
  if ((np & 1) == 0) {
    const int h2 = np / 2;
    const float r2 = 1.0f / (float)h2;
    for (int i = threadIdx.x; i < M * h2; i += blockDim.x) {
      const int e = fdiv(i, r2), g2 = i - e * h2;
      const float2 a = buf[2 * g2 * LS + e], c = buf[(2 * g2 + 1) * LS + e];
      reinterpret_cast<float4*>(dst + (size_t)e * estride)[g2] = make_float4(a.x, a.y, c.x, c.y);
    }
  } else {
    const float r = 1.0f / (float)np;
    for (int i = threadIdx.x; i < M * np; i += blockDim.x) {
      const int e = fdiv(i, r), g = i - e * np;
      dst[(size_t)e * estride + g] = buf[g * LS + e];
    }
  }
}

// Pass 1: grid row y of (b, h) = bh0 + blockIdx.y, tensor blockIdx.z (Q, K,
// V): the x-DFT of its npair signals into xs[z][bhl][y][slot][g].  vec: the
// head's channels come in whole 16-byte chunks (dh and D multiples of the
// chunk), else pair by pair.
template <typename T, int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_rows_fwd(const T* __restrict__ X0, const T* __restrict__ X1, const T* __restrict__ X2,
            float2* __restrict__ xs, size_t tstride, const float2* __restrict__ tw, int D, int H,
            int dh, int np, int bh0, int vec) {
  constexpr int M = 32 * R, LS = M + 1;
  extern __shared__ float4 smem4[];
  float2* twm = reinterpret_cast<float2*>(smem4);
  float2* buf = twm + M;
  const int y = blockIdx.x, bhl = blockIdx.y, z = blockIdx.z;
  const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
  const T* X = z == 0 ? X0 : (z == 1 ? X1 : X2);
  Twm<R> tv;
  tv.fetch(tw);
  const T* row = X + ((size_t)b * M * M + (size_t)y * M) * D + (size_t)h * dh;
  if (vec) {
    constexpr int E = 16 / (int)sizeof(T), PV = E / 2;
    const int vpr = dh / E;
    const float rv = 1.0f / (float)vpr;
    batched<8, uint4>(
        M * vpr,
        [&](int i) {
          const int x = fdiv(i, rv), j = i - x * vpr;
          return __ldg(reinterpret_cast<const uint4*>(row + (size_t)x * D + j * E));
        },
        [&](int i, uint4 u) {
          const int x = fdiv(i, rv), j = i - x * vpr;
          float2 v[PV];
          Chunk16<T>::unpack(u, v);
#pragma unroll
          for (int k = 0; k < PV; ++k) buf[(j * PV + k) * LS + x] = v[k];
        });
  } else {
    const bool aligned = ((h * dh) % 2) == 0 && (D % 2) == 0;
    const float r = 1.0f / (float)np;
    batched<16, float2>(
        M * np,
        [&](int i) {
          const int x = fdiv(i, r), g = i - x * np;
          return ld_chan_pair(row + (size_t)x * D + 2 * g, 2 * g + 1 < dh, aligned);
        },
        [&](int i, float2 v) {
          const int x = fdiv(i, r), g = i - x * np;
          buf[g * LS + x] = v;
        });
  }
  tv.put(twm);
  __syncthreads();
  dft_m<R, false>(buf, np, twm);
  scr_store<R>(buf, xs + z * tstride + ((size_t)bhl * M + y) * M * np, np, np);
}

// Pass 2: column slot kx = blockIdx.x of (b, h) row bhl = blockIdx.y: the
// y-DFT of Q's and K's npair signals, Σ_g Q̂_g·conj(K̂_g) in the order g = 0,
// 1, …, and its inverse y-DFT into tsc[bhl][y][kx].
template <int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_cols_scores(const float2* __restrict__ qs, const float2* __restrict__ ks,
               float2* __restrict__ tsc, const float2* __restrict__ tw, int np) {
  constexpr int M = 32 * R, LS = M + 1;
  extern __shared__ float4 smem4[];
  float2* twm = reinterpret_cast<float2*>(smem4);
  float2* buf = twm + M;               // Q's signals, then K's
  float2* sum = buf + 2 * np * LS;
  const int kx = blockIdx.x, bhl = blockIdx.y;
  Twm<R> tv;
  tv.fetch(tw);
  const size_t base = (size_t)bhl * M * M * np + (size_t)kx * np;
  scr_load<R>(buf, 0, qs + base, (size_t)M * np, np);
  scr_load<R>(buf, np, ks + base, (size_t)M * np, np);
  tv.put(twm);
  __syncthreads();
  dft_m<R, false>(buf, 2 * np, twm);
  for (int s = threadIdx.x; s < M; s += blockDim.x) {
    float2 acc = make_float2(0.f, 0.f);
    for (int g = 0; g < np; ++g) {
      const float2 q = buf[g * LS + s], k = buf[(np + g) * LS + s];
      acc.x = fmaf(q.x, k.x, fmaf(q.y, k.y, acc.x));
      acc.y = fmaf(q.y, k.x, fmaf(-q.x, k.y, acc.y));
    }
    sum[s] = acc;
  }
  __syncthreads();
  dft_m<R, true>(sum, 1, twm);
  float2* dst = tsc + (size_t)bhl * M * M + kx;
  for (int y = threadIdx.x; y < M; y += blockDim.x) dst[(size_t)y * M] = sum[y];
}

// Pass 3: grid rows y0 .. y0 + 7 (one warp each) of (b, h) row bhl: the
// inverse x-DFT gives a (× scale = 1/(dh·N)), written to aout[bh][y·M + x]
// when given; with esp, the row's max m and sum s of exp(a − m) go to
// stats[bhl][y] and the x-DFT of exp(a − m) to esp[bhl][y][slot].
template <int R>
__global__ void __launch_bounds__(32 * kGpRowsPerCta)
gp_rows_scores(const float2* __restrict__ tsc, float2* __restrict__ esp,
               float2* __restrict__ stats, float* __restrict__ aout,
               const float2* __restrict__ tw, int bh0, float scale) {
  constexpr int M = 32 * R, LS = M + 1, RB = kGpRowsPerCta;
  extern __shared__ float4 smem4[];
  float2* twm = reinterpret_cast<float2*>(smem4);
  float2* buf = twm + M;
  const int bhl = blockIdx.y, bh = bh0 + bhl, y0 = blockIdx.x * RB;
  Twm<R> tv;
  tv.fetch(tw);
  const float rM = 1.0f / (float)M;
  batched<4, float2>(
      RB * M, [&](int i) { return tsc[((size_t)bhl * M + y0) * M + i]; },
      [&](int i, float2 v) {
        const int r = fdiv(i, rM), s = i - r * M;
        buf[r * LS + s] = v;
      });
  tv.put(twm);
  __syncthreads();
  dft_m<R, true>(buf, RB, twm);
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
  dft_m<R, false>(buf, RB, twm);
  for (int i = threadIdx.x; i < RB * M; i += blockDim.x) {
    const int r = fdiv(i, rM), sl = i - r * M;
    esp[((size_t)bhl * M + y0 + r) * M + sl] = buf[r * LS + sl];
  }
}

// Pass 4: column slot kx of (b, h) row bhl.  The softmax's scale of grid
// row y is c_y = exp(m_y − m) / Σ_y' s_y'·exp(m_y' − m), m = max_y m_y, the
// same in every CTA of the row; the column of σ's x-spectrum times c_y / N
// is y-transformed together with V's npair columns, V's spectra are
// multiplied by it and inverse y-transformed back into vs.
template <int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_cols_conv(float2* __restrict__ vs, const float2* __restrict__ esp,
             const float2* __restrict__ stats, const float2* __restrict__ tw, int np,
             float invN) {
  constexpr int M = 32 * R, LS = M + 1;
  extern __shared__ float4 smem4[];
  float2* twm = reinterpret_cast<float2*>(smem4);
  float2* sig = twm + M;               // σ's column, then V's npair columns
  float2* vb = sig + LS;
  float* cy = reinterpret_cast<float*>(vb + np * LS);
  const int kx = blockIdx.x, bhl = blockIdx.y;
  Twm<R> tv;
  tv.fetch(tw);
  // σ's column and (warp 0) the row statistics, fetched with the rest.
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
  const size_t base = (size_t)bhl * M * M * np + (size_t)kx * np;
  scr_load<R>(vb, 0, vs + base, (size_t)M * np, np);
  tv.put(twm);
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
    if (y < M) sig[y] = cscale(ev[u], cy[y]);
  }
  __syncthreads();
  dft_m<R, false>(sig, np + 1, twm);
  const float rM = 1.0f / (float)M;
  for (int i = threadIdx.x; i < M * np; i += blockDim.x) {
    const int g = fdiv(i, rM), s = i - g * M;
    vb[g * LS + s] = cmul(vb[g * LS + s], sig[s]);
  }
  __syncthreads();
  dft_m<R, true>(vb, np, twm);
  scr_store<R>(vb, vs + base, (size_t)M * np, np);
}

// Pass 5: grid row y of (b, h) row bhl: the inverse x-DFT of V's npair
// signals, stored as O's channels (2g, 2g + 1); vec as in pass 1.
template <typename T, int R>
__global__ void __launch_bounds__(kGpMaxThreads)
gp_rows_out(const float2* __restrict__ vs, T* __restrict__ O, const float2* __restrict__ tw,
            int D, int H, int dh, int np, int bh0, int vec) {
  constexpr int M = 32 * R, LS = M + 1;
  extern __shared__ float4 smem4[];
  float2* twm = reinterpret_cast<float2*>(smem4);
  float2* buf = twm + M;
  const int y = blockIdx.x, bhl = blockIdx.y;
  const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
  Twm<R> tv;
  tv.fetch(tw);
  scr_load<R>(buf, 0, vs + ((size_t)bhl * M + y) * M * np, np, np);
  tv.put(twm);
  __syncthreads();
  dft_m<R, true>(buf, np, twm);
  T* row = O + ((size_t)b * M * M + (size_t)y * M) * D + (size_t)h * dh;
  if (vec) {
    constexpr int E = 16 / (int)sizeof(T), PV = E / 2;
    const int vpr = dh / E;
    const float rv = 1.0f / (float)vpr;
    for (int i = threadIdx.x; i < M * vpr; i += blockDim.x) {
      const int x = fdiv(i, rv), j = i - x * vpr;
      float2 v[PV];
#pragma unroll
      for (int k = 0; k < PV; ++k) v[k] = buf[(j * PV + k) * LS + x];
      *reinterpret_cast<uint4*>(row + (size_t)x * D + j * E) = Chunk16<T>::pack(v);
    }
  } else {
    const bool aligned = ((h * dh) % 2) == 0 && (D % 2) == 0;
    const float r = 1.0f / (float)np;
    for (int i = threadIdx.x; i < M * np; i += blockDim.x) {
      const int x = fdiv(i, r), g = i - x * np;
      st_chan_pair(row + (size_t)x * D + 2 * g, buf[g * LS + x], 2 * g + 1 < dh, aligned);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.

namespace {

int gp_threads(int tasks) {
  int t = (tasks + 31) / 32 * 32;
  return t < 64 ? 64 : (t > kGpMaxThreads ? kGpMaxThreads : t);
}

size_t smem_rows(int M, int np) { return ((size_t)M + (size_t)np * (M + 1)) * sizeof(float2); }
size_t smem_cols_scores(int M, int np) {
  return ((size_t)M + (size_t)(2 * np + 1) * (M + 1)) * sizeof(float2);
}
size_t smem_rows_scores(int M) {
  return ((size_t)M + (size_t)kGpRowsPerCta * (M + 1)) * sizeof(float2);
}
size_t smem_cols_conv(int M, int np) {
  return ((size_t)M + (size_t)(np + 1) * (M + 1)) * sizeof(float2) + (size_t)M * sizeof(float);
}

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

struct Bufs {
  float2* xs;      // [3][chunk][M][M][np]
  size_t tstride;  // chunk·M²·np
  float2* tsc;     // [chunk][M][M]
  float2* esp;     // [chunk][M][M]
  float2* stats;   // [chunk][M]
};

Bufs bufs(const cat_plan_s* p) {
  const int M = p->gp.M, np = p->npair, c = p->gp.chunk;
  Bufs b;
  b.xs = p->scratch;
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
  // Whole 16-byte chunks of channels per head (the API's 16-byte aligned
  // tensors then give aligned chunks).
  const int E = 16 / (int)sizeof(T);
  const int vec = (p->dh % E == 0 && p->D % E == 0) ? 1 : 0;
  gp_rows_fwd<T, R><<<dim3(M, nb, ntens), gp_threads(np * R), smem_rows(M, np), st>>>(
      Q, K, V, bf.xs, bf.tstride, p->tw, p->D, p->H, p->dh, np, bh0, vec);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gp_cols_scores<R><<<dim3(M, nb), gp_threads(2 * np * R), smem_cols_scores(M, np), st>>>(
      bf.xs, bf.xs + bf.tstride, bf.tsc, p->tw, np);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const float scale = 1.0f / ((float)p->dh * (float)(M * M));
  gp_rows_scores<R><<<dim3(M / kGpRowsPerCta, nb), 32 * kGpRowsPerCta, smem_rows_scores(M), st>>>(
      bf.tsc, fwd ? bf.esp : nullptr, bf.stats, aout, p->tw, bh0, scale);
  if ((e = cudaGetLastError()) != cudaSuccess || !fwd) return e;
  gp_cols_conv<R><<<dim3(M, nb), gp_threads((np + 1) * R), smem_cols_conv(M, np), st>>>(
      bf.xs + 2 * bf.tstride, bf.esp, bf.stats, p->tw, np, 1.0f / (float)(M * M));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gp_rows_out<T, R><<<dim3(M, nb), gp_threads(np * R), smem_rows(M, np), st>>>(
      bf.xs + 2 * bf.tstride, O, p->tw, p->D, p->H, p->dh, np, bh0, vec);
  return cudaGetLastError();
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
  g.scratch_bytes = (size_t)g.chunk * one;
  return CAT_OK;
}

cudaError_t setup_grid_pass(const cat_plan_s* p) {
  cudaError_t e = p->dtype == 1 ? setup_r<__nv_bfloat16, 2>() : setup_r<float, 2>();
  if (e == cudaSuccess) e = p->dtype == 1 ? setup_r<__nv_bfloat16, 3>() : setup_r<float, 3>();
  if (e == cudaSuccess) e = p->dtype == 1 ? setup_r<__nv_bfloat16, 4>() : setup_r<float, 4>();
  return e;
}

cudaError_t launch_grid_pass(const cat_plan_s* p, const void* Q, const void* K, const void* V,
                             void* O, float* aout) {
  if (p->B == 0) return cudaSuccess;
  return p->dtype == 1 ? run_all<__nv_bfloat16>(p, Q, K, V, O, aout)
                       : run_all<float>(p, Q, K, V, O, aout);
}

}  // namespace cat
