// Score projection and softmax over tokens — the "circulant attention matrix
// construction" design of the notes page "CAT: Circular-Convolutional
// Attention for Sub-Quadratic Transformers" (section 关键设计):
//     z[b, h, n] = sum_d X[b, n, d] · W_A[d, h]
//     z*[b, h, :] = softmax over the N tokens of z[b, h, :]
// plus, for the shared-memory path, the spectrum of z* (the "FFT
// acceleration" design) fused into the softmax kernel.
#include <cuda_bf16.h>

#include "cat_internal.h"
#include "elem.cuh"

namespace cat {

constexpr int kScoreThreads = 128;
constexpr int kScoreTokPerThread = 2;
constexpr int kScoreTokPerCta = kScoreThreads * kScoreTokPerThread;
constexpr int kScoreMaxHeads = 16;
constexpr int kScoreSmemBudget = 200 << 10;

}  // namespace cat

// Heads per pass over X: as many as 16, limited by W_A's fp32 slice
// ([D][HP], HP = heads rounded up to 4) fitting the shared-memory budget.
int score_heads_per_pass(int D) {
  int hp = (cat::kScoreSmemBudget / (4 * D)) / 4 * 4;
  if (hp < 1) hp = 1;
  return hp < cat::kScoreMaxHeads ? hp : cat::kScoreMaxHeads;
}

namespace cat {

// 16-byte vector of storage elements and its widening to fp32.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int n = 4;
  static __device__ __forceinline__ void load(const float* p, float* out) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int n = 8;
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* out) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    unsigned int w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// Adds p to the double-float accumulator (hi, lo): hi + p is split exactly
// into its rounded sum and rounding error (Knuth's TwoSum), the error joins
// lo.
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float p) {
  float s = hi + p;
  float bp = s - hi;
  float err = (hi - (s - bp)) + (p - bp);
  hi = s;
  lo += err;
}

// One pass over X computes HT heads [h0, h0 + HT) for kScoreTokPerCta
// tokens of one batch.  W_A's HT columns sit in shared memory as fp32
// [D][HP] (HP = HT rounded up to 4); every lane of a warp reads the same
// W_A row at the same time (a broadcast).  Each thread owns two tokens and
// walks their rows in 16-byte vectors when the layout allows (VEC), else
// element by element.
// Accuracy: the products of each run of kChunk consecutive d are summed by
// fp32 FMA into a fresh register; the chunk sums are combined with TwoSum
// into a double-float (hi, lo), so the result carries no rounding from the
// large running total.  z is stored as the pair (hi, lo).
constexpr int kChunk = 16;

template <typename T, int HT, bool VEC>
__global__ void __launch_bounds__(kScoreThreads)
score_kernel(const T* __restrict__ X, const T* __restrict__ WA, float2* __restrict__ z,
             int N, int D, int H, int h0) {
  constexpr int HP = (HT + 3) & ~3;
  constexpr int TP = kScoreTokPerThread;
  extern __shared__ float4 ws4[];
  float* ws = reinterpret_cast<float*>(ws4);
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < D * HP; i += blockDim.x) {
    int d = i / HP, h = i - d * HP;
    ws[i] = (h < HT) ? ld_elem(WA + (size_t)d * H + h0 + h) : 0.f;
  }
  __syncthreads();
  const int nbase = blockIdx.x * kScoreTokPerCta + threadIdx.x;
  int nn[TP];
  bool ok[TP];
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    nn[t] = nbase + t * kScoreThreads;
    ok[t] = nn[t] < N;
  }
  float hi[TP][HT], lo[TP][HT];
#pragma unroll
  for (int t = 0; t < TP; ++t)
#pragma unroll
    for (int h = 0; h < HT; ++h) hi[t][h] = lo[t][h] = 0.f;

  const T* xr[TP];
#pragma unroll
  for (int t = 0; t < TP; ++t) xr[t] = X + ((size_t)b * N + (ok[t] ? nn[t] : 0)) * D;

  constexpr int V = VEC ? Vec16<T>::n : 1;
  for (int c0 = 0; c0 < D; c0 += kChunk) {
    const int c1 = min(D, c0 + kChunk);
    float part[TP][HT];
#pragma unroll
    for (int t = 0; t < TP; ++t)
#pragma unroll
      for (int h = 0; h < HT; ++h) part[t][h] = 0.f;
    for (int d0 = c0; d0 < c1; d0 += V) {
      float xv[TP][V];
#pragma unroll
      for (int t = 0; t < TP; ++t) {
        if (VEC) Vec16<T>::load(xr[t] + d0, xv[t]);
        else xv[t][0] = ld_elem(xr[t] + d0);
      }
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const float4* wrow = ws4 + (size_t)(d0 + j) * (HP / 4);
#pragma unroll
        for (int q = 0; q < HP / 4; ++q) {
          float4 w = wrow[q];
          float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (q * 4 + e < HT) {
#pragma unroll
              for (int t = 0; t < TP; ++t)
                part[t][q * 4 + e] = fmaf(xv[t][j], wv[e], part[t][q * 4 + e]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TP; ++t)
#pragma unroll
      for (int h = 0; h < HT; ++h) two_sum_acc(hi[t][h], lo[t][h], part[t][h]);
  }
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    if (ok[t]) {
#pragma unroll
      for (int h = 0; h < HT; ++h)
        z[((size_t)b * H + h0 + h) * N + nn[t]] = make_float2(hi[t][h], lo[t][h]);
    }
  }
}

template <typename T>
static bool score_vec_ok(const cat_plan_s* p, const void* X) {
  const int V = 16 / (int)sizeof(T);
  return (p->D % V) == 0 && ((uintptr_t)X % 16) == 0;
}

template <typename T, int HT, bool VEC>
static cudaError_t run_score(const cat_plan_s* p, const T* X, const T* WA, int h0, bool setup) {
  constexpr int HP = (HT + 3) & ~3;
  size_t smem = (size_t)HP * p->D * sizeof(float);
  auto k = score_kernel<T, HT, VEC>;
  if (setup) return allow_max_smem(k);
  dim3 grid((p->N + kScoreTokPerCta - 1) / kScoreTokPerCta, p->B);
  k<<<grid, kScoreThreads, smem, p->stream>>>(X, WA, p->z2, p->N, p->D, p->H, h0);
  return cudaGetLastError();
}

template <typename T, bool VEC>
static cudaError_t score_heads(const cat_plan_s* p, const T* X, const T* WA, bool setup) {
  const int hpp = score_heads_per_pass(p->D);
  for (int h0 = 0; h0 < p->H; h0 += hpp) {
    int ht = p->H - h0 < hpp ? p->H - h0 : hpp;
    cudaError_t e;
    switch (ht) {
#define CAT_HT(n) case n: e = run_score<T, n, VEC>(p, X, WA, h0, setup); break;
      CAT_HT(1) CAT_HT(2) CAT_HT(3) CAT_HT(4) CAT_HT(5) CAT_HT(6) CAT_HT(7) CAT_HT(8)
      CAT_HT(9) CAT_HT(10) CAT_HT(11) CAT_HT(12) CAT_HT(13) CAT_HT(14) CAT_HT(15) CAT_HT(16)
#undef CAT_HT
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T>
static cudaError_t score_dispatch(const cat_plan_s* p, const T* X, const T* WA, bool setup) {
  if (setup) {
    cudaError_t e = score_heads<T, true>(p, X, WA, true);
    if (e != cudaSuccess) return e;
    return score_heads<T, false>(p, X, WA, true);
  }
  if (score_vec_ok<T>(p, X)) return score_heads<T, true>(p, X, WA, false);
  return score_heads<T, false>(p, X, WA, false);
}

cudaError_t launch_score(const cat_plan_s* p, const void* X, const void* WA) {
  if (p->B == 0) return cudaSuccess;
  if (p->dtype == 1)
    return score_dispatch(p, (const __nv_bfloat16*)X, (const __nv_bfloat16*)WA, false);
  return score_dispatch(p, (const float*)X, (const float*)WA, false);
}

// exp(z - m) for a score held as the double-float (hi, lo): the difference
// hi - m is split exactly (TwoSum) and its rounding error, plus lo, enters
// as the first-order factor (1 + delta).
__device__ __forceinline__ float exp_shifted(float2 zhl, float m) {
  float s = zhl.x - m;
  float bp = s - zhl.x;
  float err = (zhl.x - (s - bp)) + (-m - bp);
  float e = expf(s);
  return fmaf(e, err + zhl.y, e);
}

// Softmax over the N tokens of each (b, h) row, one CTA per row, streaming
// through global memory: m = max of the scores, S = sum of exp(z - m), then
// z* = exp(z - m) / S written to zs.
__global__ void __launch_bounds__(1024)
softmax_kernel(const float2* __restrict__ z, float* __restrict__ zs, int N) {
  __shared__ float red[32];
  const float2* row = z + (size_t)blockIdx.x * N;
  float* out = zs + (size_t)blockIdx.x * N;
  float m = -INFINITY;
  for (int n = threadIdx.x; n < N; n += blockDim.x) m = fmaxf(m, row[n].x);
  m = block_reduce<true>(m, red);
  float s = 0.f;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float e = exp_shifted(row[n], m);
    out[n] = e;
    s += e;
  }
  s = block_reduce<false>(s, red);
  const float inv = 1.0f / s;
  for (int n = threadIdx.x; n < N; n += blockDim.x) out[n] *= inv;
}

cudaError_t launch_softmax(const cat_plan_s* p) {
  int rows = p->B * p->H;
  if (rows == 0) return cudaSuccess;
  softmax_kernel<<<rows, 1024, 0, p->stream>>>(p->z2, p->zs, p->N);
  return cudaGetLastError();
}

// Softmax of one (b, h) row held in shared memory, then its spectrum:
// zf[k] = (1/N) sum_n z*[n] exp(-2πi kn/N).  One CTA per row; N <= 16384.
// z* is also written to zs.
__global__ void __launch_bounds__(1024)
softmax_spectrum_kernel(const float2* __restrict__ z, float* __restrict__ zs,
                        float2* __restrict__ zf, RadixPlan rp, const float2* __restrict__ W,
                        unsigned int* status) {
  extern __shared__ float2 sbuf[];
  __shared__ float red[32];
  const int N = rp.L;
  if (N > vals_capacity(rp) * (int)blockDim.x) {
    report(status, 0x101);
    return;
  }
  const float2* row = z + (size_t)blockIdx.x * N;
  float m = -INFINITY;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float2 v = row[n];
    sbuf[n] = v;
    m = fmaxf(m, v.x);
  }
  m = block_reduce<true>(m, red);
  float s = 0.f;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float e = exp_shifted(sbuf[n], m);
    sbuf[n].x = e;
    s += e;
  }
  s = block_reduce<false>(s, red);
  const float inv = 1.0f / s;
  float* out = zs + (size_t)blockIdx.x * N;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float v = sbuf[n].x * inv;
    out[n] = v;
    sbuf[n] = make_float2(v, 0.f);
  }
  __syncthreads();
  block_fft<false>(sbuf, rp, 1, N, W, 1);
  const float invN = 1.0f / (float)N;
  float2* spec = zf + (size_t)blockIdx.x * N;
  for (int k = threadIdx.x; k < N; k += blockDim.x) spec[k] = cscale(sbuf[k], invN);
}

cudaError_t setup_score_kernels(const cat_plan_s* p) {
  cudaError_t e = p->dtype == 1
      ? score_dispatch<__nv_bfloat16>(p, nullptr, nullptr, true)
      : score_dispatch<float>(p, nullptr, nullptr, true);
  if (e != cudaSuccess) return e;
  if (p->path == PATH_SMEM) e = allow_max_smem(softmax_spectrum_kernel);
  return e;
}

cudaError_t launch_softmax_spectrum(const cat_plan_s* p) {
  int rows = p->B * p->H;
  if (rows == 0) return cudaSuccess;
  softmax_spectrum_kernel<<<rows, p->sm.spec_threads, p->sm.spec_smem, p->stream>>>(
      p->z2, p->zs, p->zf, p->rpN, p->tw, p->status);
  return cudaGetLastError();
}

}  // namespace cat
