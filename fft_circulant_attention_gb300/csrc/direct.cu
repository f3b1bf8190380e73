// Direct ("gather") circulant product for short sequences: the plain
// O(N²·dh) evaluation of the CAT output, no transforms.  The notes page
// "CAT: Circular-Convolutional Attention for Sub-Quadratic Transformers"
// reports (section 局限与展望, limitations) that at N = 256 its FFT
// implementation's overhead cancels the theoretical gain and that a
// gather-based O(N²) version ran about 10 % faster than standard attention;
// this is that gather-based evaluation, for the lengths where it is the
// faster one here.  Per (b, h), with circ(z*)[i, j] = z*[(i - j) mod N]
// (section 关键设计, circulant attention matrix construction):
//     O[b, i, c] = sum_j z*[b, h, (i - j) mod N] · V[b, j, c],  c in head h.
//
// One CTA per (row tile, b·H + h).  It computes the row's softmax statistics
// itself (from the scores of the score kernel, or — fused, for small N·D —
// from X and W_A directly, so that the whole forward is one launch), writes
// z* into shared memory padded on both sides so that every weight index
// (i - j) is a plain offset, and then streams V's rows through shared memory
// in chunks of kDirJC.  Thread (rg, cg) owns rows i0 .. i0 + TR - 1 and four
// columns: for TR consecutive j it needs the 2·TR - 1 weights
// z*[i0 - j .. i0 - j + TR - 1 + TR - 1], loaded once into registers, so a
// block of TR j costs 2·TR - 1 weight loads, TR four-wide loads of V and
// TR·TR·4 FMAs.  All arithmetic is fp32; each output is one fp32 sum over j
// in ascending order.
#include <cuda_bf16.h>

#include "cat_internal.h"
#include "elem.cuh"

namespace cat {

constexpr int kDirJC = 64;   // rows of V staged per chunk
constexpr int kDirTC = 4;    // output columns per thread

// Four consecutive storage elements as fp32 (8-byte aligned for bf16,
// 16-byte for fp32).
__device__ __forceinline__ float4 ld4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<unsigned int*>(&lo);
  u.y = *reinterpret_cast<unsigned int*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// Shared-memory layout (floats) of a CTA: zz [L] z* padded, zhl [2N] the
// row's scores (hi, lo) when fused, wa [D] W_A's column h when fused,
// vs [kDirJC][dh] the staged V chunk, red [32].
struct DirLayout {
  int L, zz, zhl, wa, vs, red, total;
  __host__ __device__ DirLayout(int N, int D, int dh, int R, bool fused) {
    L = 2 * N + kDirJC + R;
    zz = 0;
    zhl = (L + 3) & ~3;
    wa = zhl + (fused ? 2 * N : 0);
    vs = (wa + (fused ? D : 0) + 3) & ~3;
    red = vs + kDirJC * dh;
    total = red + 32;
  }
};

size_t direct_smem(int N, int D, int dh, int R, bool fused) {
  return (size_t)DirLayout(N, D, dh, R, fused).total * sizeof(float);
}

// The row's score z[n] = sum_d X[b, n, d] W_A[d, h] as a double-float: runs
// of 16 products summed by fp32 FMA into a fresh register, the run sums
// combined by TwoSum (as the score kernels do).
template <typename T>
__device__ __forceinline__ float2 row_score(const T* __restrict__ xrow, const float* wa, int D) {
  float hi = 0.f, lo = 0.f;
  for (int d0 = 0; d0 < D; d0 += 16) {
    float part = 0.f;
    const int d1 = min(D, d0 + 16);
    for (int d = d0; d < d1; d += 4) {
      const float4 x = ld4(xrow + d);
      part = fmaf(x.x, wa[d], part);
      part = fmaf(x.y, wa[d + 1], part);
      part = fmaf(x.z, wa[d + 2], part);
      part = fmaf(x.w, wa[d + 3], part);
    }
    two_sum_acc(hi, lo, part);
  }
  return make_float2(hi, lo);
}

template <typename T, int TR, bool FUSED>
__global__ void __launch_bounds__(512)
direct_kernel(const T* __restrict__ X, const T* __restrict__ WA, const float2* __restrict__ z2,
              const T* __restrict__ V, T* __restrict__ O, int N, int D, int H, int R) {
  extern __shared__ float4 dsm4[];
  float* sm = reinterpret_cast<float*>(dsm4);
  const int dh = D / H, ncg = dh / kDirTC;
  const DirLayout lay(N, D, dh, R, FUSED);
  float* zz = sm + lay.zz;
  float2* zhl = reinterpret_cast<float2*>(sm + lay.zhl);
  float* wa = sm + lay.wa;
  float4* vs4 = reinterpret_cast<float4*>(sm + lay.vs);
  float* red = sm + lay.red;
  const int nt = blockDim.x, tid = threadIdx.x;
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H;

  // Scores of the row (fused: from X and W_A), then m = max z and
  // S = sum exp(z - m).
  if (FUSED) {
    for (int d = tid; d < D; d += nt) wa[d] = ld_elem(WA + (size_t)d * H + h);
    __syncthreads();
    for (int n = tid; n < N; n += nt) zhl[n] = row_score(X + ((size_t)b * N + n) * D, wa, D);
    __syncthreads();
  }
  const float2* zrow = FUSED ? zhl : z2 + (size_t)bh * N;
  float m = -INFINITY;
  for (int n = tid; n < N; n += nt) m = fmaxf(m, zrow[n].x);
  m = block_reduce<true>(m, red);
  float s = 0.f;
  for (int n = tid; n < N; n += nt) s += exp_shifted(zrow[n], m);
  s = block_reduce<false>(s, red);
  const float inv = 1.0f / s;
  // zz[x] = z*[(x - off) mod N] for x < L, off = N + kDirJC: every weight
  // index off + i - j below falls in [0, L).
  const int off = N + kDirJC;
  for (int x = tid; x < lay.L; x += nt) {
    int n = (x - off) % N;
    if (n < 0) n += N;
    zz[x] = exp_shifted(zrow[n], m) * inv;
  }

  const int cg = tid % ncg, rg = tid / ncg;
  const int i0 = blockIdx.x * R + rg * TR;
  float acc[TR][kDirTC];
#pragma unroll
  for (int r = 0; r < TR; ++r)
#pragma unroll
    for (int c = 0; c < kDirTC; ++c) acc[r][c] = 0.f;
  const T* vbase = V + (size_t)b * N * D + h * dh;
  for (int j0 = 0; j0 < N; j0 += kDirJC) {
    __syncthreads();   // z* written; the previous chunk consumed
    for (int q = tid; q < kDirJC * ncg; q += nt) {
      const int jr = q / ncg, c4 = q - jr * ncg;
      const int j = j0 + jr;
      vs4[q] = j < N ? ld4(vbase + (size_t)j * D + kDirTC * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll 1
    for (int jj0 = 0; jj0 < kDirJC; jj0 += TR) {
      const float* src = zz + off + i0 - j0 - jj0 - (TR - 1);
      float e[2 * TR - 1];
#pragma unroll
      for (int k = 0; k < 2 * TR - 1; ++k) e[k] = src[k];
#pragma unroll
      for (int jj = 0; jj < TR; ++jj) {
        const float4 v = vs4[(jj0 + jj) * ncg + cg];
#pragma unroll
        for (int r = 0; r < TR; ++r) {
          const float w = e[r - jj + TR - 1];
          acc[r][0] = fmaf(w, v.x, acc[r][0]);
          acc[r][1] = fmaf(w, v.y, acc[r][1]);
          acc[r][2] = fmaf(w, v.z, acc[r][2]);
          acc[r][3] = fmaf(w, v.w, acc[r][3]);
        }
      }
    }
  }
  T* obase = O + (size_t)b * N * D + h * dh + kDirTC * cg;
#pragma unroll
  for (int r = 0; r < TR; ++r) {
    const int i = i0 + r;
    if (i < N) st4(obase + (size_t)i * D, acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
}

template <typename T, int TR, bool FUSED>
static cudaError_t run_direct(const cat_plan_s* p, const void* X, const void* WA, const void* V,
                              void* O, bool setup) {
  auto k = direct_kernel<T, TR, FUSED>;
  if (setup) return allow_max_smem(k);
  const DirectCfg& c = p->dir;
  dim3 grid((p->N + c.R - 1) / c.R, p->B * p->H);
  k<<<grid, c.threads, c.smem, p->stream>>>((const T*)X, (const T*)WA, p->z2, (const T*)V, (T*)O,
                                            p->N, p->D, p->H, c.R);
  return cudaGetLastError();
}

template <typename T, bool FUSED>
static cudaError_t direct_tr(const cat_plan_s* p, const void* X, const void* WA, const void* V,
                             void* O, bool setup) {
  if (setup) {
    cudaError_t e = run_direct<T, 2, FUSED>(p, X, WA, V, O, true);
    if (e == cudaSuccess) e = run_direct<T, 4, FUSED>(p, X, WA, V, O, true);
    if (e == cudaSuccess) e = run_direct<T, 8, FUSED>(p, X, WA, V, O, true);
    return e;
  }
  switch (p->dir.TR) {
    case 2: return run_direct<T, 2, FUSED>(p, X, WA, V, O, false);
    case 4: return run_direct<T, 4, FUSED>(p, X, WA, V, O, false);
    default: return run_direct<T, 8, FUSED>(p, X, WA, V, O, false);
  }
}

template <typename T>
static cudaError_t direct_t(const cat_plan_s* p, const void* X, const void* WA, const void* V,
                            void* O, bool fused, bool setup) {
  if (setup) {
    cudaError_t e = direct_tr<T, false>(p, X, WA, V, O, true);
    return e == cudaSuccess ? direct_tr<T, true>(p, X, WA, V, O, true) : e;
  }
  return fused ? direct_tr<T, true>(p, X, WA, V, O, false)
               : direct_tr<T, false>(p, X, WA, V, O, false);
}

cudaError_t setup_direct_kernels(const cat_plan_s* p) {
  return p->dtype == 1 ? direct_t<__nv_bfloat16>(p, nullptr, nullptr, nullptr, nullptr, false, true)
                       : direct_t<float>(p, nullptr, nullptr, nullptr, nullptr, false, true);
}

cudaError_t launch_direct(const cat_plan_s* p, const void* X, const void* WA, const void* V,
                          void* O, bool fused) {
  return p->dtype == 1 ? direct_t<__nv_bfloat16>(p, X, WA, V, O, fused, false)
                       : direct_t<float>(p, X, WA, V, O, fused, false);
}

}  // namespace cat
