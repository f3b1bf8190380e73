// Fast long-sequence circulant product for head width 64 (32 packed column
// pairs per head) and N = 512·N2, N2 in {32, 64, 128, 256}: the "FFT
// acceleration" design of the notes page "CAT: Circular-Convolutional
// Attention for Sub-Quadratic Transformers" (section 关键设计),
//     O_h[:, c] = IFFT( FFT(z*_h) ⊙ FFT(V_h[:, c]) ),
// by the four-step split N = N1·N2 (N1 = 512), n = n1 + N1·n2,
// k = N2·k1 + k2, in three passes over an L2-resident scratch:
//   A (per n1): DFT over n2 of the head's 32 pairs, times w_N^{n1 k2};
//   B (per k2): DFT over n1, product with FFT(z*)/N, inverse DFT over k1,
//               times w_N^{-n1 k2};
//   C (per n1): inverse DFT over k2, store the output rows n1 + N1·n2.
// A warp's 32 lanes are the head's 32 pairs, so every global access of V,
// O and the scratch is a contiguous run of the head's row.
//
// Within a pass each thread holds 32 values in registers and the transform
// is a sequence of Stockham steps (radix R, span Ls; task i takes the
// inputs i + u·L/R, twiddles them by w_{R·Ls}^{u·(i mod Ls)}, and writes
// the R outputs (i / Ls)·R·Ls + (i mod Ls) + s·Ls).  Between steps the
// values go through shared memory; the last forward step leaves each thread
// holding exactly the bins the first inverse step needs, so pass B takes
// the product and starts the inverse without touching shared memory.
//
// The spectrum of z* is computed once per (b, h) by spec_a/spec_b (generic
// Stockham in shared memory) and stored in the order pass B's threads hold
// the bins: thread j of the CTA for k2 holds k1 = 2j + e + 32s (e < 2,
// s < 16), stored at ((k2·16 + j)·16 + s)·2 + e.
#include <cuda_bf16.h>

#include "cat_internal.h"
#include "elem.cuh"
#include "fft_reg.cuh"

namespace cat {

constexpr int kFastN1 = 512;
constexpr int kFastPairs = 32;
constexpr int kRowB = kFastN1 + 2;   // shared row (complex) of one signal in pass B

__device__ __forceinline__ size_t scr_idx(int bhl, int N2, int k2, int n1, int pair) {
  return (((size_t)bhl * N2 + k2) * kFastN1 + n1) * kFastPairs + pair;
}

__device__ __forceinline__ void st_sh2(float2* p, float2 a, float2 b) {
  *reinterpret_cast<float4*>(p) = make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void ld_sh2(const float2* p, float2& a, float2& b) {
  float4 v = *reinterpret_cast<const float4*>(p);
  a = make_float2(v.x, v.y);
  b = make_float2(v.z, v.w);
}

// ---------------------------------------------------------------------------
// Pass A.  N2 == 32: a warp per n1 (8 per CTA), one thread per pair holds the
// whole length-32 transform.  N2 > 32: a CTA per n1, T = N2/32 warps; step 1
// (radix 32, span 1) then step 2 (radix N2/32, span 32) with thread j taking
// the tasks per·j + e, per = 32/T.
// ---------------------------------------------------------------------------
template <typename T, int N2>
__global__ void __launch_bounds__(256)
fsf_pass_a(const T* __restrict__ V, float2* __restrict__ scr, const float2* __restrict__ W,
           int N, int D, int H, int bh0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if constexpr (N2 == 32) {
    const int n1 = (blockIdx.x % (kFastN1 / 8)) * 8 + warp;
    const int bhl = blockIdx.x / (kFastN1 / 8);
    const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
    const T* src = V + ((size_t)b * N + n1) * D + h * 64 + 2 * lane;
    const size_t rs = (size_t)kFastN1 * D;
    float2 a[32];
#pragma unroll
    for (int n2 = 0; n2 < 32; ++n2) a[n2] = ld_pair(src + n2 * rs);
    dft<32, false>(a);
#pragma unroll
    for (int k2 = 0; k2 < 32; ++k2)
      scr[scr_idx(bhl, 32, k2, n1, lane)] = cmul(a[k2], __ldg(&W[(size_t)n1 * k2]));
  } else {
    constexpr int TS = N2 / 32;        // threads per signal
    constexpr int R2 = N2 / 32;        // radix of step 2
    constexpr int PER = 32 / TS;       // step-2 tasks per thread
    constexpr int RS = N2 + 2;         // shared row of one pair
    extern __shared__ float4 smem4[];
    float2* buf = reinterpret_cast<float2*>(smem4);
    const int j = warp;
    const int n1 = blockIdx.x % kFastN1;
    const int bhl = blockIdx.x / kFastN1;
    const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
    const T* src = V + ((size_t)b * N + n1) * D + h * 64 + 2 * lane;
    const size_t rs = (size_t)kFastN1 * D;
    float2 a[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) a[u] = ld_pair(src + (size_t)(j + TS * u) * rs);
    dft<32, false>(a);
    float2* row = buf + lane * RS;
#pragma unroll
    for (int s = 0; s < 32; s += 2) st_sh2(row + 32 * j + s, a[s], a[s + 1]);
    __syncthreads();
    float2 c[PER][R2];
#pragma unroll
    for (int u = 0; u < R2; ++u)
#pragma unroll
      for (int e = 0; e < PER; e += 2) ld_sh2(row + PER * j + e + 32 * u, c[e][u], c[e + 1][u]);
    const int wstep = N / N2;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int k = PER * j + e;
#pragma unroll
      for (int u = 1; u < R2; ++u) c[e][u] = cmul(c[e][u], __ldg(&W[(size_t)(u * k) * wstep]));
      dft<R2, false>(c[e]);
#pragma unroll
      for (int s = 0; s < R2; ++s) {
        const int k2 = k + 32 * s;
        scr[scr_idx(bhl, N2, k2, n1, lane)] = cmul(c[e][s], __ldg(&W[(size_t)n1 * k2]));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Pass C: the inverse of pass A's transform over k2, then the output rows.
// ---------------------------------------------------------------------------
template <typename T, int N2>
__global__ void __launch_bounds__(256)
fsf_pass_c(const float2* __restrict__ scr, T* __restrict__ O, const float2* __restrict__ W,
           int N, int D, int H, int bh0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if constexpr (N2 == 32) {
    const int n1 = (blockIdx.x % (kFastN1 / 8)) * 8 + warp;
    const int bhl = blockIdx.x / (kFastN1 / 8);
    const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
    float2 a[32];
#pragma unroll
    for (int k2 = 0; k2 < 32; ++k2) a[k2] = scr[scr_idx(bhl, 32, k2, n1, lane)];
    dft<32, true>(a);
    T* dst = O + ((size_t)b * N + n1) * D + h * 64 + 2 * lane;
    const size_t rs = (size_t)kFastN1 * D;
#pragma unroll
    for (int n2 = 0; n2 < 32; ++n2) st_pair(dst + n2 * rs, a[n2]);
  } else {
    constexpr int TS = N2 / 32;
    constexpr int R2 = N2 / 32;
    constexpr int PER = 32 / TS;
    constexpr int RS = N2 + 2;
    extern __shared__ float4 smem4[];
    float2* buf = reinterpret_cast<float2*>(smem4);
    const int j = warp;
    const int n1 = blockIdx.x % kFastN1;
    const int bhl = blockIdx.x / kFastN1;
    const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
    float2 a[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) a[u] = scr[scr_idx(bhl, N2, j + TS * u, n1, lane)];
    dft<32, true>(a);
    float2* row = buf + lane * RS;
#pragma unroll
    for (int s = 0; s < 32; s += 2) st_sh2(row + 32 * j + s, a[s], a[s + 1]);
    __syncthreads();
    float2 c[PER][R2];
#pragma unroll
    for (int u = 0; u < R2; ++u)
#pragma unroll
      for (int e = 0; e < PER; e += 2) ld_sh2(row + PER * j + e + 32 * u, c[e][u], c[e + 1][u]);
    const int wstep = N / N2;
    T* dst = O + ((size_t)b * N + n1) * D + h * 64 + 2 * lane;
    const size_t rs = (size_t)kFastN1 * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int k = PER * j + e;
#pragma unroll
      for (int u = 1; u < R2; ++u) c[e][u] = cmulc(c[e][u], __ldg(&W[(size_t)(u * k) * wstep]));
      dft<R2, true>(c[e]);
#pragma unroll
      for (int s = 0; s < R2; ++s) st_pair(dst + (size_t)(k + 32 * s) * rs, c[e][s]);
    }
  }
}

// ---------------------------------------------------------------------------
// Pass B: per (b, h, k2) and half of the head's pairs (16 signals of length
// 512).  Forward: step F1 (radix 32, span 1; thread j task j), step F2
// (radix 16, span 32; tasks 2j, 2j+1).  Product with the spectrum of z*.
// Inverse: step I1 (radix 16, span 1; tasks 2j, 2j+1 — exactly the bins the
// thread holds), step I2 (radix 32, span 16; task j), leaving n1 = j + 16s.
// Lane l: pair (l & 15) of the half, j = 2·warp + (l >> 4).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 2)
fsf_pass_b(float2* __restrict__ scr, const float2* __restrict__ zft, const float2* __restrict__ W,
           int N, int N2, int bh0) {
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pl = lane & 15;
  const int j = 2 * warp + (lane >> 4);
  const int grp = blockIdx.x & 1;
  const int k2 = (blockIdx.x >> 1) % N2;
  const int bhl = (blockIdx.x >> 1) / N2;
  const int pair = grp * 16 + pl;
  const int wstep = N / kFastN1;
  float2* row = buf + pl * kRowB;

  float2 a[32];
#pragma unroll
  for (int u = 0; u < 32; ++u) a[u] = scr[scr_idx(bhl, N2, k2, j + 16 * u, pair)];
  dft<32, false>(a);
#pragma unroll
  for (int s = 0; s < 32; s += 2) st_sh2(row + 32 * j + s, a[s], a[s + 1]);
  __syncthreads();

  float2 c[2][16];
#pragma unroll
  for (int u = 0; u < 16; ++u) ld_sh2(row + 2 * j + 32 * u, c[0][u], c[1][u]);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int k = 2 * j + e;
#pragma unroll
    for (int u = 1; u < 16; ++u) c[e][u] = cmul(c[e][u], __ldg(&W[(size_t)(u * k) * wstep]));
    dft<16, false>(c[e]);
  }
  // Product with FFT(z*)/N at bins k1 = 2j + e + 32s.
  const float4* zrow = reinterpret_cast<const float4*>(zft) +
                       (((size_t)(bh0 + bhl) * N2 + k2) * 16 + j) * 16;
#pragma unroll
  for (int s = 0; s < 16; ++s) {
    float4 z = __ldg(zrow + s);
    c[0][s] = cmul(c[0][s], make_float2(z.x, z.y));
    c[1][s] = cmul(c[1][s], make_float2(z.z, z.w));
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    dft<16, true>(c[e]);
#pragma unroll
    for (int s = 0; s < 16; s += 2) st_sh2(row + 32 * j + 16 * e + s, c[e][s], c[e][s + 1]);
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 32; ++u) a[u] = row[j + 16 * u];
#pragma unroll
  for (int u = 1; u < 32; ++u) a[u] = cmulc(a[u], __ldg(&W[(size_t)(u * j) * wstep]));
  dft<32, true>(a);
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    const int n1 = j + 16 * s;
    scr[scr_idx(bhl, N2, k2, n1, pair)] = cmulc(a[s], __ldg(&W[(size_t)n1 * k2]));
  }
}

// ---------------------------------------------------------------------------
// Spectrum of z* in pass B's order (generic Stockham in shared memory).
// spec_a: CTA per (b, h, tile of TZ n1 values): DFT over n2, twiddle into
// zscr[bh][k2][n1].  spec_b: CTA per (b, h, k2): DFT over n1, /N, scatter.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
fsf_spec_a(const float* __restrict__ zs, float2* __restrict__ zscr, const float2* __restrict__ W,
           RadixPlan rp2, int N, int TZ, unsigned int* status) {
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  const int N2 = rp2.L;
  const int ntile = kFastN1 / TZ;
  const int bh = blockIdx.x / ntile, n10 = (blockIdx.x % ntile) * TZ;
  if (TZ * N2 > vals_capacity(rp2) * (int)blockDim.x) {
    report(status, 0x401);
    return;
  }
  const float* zrow = zs + (size_t)bh * N;
  for (int idx = threadIdx.x; idx < TZ * N2; idx += blockDim.x) {
    int t = idx % TZ, n2 = idx / TZ;
    buf[t * N2 + n2] = make_float2(__ldg(zrow + n10 + t + kFastN1 * n2), 0.f);
  }
  __syncthreads();
  block_fft<false>(buf, rp2, TZ, N2, W, kFastN1);
  float2* out = zscr + (size_t)bh * N;
  for (int idx = threadIdx.x; idx < TZ * N2; idx += blockDim.x) {
    int t = idx % TZ, k2 = idx / TZ;
    int n1 = n10 + t;
    out[(size_t)k2 * kFastN1 + n1] = cmul(buf[t * N2 + k2], __ldg(&W[(size_t)n1 * k2]));
  }
}

__global__ void __launch_bounds__(1024)
fsf_spec_b(const float2* __restrict__ zscr, float2* __restrict__ zft, const float2* __restrict__ W,
           RadixPlan rp1, int N, int N2, unsigned int* status) {
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  const int bh = blockIdx.x / N2, k2 = blockIdx.x % N2;
  if (kFastN1 > vals_capacity(rp1) * (int)blockDim.x) {
    report(status, 0x402);
    return;
  }
  const float2* in = zscr + (size_t)bh * N + (size_t)k2 * kFastN1;
  for (int n1 = threadIdx.x; n1 < kFastN1; n1 += blockDim.x) buf[n1] = in[n1];
  __syncthreads();
  block_fft<false>(buf, rp1, 1, kFastN1, W, N2);
  const float invN = 1.0f / (float)N;
  float2* out = zft + ((size_t)bh * N2 + k2) * kFastN1;
  for (int k1 = threadIdx.x; k1 < kFastN1; k1 += blockDim.x) {
    int jj = (k1 & 31) >> 1, e = k1 & 1, s = k1 >> 5;
    out[(jj * 16 + s) * 2 + e] = cscale(buf[k1], invN);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
constexpr int kSpecTZ = 8;   // n1 values per spec_a CTA

size_t fast_smem_a(int N2) { return N2 == 32 ? 0 : (size_t)kFastPairs * (N2 + 2) * sizeof(float2); }
size_t fast_smem_b() { return (size_t)16 * kRowB * sizeof(float2); }

template <typename T>
static cudaError_t setup_t(int N2) {
  cudaError_t e = cudaSuccess;
  switch (N2) {
#define CAT_N2(n)                                                   \
  case n:                                                           \
    e = allow_max_smem(fsf_pass_a<T, n>);                           \
    if (e == cudaSuccess) e = allow_max_smem(fsf_pass_c<T, n>);     \
    break;
    CAT_N2(32) CAT_N2(64) CAT_N2(128) CAT_N2(256)
#undef CAT_N2
    default: return cudaErrorInvalidValue;
  }
  if (e == cudaSuccess) e = allow_max_smem(fsf_pass_b);
  if (e == cudaSuccess) e = allow_max_smem(fsf_spec_a);
  if (e == cudaSuccess) e = allow_max_smem(fsf_spec_b);
  return e;
}

cudaError_t setup_fast_kernels(const cat_plan_s* p) {
  return p->dtype == 1 ? setup_t<__nv_bfloat16>(p->fs.N2) : setup_t<float>(p->fs.N2);
}

template <typename T, int N2>
static void launch_ac(const cat_plan_s* p, const T* V, T* O, int bh0, int nb, bool pass_a) {
  const int grid = N2 == 32 ? nb * (kFastN1 / 8) : nb * kFastN1;
  const int threads = N2 == 32 ? 256 : N2;
  const size_t smem = fast_smem_a(N2);
  if (pass_a)
    fsf_pass_a<T, N2><<<grid, threads, smem, p->stream>>>(V, p->scratch, p->tw, p->N, p->D, p->H, bh0);
  else
    fsf_pass_c<T, N2><<<grid, threads, smem, p->stream>>>(p->scratch, O, p->tw, p->N, p->D, p->H, bh0);
}

template <typename T>
static cudaError_t run_t(const cat_plan_s* p, const T* V, T* O) {
  const FourStepCfg& f = p->fs;
  const int rows = p->B * p->H;
  const int N2 = f.N2;
  // Spectrum of z*, once per (b, h).
  const int ga = rows * (kFastN1 / kSpecTZ);
  fsf_spec_a<<<ga, 256, (size_t)kSpecTZ * N2 * sizeof(float2), p->stream>>>(
      p->zs, p->zscr, p->tw, f.rp2, p->N, kSpecTZ, p->status);
  fsf_spec_b<<<rows * N2, 64, (size_t)kFastN1 * sizeof(float2), p->stream>>>(
      p->zscr, p->zf, p->tw, f.rp1, p->N, N2, p->status);
  for (int bh0 = 0; bh0 < rows; bh0 += f.chunk_bh) {
    const int nb = rows - bh0 < f.chunk_bh ? rows - bh0 : f.chunk_bh;
    auto ac = [&](bool pass_a) {
      switch (N2) {
        case 32: launch_ac<T, 32>(p, V, O, bh0, nb, pass_a); break;
        case 64: launch_ac<T, 64>(p, V, O, bh0, nb, pass_a); break;
        case 128: launch_ac<T, 128>(p, V, O, bh0, nb, pass_a); break;
        default: launch_ac<T, 256>(p, V, O, bh0, nb, pass_a); break;
      }
    };
    ac(true);
    fsf_pass_b<<<nb * N2 * 2, 256, fast_smem_b(), p->stream>>>(p->scratch, p->zf, p->tw, p->N,
                                                                N2, bh0);
    ac(false);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_fast_conv(const cat_plan_s* p, const void* V, void* O) {
  if (p->B == 0) return cudaSuccess;
  if (p->dtype == 1) return run_t(p, (const __nv_bfloat16*)V, (__nv_bfloat16*)O);
  return run_t(p, (const float*)V, (float*)O);
}

}  // namespace cat
