// Measurement probe: one length-32 DFT stage on the FP32 pipe against the
// same stage as a dense contraction on the tensor cores (tcgen05), for the
// choice of where the small-DFT stages of the circulant product run.  Not
// part of the forward or backward path.
//
// Both variants transform `nsig` complex signals of length 32, each kept on
// chip for `rounds` applications of the stage (every application scaled by
// 1/sqrt(32), so that magnitudes stay put), so the time is the stage's own
// cost, not the memory's:
//  - FP32: one signal per thread, the register DFT-32 of the fast path's
//    passes A and C.
//  - Tensor: 128 signals per CTA (one thread and one tensor-memory lane
//    each), as real vectors of 64 (re, im interleaved) times the 64 x 64 real
//    matrix of the DFT; per round each thread splits its fp32 values into
//    `terms` bf16 parts and writes them to shared memory in the 128-byte
//    swizzled K-major layout, one thread issues the MMAs of every term pair
//    of total order < terms (3 sets for 2 terms, 6 for 3; 4 MMAs of K = 16
//    each), and the accumulator comes back by tcgen05.ld.  Two terms carry
//    about 16 significant bits, three about 24 (fp32 class).
#include <cuda_bf16.h>

#include <cmath>

#include "../../include/cat.h"
#include "cat_internal.h"
#include "elem.cuh"
#include "fft_reg.cuh"
#include "tc.cuh"

namespace cat {

__global__ void __launch_bounds__(256)
probe_dft32_fp32(const float2* __restrict__ x, float2* __restrict__ y, int nsig, int rounds) {
  const int sig = blockIdx.x * blockDim.x + threadIdx.x;
  if (sig >= nsig) return;
  float2 a[32];
#pragma unroll
  for (int n = 0; n < 32; ++n) a[n] = x[(size_t)sig * 32 + n];
  const float s = 0.17677669529663687f;   // 1/sqrt(32)
  for (int r = 0; r < rounds; ++r) {
    dft<32, false>(a);
#pragma unroll
    for (int n = 0; n < 32; ++n) a[n] = make_float2(a[n].x * s, a[n].y * s);
  }
#pragma unroll
  for (int n = 0; n < 32; ++n) y[(size_t)sig * 32 + n] = a[n];
}

constexpr int kPrRows = 128;   // signals per CTA (MMA M)
constexpr int kPrK = 64;       // real input length (MMA K)
constexpr int kPrN = 64;       // real output length (MMA N)
constexpr int kPrTile = kPrRows * kPrK * 2;   // one bf16 A tile, 16 KB
constexpr int kPrB = kPrN * kPrK * 2;         // one bf16 B tile, 8 KB

// Byte offset of element (row, k) of a 128-byte-swizzled K-major bf16 tile.
__device__ __forceinline__ uint32_t sw128(int row, int k) {
  const int chunk = (k >> 3) ^ (row & 7);
  return (uint32_t)(row * 128 + chunk * 16 + (k & 7) * 2);
}

template <int TERMS>
__global__ void __launch_bounds__(kPrRows, 1)
probe_dft32_tc(const float2* __restrict__ x, float2* __restrict__ y,
               const __nv_bfloat16* __restrict__ fparts, int nsig, int rounds,
               unsigned int* status) {
  extern __shared__ unsigned char pr_raw[];
  const uint32_t raw = smem_addr(pr_raw);
  unsigned char* sm = pr_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char* atile = sm;                              // TERMS A tiles
  unsigned char* btile = sm + TERMS * kPrTile;            // TERMS B tiles
  uint64_t* bar = reinterpret_cast<uint64_t*>(btile + TERMS * kPrB);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int t = threadIdx.x, warp = t >> 5;
  const int sig = blockIdx.x * kPrRows + t;

  // B: the DFT matrix parts (rows = 64 outputs, K-major), swizzled.
  for (int i = t; i < TERMS * kPrN * kPrK; i += blockDim.x) {
    const int part = i / (kPrN * kPrK), e = i % (kPrN * kPrK);
    const int row = e / kPrK, k = e % kPrK;
    *reinterpret_cast<__nv_bfloat16*>(btile + part * kPrB + sw128(row, k)) = fparts[i];
  }
  if (t == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tslot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);

  float v[64];
#pragma unroll
  for (int n = 0; n < 32; ++n) {
    const float2 q = sig < nsig ? x[(size_t)sig * 32 + n] : make_float2(0.f, 0.f);
    v[2 * n] = q.x;
    v[2 * n + 1] = q.y;
  }
  const float s = 0.17677669529663687f;
  constexpr uint32_t idesc = idesc_bf16_f32(kPrRows, kPrN);
  bool ok = true;
  for (int r = 0; r < rounds && ok; ++r) {
    // Split this thread's row into TERMS bf16 parts.
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      float rest = v[k];
#pragma unroll
      for (int part = 0; part < TERMS; ++part) {
        const __nv_bfloat16 h = __float2bfloat16_rn(rest);
        *reinterpret_cast<__nv_bfloat16*>(atile + part * kPrTile + sw128(t, k)) = h;
        rest -= __bfloat162float(h);
      }
    }
    fence_proxy_async_smem();   // the generic stores before the MMAs read them
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      int first = 1;
#pragma unroll
      for (int pa = 0; pa < TERMS; ++pa)
#pragma unroll
        for (int pb = 0; pb + pa < TERMS; ++pb)
#pragma unroll
          for (int kk = 0; kk < kPrK / 16; ++kk) {
            tc_mma_bf16(tmem, sdesc_k128(atile + pa * kPrTile + 32 * kk),
                        sdesc_k128(btile + pb * kPrB + 32 * kk), idesc, first ? 0u : 1u);
            first = 0;
          }
      tc_commit(bar);
    }
    if (!mbar_wait(bar, (uint32_t)(r & 1), status, 0x701)) ok = false;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < 64; c += 16) tc_ld16(taddr + c, v + c);
#pragma unroll
    for (int k = 0; k < 64; ++k) v[k] *= s;
    tc_fence_before();
    __syncthreads();   // every thread's reads of the accumulator are done
  }
  if (sig < nsig) {
#pragma unroll
    for (int n = 0; n < 32; ++n) y[(size_t)sig * 32 + n] = make_float2(v[2 * n], v[2 * n + 1]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

static size_t probe_smem(int terms) { return 1024 + (size_t)terms * (kPrTile + kPrB) + 64; }

}  // namespace cat

namespace {
// The DFT-32 matrix as 64 x 64 real (rows: outputs re/im interleaved, columns:
// inputs re/im interleaved), split into `terms` bf16 parts, in fp64 on the
// host: w = exp(-2πi kn/32) = c - i s acts on (xr, xi) as
// (xr c + xi s, xi c - xr s).
int g_terms_built = 0;
__nv_bfloat16* g_parts = nullptr;
}  // namespace

extern "C" int cat_probe_dft32(const void* x, void* y, int nsig, int mode, int rounds,
                               void* stream) {
  using namespace cat;
  if (!x || !y || nsig < 0 || rounds < 1 || mode < 0 || mode > 2) return CAT_ERR_INVALID_ARG;
  if (nsig == 0) return CAT_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (mode == 0) {
    probe_dft32_fp32<<<(nsig + 255) / 256, 256, 0, st>>>((const float2*)x, (float2*)y, nsig,
                                                         rounds);
    return cudaGetLastError() == cudaSuccess ? CAT_OK : CAT_ERR_CUDA;
  }
  const int terms = mode == 1 ? 2 : 3;
  if (!g_parts) {
    __nv_bfloat16 host[3 * 64 * 64];
    const double two_pi = 6.283185307179586476925286766559;
    for (int row = 0; row < 64; ++row)
      for (int col = 0; col < 64; ++col) {
        const int k = row / 2, n = col / 2;
        const double a = two_pi * (double)((k * n) % 32) / 32.0;
        const double c = std::cos(a), s = std::sin(a);
        double f;
        if ((row & 1) == 0) f = (col & 1) == 0 ? c : s;
        else f = (col & 1) == 0 ? -s : c;
        double rest = f;
        for (int part = 0; part < 3; ++part) {
          const __nv_bfloat16 h = __float2bfloat16_rn((float)rest);
          host[part * 4096 + row * 64 + col] = h;
          rest -= (double)__bfloat162float(h);
        }
      }
    if (cudaMalloc(&g_parts, sizeof(host)) != cudaSuccess) {
      cudaGetLastError();
      g_parts = nullptr;
      return CAT_ERR_ALLOC;
    }
    if (cudaMemcpy(g_parts, host, sizeof(host), cudaMemcpyHostToDevice) != cudaSuccess)
      return CAT_ERR_CUDA;
  }
  static unsigned int* status = nullptr;
  if (!status) {
    if (cudaMalloc(&status, sizeof(unsigned int)) != cudaSuccess) return CAT_ERR_ALLOC;
    if (cudaMemset(status, 0, sizeof(unsigned int)) != cudaSuccess) return CAT_ERR_CUDA;
  }
  const size_t smem = probe_smem(terms);
  const int grid = (nsig + kPrRows - 1) / kPrRows;
  if (terms == 2) {
    if (cudaFuncSetAttribute(probe_dft32_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return CAT_ERR_CUDA;
    probe_dft32_tc<2><<<grid, kPrRows, smem, st>>>((const float2*)x, (float2*)y, g_parts, nsig,
                                                   rounds, status);
  } else {
    if (cudaFuncSetAttribute(probe_dft32_tc<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return CAT_ERR_CUDA;
    probe_dft32_tc<3><<<grid, kPrRows, smem, st>>>((const float2*)x, (float2*)y, g_parts, nsig,
                                                   rounds, status);
  }
  return cudaGetLastError() == cudaSuccess ? CAT_OK : CAT_ERR_CUDA;
}
