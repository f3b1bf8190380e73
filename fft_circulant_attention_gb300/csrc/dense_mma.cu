// The backward's two dense contractions on the tensor cores (bf16 data):
//
//   dW_A[d, h] = sum over tokens t of X[t, d] · dz[h, t]     (K = B·N tokens)
//   dX[t, d]   = sum over heads h of dz[h, t] · W_A[d, h]    (K = H <= 16)
//
// (the chain rule through the score z = X·W_A of the CAT notes page, section
// 方法详解).  X and W_A are bf16 and enter the products exactly; dz is fp32
// and is split into two bf16 terms, dz = hi + lo + r with hi = bf16(dz),
// lo = bf16(dz - hi) and |r| <= 2^-18 |dz|, so each product carries the
// split's 2^-18 relative error and the sums accumulate in fp32 (mma.sync
// m16n8k16, bf16 in, fp32 out), as the FP32 kernels they replace do.  Both
// kernels are bound by their one pass over X or dX in HBM; on the FP32 pipe
// the 2·B·N·D·H flops of each took longer than that pass.
//
// dwa_mma_kernel: CTA (d-group g of 256 columns, token split s) streams
// tiles of 64 tokens: a producer warp waits for a free stage, writes the
// tile's dz (hi, lo) as bf16 [h][token] into it and issues four 2-D tensor
// copies (64 tokens x 64 d each, 128-byte swizzle); each of four consumer
// warps takes its 64 columns (four 16-row A tiles, read transposed with
// ldmatrix) against the 16 heads (two 8-column B tiles), 16 MMAs per 16
// tokens.  The CTA's sums go to part[s][h][d]; dwa_reduce_kernel adds the
// splits in order.
//
// dx_mma_kernel: W_A staged once per CTA as bf16 [d][h] (padded); each warp
// takes tiles of 16 tokens: dz's A fragment (hi and lo), then for every 64
// columns eight B tiles and 16 MMAs, the 16 x 64 result rounded to bf16 and
// staged in shared memory, and written as 128-byte row segments.
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "bulk.cuh"
#include "cat_internal.h"
#include "elem.cuh"
#include "fft_device.cuh"
#include "mma.cuh"

namespace cat {

// bf16 bit patterns of the two-term split of x.
static __device__ __forceinline__ void split_bf16(float x, unsigned short& hi, unsigned short& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}

static __device__ __forceinline__ unsigned pack2(unsigned short a, unsigned short b) {
  return (unsigned)a | ((unsigned)b << 16);
}

// Offset of dz[b, 0, n] for token row r = b·N + n of B·N, or -1 past the
// end (dz[h, r] is then at that offset + h·N).
static __device__ __forceinline__ long long dz_row(long long r, long long rows, int H, int N) {
  if (r >= rows) return -1;
  const long long b = r / N;
  return b * H * (long long)N + (r - b * N);
}

// ---------------------------------------------------------------------------
// dW_A
// ---------------------------------------------------------------------------
constexpr int kDmTok = 64;                       // tokens a tile
constexpr int kDmCons = 4;                       // consumer warps (64 columns each)
constexpr int kDmCols = kDmCons * 64;            // columns a CTA
constexpr int kDmStages = 3;
constexpr int kDmThreads = (kDmCons + 1) * 32;
constexpr int kDmBox = kDmTok * 64 * 2;          // one tensor copy: 64 tokens x 64 d
constexpr int kDmXStage = kDmCons * kDmBox;
constexpr int kDmZs = kDmTok + 8;                // dz stage row (bf16), bank-spread
constexpr int kDmZStage = 2 * 16 * kDmZs * 2;    // hi and lo rows of 16 heads
constexpr size_t kDmSmem =
    1024 + (size_t)kDmStages * (kDmXStage + kDmZStage) + 2 * kDmStages * sizeof(uint64_t);

__global__ void __launch_bounds__(kDmThreads, 2)
dwa_mma_kernel(const __grid_constant__ CUtensorMap tmX, const float* __restrict__ dz,
               float* __restrict__ part, int N, int D, int H, long long rows, int ntiles,
               unsigned int* status) {
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* xst = sm;                                         // [stage][4 boxes]
  unsigned short* zst = reinterpret_cast<unsigned short*>(sm + kDmStages * kDmXStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kDmStages * (kDmXStage + kDmZStage));
  uint64_t* empty = full + kDmStages;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int split = blockIdx.y, nsplit = gridDim.y;
  const int d0 = blockIdx.x * kDmCols;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDmStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kDmCons);
    }
  }
  mbar_fence_init();
  __syncthreads();

  if (warp == kDmCons) {   // producer
    const uint64_t stream = policy_evict_first();
    // The tile's dz: this lane's tokens are lane and lane + 32, all 16
    // heads, loaded one tile ahead (in flight while the stage is waited for).
    float v[2][16];
    auto load_dz = [&](int tile) {
      const long long r0 = (long long)tile * kDmTok;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const long long o = dz_row(r0 + lane + 32 * e, rows, H, N);
#pragma unroll
        for (int h = 0; h < 16; ++h) v[e][h] = (o >= 0 && h < H) ? dz[o + (size_t)h * N] : 0.f;
      }
    };
    if (split < ntiles) load_dz(split);
    int it = 0;
    for (int tile = split; tile < ntiles; tile += nsplit, ++it) {
      const int s = it % kDmStages, use = it / kDmStages;
      bool ok = true;
      if (use > 0 && lane == 0) ok = mbar_wait(empty + s, (use - 1) & 1, status, 0x701);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
      // dz as bf16 hi / lo rows [h][token].
      unsigned short* zh = zst + (size_t)s * (kDmZStage / 2);
      unsigned short* zl = zh + 16 * kDmZs;
      const long long r0 = (long long)tile * kDmTok;
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          unsigned short a, b;
          split_bf16(v[e][h], a, b);
          zh[h * kDmZs + lane + 32 * e] = a;
          zl[h * kDmZs + lane + 32 * e] = b;
        }
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_smem();   // the consumers' ldmatrix reads come first
        mbar_expect_tx(full + s, kDmXStage);
        for (int w = 0; w < kDmCons; ++w)
          tma_load_2d_hint(xst + s * kDmXStage + w * kDmBox, &tmX, d0 + 64 * w, (int)r0, full + s,
                           stream);
      }
      if (tile + nsplit < ntiles) load_dz(tile + nsplit);
    }
    return;
  }

  // Consumer warp: columns d0 + 64·warp + [0, 64) (zeros from the tensor copy
  // past D, not stored).
  const int g = lane >> 2, c = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;          // ldmatrix matrix / row of this lane
  float acc[4][2][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
  int it = 0;
  for (int tile = split; tile < ntiles; tile += nsplit, ++it) {
    const int s = it % kDmStages;
    if (!mbar_wait(full + s, (it / kDmStages) & 1, status, 0x702)) return;
    const uint32_t xb = smem_addr(xst + s * kDmXStage + warp * kDmBox);
    const unsigned short* zh = zst + (size_t)s * (kDmZStage / 2);
    const unsigned short* zl = zh + 16 * kDmZs;
#pragma unroll
    for (int k16 = 0; k16 < kDmTok / 16; ++k16) {
      unsigned bh[2][2], bl[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int o = (nt * 8 + g) * kDmZs + 16 * k16 + 2 * c;
        bh[nt][0] = *reinterpret_cast<const unsigned*>(zh + o);
        bh[nt][1] = *reinterpret_cast<const unsigned*>(zh + o + 8);
        bl[nt][0] = *reinterpret_cast<const unsigned*>(zl + o);
        bl[nt][1] = *reinterpret_cast<const unsigned*>(zl + o + 8);
      }
      // Matrix mi of the A tile: tokens 16·k16 + 8·(mi >> 1) + [0, 8),
      // columns 16·mt + 8·(mi & 1) + [0, 8), read transposed.
      const int row = 16 * k16 + 8 * (mi >> 1) + mr;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int chunk = 2 * mt + (mi & 1);
        unsigned a[4];
        ldmatrix_x4_trans(a, xb + row * 128 + ((chunk ^ (row & 7)) << 4));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          mma_bf16(acc[mt][nt], a, bh[nt][0], bh[nt][1]);
          mma_bf16(acc[mt][nt], a, bl[nt][0], bl[nt][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
  // acc[mt][nt][i]: column d = 16·mt + g + 8·(i >> 1), head h = 8·nt + 2c + (i & 1).
  const int dw = d0 + 64 * warp;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int d = dw + 16 * mt + g + 8 * (i >> 1), h = 8 * nt + 2 * c + (i & 1);
        if (h < H && d < D) part[((size_t)split * H + h) * D + d] = acc[mt][nt][i];
      }
}

// ---------------------------------------------------------------------------
// dX
// ---------------------------------------------------------------------------
constexpr int kDxmWarps = 8;
constexpr int kDxmWs = 24;                        // W_A row stride (bf16), bank-spread
constexpr int kDxmOs = 72;                        // output stage row stride (bf16)
constexpr int kDxmOut = 16 * kDxmOs * 2;          // one warp's 16 x 64 stage (bytes)
static size_t dx_mma_smem(int D) { return (size_t)D * kDxmWs * 2 + (size_t)kDxmWarps * kDxmOut; }

__global__ void __launch_bounds__(kDxmWarps * 32)
dx_mma_kernel(const float* __restrict__ dz, const __nv_bfloat16* __restrict__ WA,
              __nv_bfloat16* __restrict__ dX, int N, int D, int H, long long rows, int ntiles) {
  extern __shared__ __align__(16) unsigned char sm[];
  unsigned short* wa = reinterpret_cast<unsigned short*>(sm);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned short* os = reinterpret_cast<unsigned short*>(sm + (size_t)D * kDxmWs * 2) +
                       (size_t)warp * (kDxmOut / 2);
  // W_A as bf16 [d][h], heads padded to 16 with zeros; eight loads a
  // thread in flight before any is stored (one at a time, the CTA's start
  // waited D·16 / threads memory latencies).
  const unsigned short* wg = reinterpret_cast<const unsigned short*>(WA);
  for (int i0 = threadIdx.x; i0 < D * 16; i0 += 8 * blockDim.x) {
    unsigned short v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x, d = i >> 4, h = i & 15;
      v[u] = (i < D * 16 && h < H) ? wg[(size_t)d * H + h] : (unsigned short)0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < D * 16) wa[(i >> 4) * kDxmWs + (i & 15)] = v[u];
    }
  }
  __syncthreads();
  const int g = lane >> 2, c = lane & 3;
  const int gw = blockIdx.x * kDxmWarps + warp, G = gridDim.x * kDxmWarps;
  // Items (tile of 16 tokens, group of up to 4 x 64 columns), the tile's A
  // fragment loaded one item ahead.  A fragment element e (e = 0..7 in the
  // order of the packed halves): token g + 8·(e >> 1 & 1), head
  // 2c + (e & 1) + 8·(e >> 2).
  const int ngrp = (D / 64 + 3) / 4, items = ntiles * ngrp;
  float nxt[8];
  auto load_a = [&](int item) {
    const long long r0 = (long long)(item / ngrp) * 16;
    const long long o0 = dz_row(r0 + g, rows, H, N), o1 = dz_row(r0 + g + 8, rows, H, N);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const long long o = (e >> 1) & 1 ? o1 : o0;
      const int h = 2 * c + (e & 1) + 8 * (e >> 2);
      nxt[e] = (o >= 0 && h < H) ? dz[o + (size_t)h * N] : 0.f;
    }
  };
  if (gw < items) load_a(gw);
  for (int item = gw; item < items; item += G) {
    unsigned ah[4], al[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      unsigned short h0, l0, h1, l1;
      split_bf16(nxt[2 * q], h0, l0);
      split_bf16(nxt[2 * q + 1], h1, l1);
      ah[q] = pack2(h0, h1);
      al[q] = pack2(l0, l1);
    }
    if (item + G < items) load_a(item + G);
    const long long r0 = (long long)(item / ngrp) * 16;
    const int dg0 = (item % ngrp) * 4, dg1 = min(dg0 + 4, D / 64);
    for (int dg = dg0; dg < dg1; ++dg) {
      float acc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
        const unsigned short* wr = wa + (dg * 64 + nt * 8 + g) * kDxmWs + 2 * c;
        const unsigned b0 = *reinterpret_cast<const unsigned*>(wr);
        const unsigned b1 = *reinterpret_cast<const unsigned*>(wr + 8);
        mma_bf16(acc[nt], ah, b0, b1);
        mma_bf16(acc[nt], al, b0, b1);
      }
      // acc[nt][i]: token g + 8·(i >> 1), column 8·nt + 2c + (i & 1).
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const __nv_bfloat162 v0 = __floats2bfloat162_rn(acc[nt][0], acc[nt][1]);
        const __nv_bfloat162 v1 = __floats2bfloat162_rn(acc[nt][2], acc[nt][3]);
        *reinterpret_cast<__nv_bfloat162*>(os + g * kDxmOs + nt * 8 + 2 * c) = v0;
        *reinterpret_cast<__nv_bfloat162*>(os + (g + 8) * kDxmOs + nt * 8 + 2 * c) = v1;
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int k = lane + 32 * q, row = k >> 3, c16 = k & 7;
        const long long r = r0 + row;
        if (r < rows) {
          const uint4 v = *reinterpret_cast<const uint4*>(os + row * kDxmOs + c16 * 8);
          *reinterpret_cast<uint4*>(dX + (size_t)r * D + dg * 64 + c16 * 8) = v;
        }
      }
      __syncwarp();
    }
  }
}

// The tensor-core kernels serve bf16 data with D a multiple of 64, at most
// 16 heads, and 16-byte aligned X and dX (tensor copies of X, 16-byte
// stores of dX).  CAT_DENSE_MMA=0 keeps the FP32 kernels.
bool dense_mma_ok(const cat_plan_s* p, const void* X, const void* dX) {
  if (const char* e = std::getenv("CAT_DENSE_MMA"))
    if (e[0] == '0') return false;
  return p->dtype == 1 && p->D % 64 == 0 && p->H <= 16 && ((uintptr_t)X % 16) == 0 &&
         ((uintptr_t)dX % 16) == 0 && dx_mma_smem(p->D) <= (200u << 10);
}

cudaError_t setup_dense_mma() {
  cudaError_t e = allow_max_smem(dwa_mma_kernel);
  if (e == cudaSuccess) e = allow_max_smem(dx_mma_kernel);
  return e;
}

// Token splits of the dW_A kernel: two CTAs per SM over the d-groups, at
// most `most` (the partial-sum buffer's splits) and the tile count.
int dwa_mma_splits(const cat_plan_s* p, int most) {
  const int groups = (p->D + kDmCols - 1) / kDmCols;
  const long long ntiles = ((long long)p->B * p->N + kDmTok - 1) / kDmTok;
  long long s = 2ll * p->sms / groups;
  if (s > most) s = most;
  if (s > ntiles) s = ntiles;
  if (s < 1) s = 1;
  return (int)s;
}

cudaError_t launch_dwa_mma(const cat_plan_s* p, const void* X, float* part, int nsplit) {
  const long long rows = (long long)p->B * p->N;
  CUtensorMap tm;
  if (!encode_map_2d_sw128(&tm, X, (unsigned long long)p->D, (unsigned long long)rows,
                           (unsigned long long)p->D * 2, 64, kDmTok))
    return cudaErrorInvalidValue;
  const int ntiles = (int)((rows + kDmTok - 1) / kDmTok);
  // The column groups of one token split are adjacent in launch order, so
  // they read the same rows of X at about the same time.
  dim3 grid((p->D + kDmCols - 1) / kDmCols, nsplit);
  dwa_mma_kernel<<<grid, kDmThreads, kDmSmem, p->stream>>>(tm, p->bw_dz, part, p->N, p->D, p->H,
                                                           rows, ntiles, p->status);
  return cudaGetLastError();
}

cudaError_t launch_dx_mma(const cat_plan_s* p, const void* WA, void* dX) {
  const long long rows = (long long)p->B * p->N;
  const int ntiles = (int)((rows + 15) / 16);
  const size_t smem = dx_mma_smem(p->D);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dx_mma_kernel, kDxmWarps * 32,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  long long grid = (long long)per_sm * p->sms;
  const long long items = (long long)ntiles * ((p->D / 64 + 3) / 4);
  const long long need = (items + kDxmWarps - 1) / kDxmWarps;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  dx_mma_kernel<<<(unsigned)grid, kDxmWarps * 32, smem, p->stream>>>(
      p->bw_dz, (const __nv_bfloat16*)WA, (__nv_bfloat16*)dX, p->N, p->D, p->H, rows, ntiles);
  return cudaGetLastError();
}

}  // namespace cat
