// Fused value and score projection on the tensor cores (tcgen05): one pass
// over X gives both V = X·W_V and the scores z = X·W_A.  The notes page
// "CAT: Circular-Convolutional Attention for Sub-Quadratic Transformers"
// (section 方法详解, 整体框架 overall framework) gives a CAT layer exactly these
// two projections of the same tokens: W_V (D x D) for the values and W_A
// (D x H, one column per head) for the scores.  Both are one GEMM,
//     [V | z] = X · [W_V | W_A],   X: [B·N, D],
// with bf16 operands, exact bf16 products and fp32 accumulation in tensor
// memory.
//
// Tiles of 128 tokens (the MMA's M, one tensor-memory lane each) by 256
// value columns, or by the 16 score columns (heads padded with zeros).  The
// kernel is persistent, one CTA per SM: CTA c takes the tiles c, c + grid,
// ... of the list ordered token block first, so the CTAs working at one time
// share their token blocks of X through L2.  Three roles:
//   - warp 0 issues the tensor copies of the X and W tiles (64-wide K
//     slices, 128-byte swizzle) into a ring of kPjStages stages, running
//     ahead across tiles;
//   - warp 1 allocates the tensor memory (two accumulators of 256 columns)
//     and one of its threads issues the MMAs of each stage, releasing the
//     stage through tcgen05.commit; a tile's last commit marks its
//     accumulator full;
//   - warps 2-5 read a full accumulator back (tcgen05.ld), store V in bf16
//     (round to nearest even) or z as a double-float, and mark it empty, so
//     the MMAs of the next tile run into the other accumulator meanwhile.
// Every mbarrier wait is bounded; a lost wait ends the role's loop.
//
// Scores: the peaked workloads need z to about 1e-6 absolute, so each
// 64-wide K slice (a group of slices when D > 1024) accumulates into its own
// 16 tensor-memory columns, and the epilogue adds the slice sums with TwoSum
// into (hi, lo), as the score kernels do.
#include <cuda_bf16.h>

#include "cat_internal.h"
#include "elem.cuh"
#include "tc.cuh"

namespace cat {

constexpr int kPjM = 128;                        // tokens per tile (MMA M)
constexpr int kPjK = 64;                         // K per stage: one 128-byte row
constexpr int kPjNV = 256;                       // value columns per tile (MMA N)
constexpr int kPjNZ = 16;                        // score columns per tile (MMA N)
constexpr int kPjStages = 4;
constexpr int kPjThreads = 192;                  // warp 0 copies, 1 MMA, 2-5 epilogue
constexpr int kPjXBytes = kPjM * kPjK * 2;       // 16 KB
constexpr int kPjWBytes = kPjNV * kPjK * 2;      // 32 KB
constexpr int kPjStageBytes = kPjXBytes + kPjWBytes;
constexpr int kPjMaxSlices = 16;                 // score accumulators
constexpr int kPjAccCols = 256;                  // one accumulator
constexpr int kPjTmemCols = 2 * kPjAccCols;      // two, all of the SM's tensor memory
constexpr size_t kPjSmem = 1024 + (size_t)kPjStages * kPjStageBytes + 256;
// More than half of an SM's shared memory: one CTA per SM, so the 512
// tensor-memory columns it allocates are always free.
static_assert(kPjSmem > 114 * 1024, "one projection CTA per SM");

__device__ __forceinline__ unsigned int pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<unsigned int*>(&h);
}

__global__ void __launch_bounds__(kPjThreads, 1)
proj_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               const __grid_constant__ CUtensorMap tmA, __nv_bfloat16* __restrict__ V,
               float2* __restrict__ z2, int Mtot, int N, int D, int H, int ntiles,
               unsigned int* status) {
  extern __shared__ unsigned char pj_raw[];
  const uint32_t raw = smem_addr(pj_raw);
  unsigned char* sm = pj_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kPjStages * kPjStageBytes);
  uint64_t* empty = full + kPjStages;
  uint64_t* tfull = empty + kPjStages;     // [2] accumulator b holds a finished tile
  uint64_t* tempty = tfull + 2;            // [2] accumulator b has been read back
  uint64_t* done = tempty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvt = (D + kPjNV - 1) / kPjNV;
  const int nt = nvt + 1;                   // value tiles, then the score tile
  const int nks = D / kPjK;
  const int per_slice = (nks + kPjMaxSlices - 1) / kPjMaxSlices;   // K steps per score slice

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPjStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 4);
    }
    mbar_init(done, 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tslot, kPjTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // Tensor copies: stage g % kPjStages once the MMAs of its previous use
    // have completed (g counts the K steps of all this CTA's tiles).
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int m0 = (t / nt) * kPjM, nti = t % nt;
        const bool ztile = nti == nvt;
        const uint32_t wbytes = (ztile ? kPjNZ : kPjNV) * kPjK * 2;
        for (int s = 0; s < nks; ++s, ++g) {
          const int st = g % kPjStages;
          if (g >= kPjStages && !mbar_wait(empty + st, ((g / kPjStages) - 1) & 1, status, 0x601)) {
            ok = false;
            break;
          }
          unsigned char* xs = sm + st * kPjStageBytes;
          mbar_expect_tx(full + st, kPjXBytes + wbytes);
          tma_load_2d(xs, &tmX, s * kPjK, m0, full + st);
          if (ztile)
            tma_load_2d(xs + kPjXBytes, &tmA, s * kPjK, 0, full + st);
          else
            tma_load_2d(xs + kPjXBytes, &tmW, s * kPjK, nti * kPjNV, full + st);
        }
      }
    }
  } else if (warp == 1) {
    // MMA issue: four K = 16 MMAs per stage from one thread, into the
    // accumulator of the tile's parity.
    int g = 0, it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
      const int nti = t % nt;
      const bool ztile = nti == nvt;
      const int NT = ztile ? kPjNZ : min(kPjNV, D - nti * kPjNV);
      const uint32_t idesc = idesc_bf16_f32(kPjM, NT);
      const int b = it & 1;
      // Lane 0 waits and issues; the warp follows its result, so that the
      // whole warp leaves a loop together.
      bool w = true;
      if (it >= 2 && lane == 0) w = mbar_wait(tempty + b, ((it >> 1) - 1) & 1, status, 0x605);
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      tc_fence_after();
      const uint32_t acc0 = tmem + (uint32_t)(b * kPjAccCols);
      for (int s = 0; s < nks; ++s, ++g) {
        const int st = g % kPjStages;
        w = true;
        if (lane == 0) w = mbar_wait(full + st, (g / kPjStages) & 1, status, 0x602);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const unsigned char* xs = sm + st * kPjStageBytes;
          const uint32_t d = ztile ? acc0 + kPjNZ * (uint32_t)(s / per_slice) : acc0;
#pragma unroll
          for (int k = 0; k < kPjK / 16; ++k) {
            const uint32_t acc = ztile ? (k > 0 || s % per_slice != 0) : (k > 0 || s > 0);
            tc_mma_bf16(d, sdesc_k128(xs + 32 * k), sdesc_k128(xs + kPjXBytes + 32 * k), idesc,
                        acc);
          }
          tc_commit(empty + st);
        }
        __syncwarp();
      }
      if (ok && lane == 0) tc_commit(tfull + b);
      __syncwarp();
    }
    if (lane == 0) tc_commit(done);
    __syncwarp();
  } else {
    // Epilogue: the four warps cover the 128 lanes by quadrant (warp % 4).
    const int q = warp & 3;
    int it = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
      const int m0 = (t / nt) * kPjM, nti = t % nt;
      const bool ztile = nti == nvt;
      const int n0 = nti * kPjNV;
      const int NT = ztile ? kPjNZ : min(kPjNV, D - n0);
      const int b = it & 1;
      // The tensor-memory loads are warp-wide: the warp goes on only if
      // every lane saw the accumulator full.
      if (!__all_sync(0xffffffffu, mbar_wait(tfull + b, (it >> 1) & 1, status, 0x603))) break;
      tc_fence_after();
      const int row = m0 + 32 * q + lane;
      const uint32_t taddr = tmem + (uint32_t)(b * kPjAccCols) + ((uint32_t)(32 * q) << 16);
      if (!ztile) {
        __nv_bfloat16* dst = V + (size_t)row * D + n0;
        for (int c0 = 0; c0 < NT; c0 += 16) {
          float v[16];
          tc_ld16(taddr + c0, v);
          if (row < Mtot) {
            uint4 a, c;
            a.x = pack_bf16x2(v[0], v[1]);   a.y = pack_bf16x2(v[2], v[3]);
            a.z = pack_bf16x2(v[4], v[5]);   a.w = pack_bf16x2(v[6], v[7]);
            c.x = pack_bf16x2(v[8], v[9]);   c.y = pack_bf16x2(v[10], v[11]);
            c.z = pack_bf16x2(v[12], v[13]); c.w = pack_bf16x2(v[14], v[15]);
            reinterpret_cast<uint4*>(dst + c0)[0] = a;
            reinterpret_cast<uint4*>(dst + c0)[1] = c;
          }
        }
      } else {
        float hi[16], lo[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) hi[h] = lo[h] = 0.f;
        const int nsl = (nks + per_slice - 1) / per_slice;
        for (int c = 0; c < nsl; ++c) {
          float v[16];
          tc_ld16(taddr + kPjNZ * c, v);
#pragma unroll
          for (int h = 0; h < 16; ++h) two_sum_acc(hi[h], lo[h], v[h]);
        }
        if (row < Mtot) {
          const int bb = row / N, n = row - bb * N;
#pragma unroll
          for (int h = 0; h < 16; ++h)
            if (h < H) z2[((size_t)bb * H + h) * N + n] = make_float2(hi[h], lo[h]);
        }
      }
      // This warp's reads of the accumulator are complete (tc_ld16 waits):
      // hand it back to the MMA warp.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + b);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // The columns are freed only after every MMA has completed (bounded).
    mbar_wait(done, 0, status, 0x604);
    tc_fence_after();
    tmem_dealloc(tmem, kPjTmemCols);
  }
}

// Wt[n][k] = W_V[k][n] (D x D) and At[h][k] = W_A[k][h] for h < H, zero for
// H <= h < 16: the B operands of the projection, K-major.
__global__ void proj_transpose_kernel(const __nv_bfloat16* __restrict__ WV,
                                      const __nv_bfloat16* __restrict__ WA,
                                      __nv_bfloat16* __restrict__ Wt, __nv_bfloat16* __restrict__ At,
                                      int D, int H) {
  __shared__ __nv_bfloat16 t[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int nb = (D + 31) / 32;
  if ((int)blockIdx.x < nb * nb) {
    const int bk = blockIdx.x / nb, bn = blockIdx.x % nb;
    for (int r = ty; r < 32; r += 8) {
      const int k = bk * 32 + r, n = bn * 32 + tx;
      t[r][tx] = (k < D && n < D) ? WV[(size_t)k * D + n] : __float2bfloat16(0.f);
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
      const int n = bn * 32 + r, k = bk * 32 + tx;
      if (n < D && k < D) Wt[(size_t)n * D + k] = t[tx][r];
    }
  } else {
    for (int i = (blockIdx.x - nb * nb) * blockDim.x + threadIdx.x; i < kPjNZ * D;
         i += (gridDim.x - nb * nb) * blockDim.x) {
      const int h = i / D, k = i - h * D;
      At[i] = h < H ? WA[(size_t)k * H + h] : __float2bfloat16(0.f);
    }
  }
}

size_t project_workspace_bytes(int D) { return ((size_t)D * D + (size_t)kPjNZ * D) * 2; }

cudaError_t setup_project_kernels() {
  return cudaFuncSetAttribute(proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kPjSmem);
}

cudaError_t launch_project(const cat_plan_s* p, const void* X, const void* WV, const void* WA,
                           void* V, void* wt) {
  const int D = p->D;
  const long long Mtot = (long long)p->B * p->N;
  __nv_bfloat16* Wt = static_cast<__nv_bfloat16*>(wt);
  __nv_bfloat16* At = Wt + (size_t)D * D;
  const int nb = (D + 31) / 32;
  proj_transpose_kernel<<<nb * nb + 16, 256, 0, p->stream>>>(
      static_cast<const __nv_bfloat16*>(WV), static_cast<const __nv_bfloat16*>(WA), Wt, At, D,
      p->H);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tmX, tmW, tmA;
  if (!encode_map_2d_sw128(&tmX, X, D, (unsigned long long)Mtot, (unsigned long long)D * 2, kPjK,
                           kPjM) ||
      !encode_map_2d_sw128(&tmW, Wt, D, D, (unsigned long long)D * 2, kPjK, kPjNV) ||
      !encode_map_2d_sw128(&tmA, At, D, kPjNZ, (unsigned long long)D * 2, kPjK, kPjNZ))
    return cudaErrorInvalidValue;
  // Tiles ordered token block first (value tiles, then the score tile of
  // each block); one persistent CTA per SM, never more CTAs than tiles.
  const long long ntiles = ((Mtot + kPjM - 1) / kPjM) * ((D + kPjNV - 1) / kPjNV + 1);
  const int grid = (int)(ntiles < p->sms ? ntiles : p->sms);
  proj_tc_kernel<<<grid, kPjThreads, kPjSmem, p->stream>>>(
      tmX, tmW, tmA, static_cast<__nv_bfloat16*>(V), p->z2, (int)Mtot, p->N, D, p->H,
      (int)ntiles, p->status);
  return cudaGetLastError();
}

}  // namespace cat
