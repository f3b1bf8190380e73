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
// O and the scratch is a contiguous run of the head's row; in passes A and C
// consecutive CTAs take consecutive heads of the same rows, so the rows of
// V and O stream through DRAM whole.
//
// Within a pass each thread holds 32 values in registers and the transform
// is a sequence of Stockham steps (radix R, span Ls; task i takes the
// inputs i + u·L/R, twiddles them by w_{R·Ls}^{u·(i mod Ls)}, and writes
// the R outputs (i / Ls)·R·Ls + (i mod Ls) + s·Ls).  Between steps the
// values go through shared memory; the last forward step leaves each thread
// holding exactly the bins the first inverse step needs, so pass B takes
// the product and starts the inverse without touching shared memory.
//
// The spectrum of z* is computed once per (b, h) — by zspec_row, one CTA per
// row, for N2 = 32; by zspec_a/zspec_b for longer rows — with the same
// register transforms, and stored in the order pass B's threads hold
// the bins: thread j of the CTA for k2 holds k1 = 2j + e + 32s (e < 2,
// s < 16), stored at ((k2·16 + j)·16 + s)·2 + e.
#include <cuda_bf16.h>

#include "bulk.cuh"
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
// Pass A for N2 > 32 (N2 = 32 takes the pipelined fsf_pass_a32 below): a
// CTA per n1, T = N2/32 warps; step 1 (radix 32, span 1) then step 2 (radix
// N2/32, span 32) with thread j taking the tasks per·j + e, per = 32/T.
// ---------------------------------------------------------------------------
template <typename T, int N2>
__global__ void __launch_bounds__(256)
fsf_pass_a(const T* __restrict__ V0, float2* __restrict__ scr0, const float2* __restrict__ W,
           const float2* __restrict__ tf, int N, int D, int H, int bh0, int nb,
           const T* __restrict__ V1 = nullptr, float2* __restrict__ scr1 = nullptr,
           int early = 0) {
  // W: w_N^m (the row twiddles w_N^{n1·k2}); tf[k][u] = w_512^{u·k}, whose
  // entry (k, (16 / R2)·u) is the step-2 twiddle w_N2^{u·k} (a 4 KB table
  // that stays in L1).
  static_assert(N2 > 32, "N2 = 32 takes fsf_pass_a32");
  if (early) pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // With V1, the grid is doubled and its second half transforms V1 into scr1
  // (the backward's correlation transforms dO and V in one launch).
  const int half = nb * kFastN1;
  const bool second = V1 != nullptr && (int)blockIdx.x >= half;
  const int bid = (int)blockIdx.x - (second ? half : 0);
  const T* V = second ? V1 : V0;
  float2* scr = second ? scr1 : scr0;
  {
    constexpr int TS = N2 / 32;        // threads per signal
    constexpr int R2 = N2 / 32;        // radix of step 2
    constexpr int PER = 32 / TS;       // step-2 tasks per thread
    constexpr int RS = N2 + 2;         // shared row of one pair
    extern __shared__ float4 smem4[];
    float2* buf = reinterpret_cast<float2*>(smem4);
    const int j = warp;
    const int n1 = bid / nb;
    const int bhl = bid % nb;
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
    // The scratch is read again by passes B and C: keep it in L2.
    const uint64_t keep = policy_evict_last();
    // Launched as a dependent of the previous chunk's pass C, which reads
    // the scratch slot this pass overwrites.
    pdl_wait();
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int k = PER * j + e;
#pragma unroll
      for (int u = 1; u < R2; ++u) c[e][u] = cmul(c[e][u], __ldg(&tf[k * 16 + (16 / R2) * u]));
      dft<R2, false>(c[e]);
#pragma unroll
      for (int s = 0; s < R2; ++s) {
        const int k2 = k + 32 * s;
        st_hint(scr + scr_idx(bhl, N2, k2, n1, lane), cmul(c[e][s], __ldg(&W[(size_t)n1 * k2])),
                keep);
      }
    }
  }
  if (!early) pdl_trigger();
}

// Two storage elements (one packed pair) read from shared memory.
__device__ __forceinline__ float2 sh_pair(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
__device__ __forceinline__ float2 sh_pair(const __nv_bfloat16* p) {
  unsigned int u = *reinterpret_cast<const unsigned int*>(p);
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// ---------------------------------------------------------------------------
// Pass A for N2 > 32, persistent and fed by tensor copies: each CTA takes
// items (b, h, n1) in turn (item, item + grid, ...).  An item's V tile — the
// N2 rows n1 + 512·n2 of the head's 64 columns — arrives by one tensor copy
// into shared memory; as soon as every thread holds its 32 values, the next
// item's copy is issued into the same buffer, so it loads while this item
// is transformed.  The transform is fsf_pass_a's (step 1 radix 32, step 2
// radix N2/32), with the step-2 twiddles in a shared table and the row
// w_N^{n1·k2} fetched once per item (one value a thread).  ntens = 2: a
// second tensor (tmV2 into scr2), its items after the first's.
// ---------------------------------------------------------------------------
template <typename T, int N2>
struct PipeAT {
  static constexpr int kTile = N2 * 64 * (int)sizeof(T);            // one V tile
  static constexpr int kOffTile = 1024;
  static constexpr int kOffTw2 = kOffTile + kTile;                   // [R2][32]
  static constexpr int kOffTwRow = kOffTw2 + (N2 / 32) * 32 * 8;     // [N2]
  static constexpr int kOffBuf = kOffTwRow + N2 * 8;                 // [32][N2 + 2]
  static constexpr size_t kSmem = (size_t)kOffBuf + (size_t)kFastPairs * (N2 + 2) * 8;
};

template <typename T, int N2>
__global__ void __launch_bounds__(N2, 2)
fsf_pass_a_tma(const __grid_constant__ CUtensorMap tmV, float2* __restrict__ scr,
               const float2* __restrict__ W, int N, int D, int H, int bh0, int nb,
               unsigned int* status, const __grid_constant__ CUtensorMap tmV2,
               float2* __restrict__ scr2, int ntens, int early) {
  static_assert(N2 > 32 && N2 <= 256, "N2 = 32 takes fsf_pass_a32");
  using P = PipeAT<T, N2>;
  constexpr int TS = N2 / 32;        // warps; threads per signal
  constexpr int R2 = N2 / 32;        // radix of step 2
  constexpr int PER = 32 / TS;       // step-2 tasks per thread
  constexpr int RS = N2 + 2;         // shared row of one pair
  if (early) pdl_trigger();
  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm);
  const T* tile = reinterpret_cast<const T*>(sm + P::kOffTile);
  float2* tw2 = reinterpret_cast<float2*>(sm + P::kOffTw2);
  float2* twrow = reinterpret_cast<float2*>(sm + P::kOffTwRow);
  float2* buf = reinterpret_cast<float2*>(sm + P::kOffBuf);
  const int t = threadIdx.x, lane = t & 31, j = t >> 5;
  const int items1 = nb * kFastN1, items = ntens * items1;
  const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
  auto issue = [&](int item) {
    fence_proxy_async_smem();   // the CTA's reads of the tile come first
    const int second = item >= items1, it1 = item - second * items1;
    const int bh = bh0 + it1 % nb, n1 = it1 / nb;
    const int b = bh / H, h = bh - b * H;
    mbar_expect_tx(bar, P::kTile);
    tma_load_4d_hint(sm + P::kOffTile, second ? &tmV2 : &tmV, h * 64, n1, 0, b, bar, stream);
  };
  if (t == 0) mbar_init(bar, 1);
  mbar_fence_init();
  {
    const int wstep = N / N2;
    for (int i = t; i < R2 * 32; i += N2) tw2[i] = W[(size_t)((i / 32) * (i % 32)) * wstep];
  }
  __syncthreads();
  if (t == 0 && (int)blockIdx.x < items) issue(blockIdx.x);
  // Launched as a dependent of the previous chunk's pass C, which reads the
  // scratch slot this pass overwrites: the first tile loads meanwhile.
  pdl_wait();
  float2* row = buf + lane * RS;
  int it = 0;
  for (int item = blockIdx.x; item < items; item += gridDim.x, ++it) {
    const bool ok = mbar_wait(bar, it & 1, status, 0x503);
    if (__syncthreads_or(!ok)) return;
    const int second = item >= items1, it1 = item - second * items1;
    float2* dst = second ? scr2 : scr;
    const int bhl = it1 % nb, n1 = it1 / nb;
    const float2 tw = __ldg(&W[(size_t)n1 * t]);   // w_N^{n1·k2}, k2 = t
    float2 a[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) a[u] = sh_pair(tile + (j + TS * u) * 64 + 2 * lane);
    __syncthreads();   // the tile is read; the previous item's row reads are done
    if (t == 0 && item + (int)gridDim.x < items) issue(item + gridDim.x);
    dft<32, false, CxPaired>(a);
#pragma unroll
    for (int q = 0; q < 32; q += 2) st_sh2(row + 32 * j + q, a[q], a[q + 1]);
    twrow[t] = tw;
    __syncthreads();
    float2 c[PER][R2];
#pragma unroll
    for (int u = 0; u < R2; ++u)
#pragma unroll
      for (int e = 0; e < PER; e += 2) ld_sh2(row + PER * j + e + 32 * u, c[e][u], c[e + 1][u]);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int k = PER * j + e;
#pragma unroll
      for (int u = 1; u < R2; ++u) c[e][u] = cmul(c[e][u], tw2[u * 32 + k]);
      dft<R2, false, CxPaired>(c[e]);
#pragma unroll
      for (int q = 0; q < R2; ++q) {
        const int k2 = k + 32 * q;
        st_hint(dst + scr_idx(bhl, N2, k2, n1, lane), cmul(c[e][q], twrow[k2]), keep);
      }
    }
  }
  if (!early) pdl_trigger();
}

// ---------------------------------------------------------------------------
// Pass C: the inverse of pass A's transform over k2, then the output rows.
// ---------------------------------------------------------------------------
template <typename T, int N2>
__global__ void __launch_bounds__(256)
fsf_pass_c(const float2* scr, T* __restrict__ O, const float2* __restrict__ tf, int N, int D,
           int H, int bh0, int nb, int early = 0) {
  // tf[k][u] = w_512^{u·k}: entry (k, (16 / R2)·u) is the step-2 twiddle.
  static_assert(N2 > 32, "N2 = 32 takes fsf_pass_c32");
  if (early) pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    constexpr int TS = N2 / 32;
    constexpr int R2 = N2 / 32;
    constexpr int PER = 32 / TS;
    constexpr int RS = N2 + 2;
    extern __shared__ float4 smem4[];
    float2* buf = reinterpret_cast<float2*>(smem4);
    const int j = warp;
    const int n1 = blockIdx.x / nb;
    const int bhl = blockIdx.x % nb;
    const int bh = bh0 + bhl, b = bh / H, h = bh - b * H;
    float2 a[32];
    pdl_wait();   // pass B ahead on the stream wrote the scratch
#pragma unroll
    for (int u = 0; u < 32; ++u) a[u] = ld_dep(scr + scr_idx(bhl, N2, j + TS * u, n1, lane));
    dft<32, true>(a);
    float2* row = buf + lane * RS;
#pragma unroll
    for (int s = 0; s < 32; s += 2) st_sh2(row + 32 * j + s, a[s], a[s + 1]);
    __syncthreads();
    {
      // Every thread has its values: the CTA's N2 scratch rows (k2, n1) are
      // dead, so their two 128-byte lines each leave L2 without a
      // write-back (the next chunk's pass A rewrites them first).
      const float2* r = scr + scr_idx(bhl, N2, threadIdx.x, n1, 0);
      discard_l2(r);
      discard_l2(r + 16);
    }
    float2 c[PER][R2];
#pragma unroll
    for (int u = 0; u < R2; ++u)
#pragma unroll
      for (int e = 0; e < PER; e += 2) ld_sh2(row + PER * j + e + 32 * u, c[e][u], c[e + 1][u]);
    T* dst = O + ((size_t)b * N + n1) * D + h * 64 + 2 * lane;
    const size_t rs = (size_t)kFastN1 * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int k = PER * j + e;
#pragma unroll
      for (int u = 1; u < R2; ++u) c[e][u] = cmulc(c[e][u], __ldg(&tf[k * 16 + (16 / R2) * u]));
      dft<R2, true>(c[e]);
#pragma unroll
      for (int s = 0; s < R2; ++s) st_pair(dst + (size_t)(k + 32 * s) * rs, c[e][s]);
    }
  }
  if (!early) pdl_trigger();
}


// ---------------------------------------------------------------------------
// Pipelined passes A and C for N2 == 32.  Every warp runs its own pipeline
// over work items (b, h, n1) — heads fastest — with STAGES shared-memory
// stages: the tile of an item (32 rows n1 + 512·n2 of the head, or 32 scratch
// rows) arrives by one tensor copy (TMA) completing on the stage's mbarrier,
// so the next items' loads are in flight while the current item is
// transformed.
// ---------------------------------------------------------------------------
constexpr int kPipeWarps = 8;

template <typename T>
struct PipeA {
  static constexpr int kRowBytes = 64 * (int)sizeof(T);   // one head row of V
  static constexpr int kStages = sizeof(T) == 2 ? 3 : 2;
  static constexpr size_t kSmem = 2304 + (size_t)kPipeWarps * kStages * 32 * kRowBytes;
};
struct PipeC {
  static constexpr int kRowBytes = kFastPairs * 8;         // one scratch row (32 pairs)
  static constexpr int kWarps = 4;
  static constexpr int kStages = 3;
  static constexpr size_t kSmem = 256 + (size_t)kWarps * kStages * 32 * kRowBytes;
};

template <typename T>
__global__ void __launch_bounds__(kPipeWarps * 32)
fsf_pass_a32(const __grid_constant__ CUtensorMap tmV, float2* __restrict__ scr,
             const float2* __restrict__ W, int N, int D, int H, int bh0, int nb,
             unsigned int* status, const __grid_constant__ CUtensorMap tmV2,
             float2* __restrict__ scr2, int ntens, int early) {
  // ntens = 2: a second tensor (tmV2 into scr2) in the same launch, its
  // items after the first's (the backward's correlation transforms dO and V
  // together).
  if (early) pdl_trigger();
  using P = PipeA<T>;
  extern __shared__ __align__(128) unsigned char sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm) + warp * P::kStages;
  unsigned char* stage = sm + 2304 + (size_t)warp * P::kStages * 32 * P::kRowBytes;
  float2* twrow = reinterpret_cast<float2*>(sm + 256) + warp * 32;   // 256 B per warp
  if (lane == 0)
    for (int s = 0; s < P::kStages; ++s) mbar_init(bar + s, 1);
  mbar_fence_init();
  __syncwarp();
  const int gw = blockIdx.x * kPipeWarps + warp, G = gridDim.x * kPipeWarps;
  const int items1 = nb * kFastN1, items = ntens * items1;
  const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
  auto issue = [&](int s, int item) {
    if (lane == 0) {
      fence_proxy_async_smem();   // the warp's reads of this stage come first
      const int second = item >= items1, it1 = item - second * items1;
      const int bh = bh0 + it1 % nb, n1 = it1 / nb;
      const int b = bh / H, h = bh - b * H;
      mbar_expect_tx(bar + s, 32 * P::kRowBytes);
      tma_load_4d_hint(stage + s * 32 * P::kRowBytes, second ? &tmV2 : &tmV, h * 64, n1, 0, b,
                       bar + s, stream);
    }
  };
#pragma unroll
  for (int k = 0; k < P::kStages; ++k)
    if (gw + k * G < items) issue(k, gw + k * G);
  // Launched as a dependent of the previous chunk's pass C, which reads the
  // scratch slot this pass overwrites: the first tiles load meanwhile.
  pdl_wait();
  int it = 0;
  for (int item = gw; item < items; item += G, ++it) {
    const int s = it % P::kStages;
    if (!mbar_wait(bar + s, (it / P::kStages) & 1, status, 0x501)) return;
    const int second = item >= items1, it1 = item - second * items1;
    float2* dst = second ? scr2 : scr;
    const int bhl = it1 % nb, n1 = it1 / nb;
    const float2 tw = __ldg(&W[(size_t)n1 * lane]);   // w_N^{n1·k2} for k2 = lane
    const T* tile = reinterpret_cast<const T*>(stage + s * 32 * P::kRowBytes) + 2 * lane;
    float2 a[32];
#pragma unroll
    for (int n2 = 0; n2 < 32; ++n2) a[n2] = sh_pair(tile + n2 * 64);
    dft<32, false, CxPaired>(a);
    __syncwarp();
    const int next = item + P::kStages * G;
    if (next < items) issue(s, next);
    twrow[lane] = tw;
    __syncwarp();
#pragma unroll
    for (int k2 = 0; k2 < 32; ++k2)
      st_hint(dst + scr_idx(bhl, 32, k2, n1, lane), cmul(a[k2], twrow[k2]), keep);
    __syncwarp();
  }
  if (!early) pdl_trigger();
}

template <typename T>
__global__ void __launch_bounds__(PipeC::kWarps * 32)
fsf_pass_c32(const __grid_constant__ CUtensorMap tmC, const float2* __restrict__ scr,
             T* __restrict__ O, int N, int D, int H, int bh0, int nb, unsigned int* status,
             int early, int row_off) {
  // row_off: the chunk's first row in tmC (scr points at that row).
  if (early) pdl_trigger();
  using P = PipeC;
  extern __shared__ __align__(128) unsigned char sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm) + warp * P::kStages;
  unsigned char* stage = sm + 256 + (size_t)warp * P::kStages * 32 * P::kRowBytes;
  if (lane == 0)
    for (int s = 0; s < P::kStages; ++s) mbar_init(bar + s, 1);
  mbar_fence_init();
  __syncwarp();
  const int gw = blockIdx.x * P::kWarps + warp, G = gridDim.x * P::kWarps;
  const int items = nb * kFastN1;
  auto issue = [&](int s, int item) {
    if (lane == 0) {
      fence_proxy_async_smem();   // the warp's reads of this stage come first
      mbar_expect_tx(bar + s, 32 * P::kRowBytes);
      tma_load_4d(stage + s * 32 * P::kRowBytes, &tmC, 0, item / nb, 0, row_off + item % nb,
                  bar + s);
    }
  };
  pdl_wait();   // pass B ahead on the stream wrote the scratch
#pragma unroll
  for (int k = 0; k < P::kStages; ++k)
    if (gw + k * G < items) issue(k, gw + k * G);
  int it = 0;
  for (int item = gw; item < items; item += G, ++it) {
    const int s = it % P::kStages;
    if (!mbar_wait(bar + s, (it / P::kStages) & 1, status, 0x502)) return;
    const float2* tile = reinterpret_cast<const float2*>(stage + s * 32 * P::kRowBytes) + lane;
    float2 a[32];
#pragma unroll
    for (int k2 = 0; k2 < 32; ++k2) a[k2] = tile[k2 * kFastPairs];
    dft<32, true, CxPaired>(a);
    __syncwarp();
    const int next = item + P::kStages * G;
    if (next < items) issue(s, next);
    {
      // The item's 32 scratch rows (256 B = two lines each) are dead now:
      // drop them from L2 without a write-back.
      const float2* r = scr + scr_idx(item % nb, 32, lane, item / nb, 0);
      discard_l2(r);
      discard_l2(r + 16);
    }
    const int bh = bh0 + item % nb, n1 = item / nb;
    const int b = bh / H, h = bh - b * H;
    T* dst = O + ((size_t)b * N + n1) * D + h * 64 + 2 * lane;
    const size_t rs = (size_t)kFastN1 * D;
#pragma unroll
    for (int n2 = 0; n2 < 32; ++n2) st_pair(dst + n2 * rs, a[n2]);
  }
  if (!early) pdl_trigger();
}

// ---------------------------------------------------------------------------
// Pass B: per (b, h, k2) and a group of kBPairs of the head's pairs (signals
// of length 512, 16 threads each).  Forward: step F1 (radix 32, span 1; thread j task j), step F2
// (radix 16, span 32; tasks 2j, 2j+1).  Product with the spectrum of z*.
// Inverse: step I1 (radix 16, span 1; tasks 2j, 2j+1 — exactly the bins the
// thread holds), step I2 (radix 32, span 16; task j), leaving n1 = j + 16s.
// Lane l: pair l mod kBPairs of the group, j = (32/kBPairs)·warp + l/kBPairs.
// Everything the compute steps read besides the exchange buffer — the
// length-512 twiddles, the row w_N^{n1·k2} and the spectrum of z* at this
// k2 — is loaded into shared memory at the start, together with the 32
// scratch values, so no global load waits inside the transforms.
// ---------------------------------------------------------------------------
constexpr int kBPairs = 16;  // pairs (signals) per pass-B CTA; 16 threads each
// Shared tables of pass B, all in the order the threads read them (float2):
//   tf[k][u]  = w_512^{u·k}           k < 32, u < 16   (step F2)
//   ti[j][u]  = w_512^{u·j}           j < 16, u < 32   (step I2, conjugated)
//   tx[j][q]  = w_N^{(j+16q)·k2}      j < 16, q < 32   (inter-pass, conjugated)
//   zf[j][q][e] = FFT(z*)/N at k1 = 2j + e + 32q       (the product)
// tf and ti are the same for every CTA and tx for every CTA of one k2; the
// plan builds them once (fast_tables).  Each is 4 KB.
constexpr int kTabB = 512;   // complex entries per table
constexpr size_t kSmemB =
    (size_t)kBPairs * kRowB * sizeof(float2) + 4 * kTabB * sizeof(float2);

__global__ void __launch_bounds__(kBPairs * 16, 2)
fsf_pass_b(float2* __restrict__ scr, const float2* __restrict__ zft,
           const float2* __restrict__ tabs, int N2, int bh0, int early, int conj) {
  if (early) pdl_trigger();
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  float2* tf = buf + kBPairs * kRowB;
  float2* ti = tf + kTabB;
  float2* tx = ti + kTabB;
  float2* zf = tx + kTabB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pl = lane & (kBPairs - 1);
  const int j = (32 / kBPairs) * warp + lane / kBPairs;
  constexpr int G = kFastPairs / kBPairs;     // CTAs per (b, h, k2)
  const int grp = blockIdx.x % G;
  const int k2 = (blockIdx.x / G) % N2;
  const int bhl = (blockIdx.x / G) / N2;
  const int pair = grp * kBPairs + pl;
  float2* row = buf + pl * kRowB;

  const uint64_t keep = policy_evict_last();
  // Tables: 4 x 4 KB, one 16-byte load of each per thread (256 threads).
  // The plan's tables are loaded before the wait for pass A (this launch may
  // be its programmatic dependent); the spectrum of z* was complete before
  // the stream's first pass B started.
  const int t = threadIdx.x;
  const float4* g4 = reinterpret_cast<const float4*>(tabs);
  const float4 q0 = __ldg(g4 + t);                                   // tf, ti
  const float4 q1 = __ldg(g4 + 256 + t);
  const float4 q2 = __ldg(g4 + 512 + (size_t)k2 * 256 + t);          // tx of this k2
  float4 q3 = __ldg(reinterpret_cast<const float4*>(zft) +
                    ((size_t)(bh0 + bhl) * N2 + k2) * (kFastN1 / 2) + t);
  if (conj) {   // conj(FFT(z*)): the spectrum of the reversed z* (dV of the backward)
    q3.y = -q3.y;
    q3.w = -q3.w;
  }
  pdl_wait();
  float2 a[32];
#pragma unroll
  for (int u = 0; u < 32; ++u) a[u] = ld_hint(scr + scr_idx(bhl, N2, k2, j + 16 * u, pair), keep);
  dft<32, false, CxPaired>(a);
#pragma unroll
  for (int q = 0; q < 32; q += 2) st_sh2(row + 32 * j + q, a[q], a[q + 1]);
  float4* tf4 = reinterpret_cast<float4*>(tf);
  tf4[t] = q0;
  tf4[256 + t] = q1;
  tf4[512 + t] = q2;
  tf4[768 + t] = q3;
  __syncthreads();

  float2 c[2][16];
#pragma unroll
  for (int u = 0; u < 16; ++u) ld_sh2(row + 2 * j + 32 * u, c[0][u], c[1][u]);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float2* tw = tf + (2 * j + e) * 16;
#pragma unroll
    for (int u = 2; u < 16; u += 2) {
      float2 w0, w1;
      ld_sh2(tw + u, w0, w1);
      c[e][u] = cmul(c[e][u], w0);
      c[e][u + 1] = cmul(c[e][u + 1], w1);
    }
    c[e][1] = cmul(c[e][1], tw[1]);
    dft<16, false, CxPaired>(c[e]);
  }
  // Product with FFT(z*)/N at bins k1 = 2j + e + 32s.
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    float2 z0, z1;
    ld_sh2(zf + (j * 16 + q) * 2, z0, z1);
    c[0][q] = cmul(c[0][q], z0);
    c[1][q] = cmul(c[1][q], z1);
  }
  __syncthreads();
  // Inverse step I1 writes position p = 32j + 16e + s to storage
  // 32·(p mod 16) + p / 16 = 32s + 2j + e, so that I2's 32 inputs
  // (positions j + 16u) sit at 32j + u: both sides move 16-byte pairs.
#pragma unroll
  for (int e = 0; e < 2; ++e) dft<16, true, CxPaired>(c[e]);
#pragma unroll
  for (int q = 0; q < 16; ++q) st_sh2(row + 32 * q + 2 * j, c[0][q], c[1][q]);
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 32; u += 2) ld_sh2(row + 32 * j + u, a[u], a[u + 1]);
  {
    const float2* tw = ti + j * 32;
#pragma unroll
    for (int u = 2; u < 32; u += 2) {
      float2 w0, w1;
      ld_sh2(tw + u, w0, w1);
      a[u] = cmulc(a[u], w0);
      a[u + 1] = cmulc(a[u + 1], w1);
    }
    a[1] = cmulc(a[1], tw[1]);
  }
  dft<32, true, CxPaired>(a);
  {
    const float2* tw = tx + j * 32;
#pragma unroll
    for (int q = 0; q < 32; q += 2) {
      float2 w0, w1;
      ld_sh2(tw + q, w0, w1);
      st_hint(scr + scr_idx(bhl, N2, k2, j + 16 * q, pair), cmulc(a[q], w0), keep);
      st_hint(scr + scr_idx(bhl, N2, k2, j + 16 * (q + 1), pair), cmulc(a[q + 1], w1), keep);
    }
  }
  if (!early) pdl_trigger();
}


// ---------------------------------------------------------------------------
// Backward correlation, pass B (the fast path's layout; see backward.cu for
// the method): per (b, h, k2), the length-512 DFTs over n1 of the head's 32
// dO pairs (scratch slot 0) and 32 V pairs (slot 1), both after pass A; the
// sum over pairs of FFT(g)·conj(FFT(v)) at every bin k1; the inverse DFT over
// k1 of that one signal; the conjugate twiddle w_N^{-n1 k2}; into
// y[bhl][k2][n1].  256 threads: signal sig = lane mod 16 (0..7 dO, 8..15 V;
// pairs sig mod 8 + 8r in round r), j = 2·warp + lane / 16, with pass B's
// forward steps F1, F2 (thread j then holds bins k1 = 2j + e + 32q).  The V
// threads hand their bins over through shared memory, the dO threads keep
// running sums; the 8 sums are added in a fixed order and one warp runs
// pass B's inverse steps I1, I2 on the result.  The running sums live in
// shared memory (rows of kRowB per signal, at the position the thread's bins
// take in the exchange rows), so that two CTAs fit an SM.
// ---------------------------------------------------------------------------
constexpr size_t kSmemCorrB =
    (size_t)16 * kRowB * sizeof(float2) + kTabB * sizeof(float2) + 8 * (size_t)kRowB * sizeof(float2);

__global__ void __launch_bounds__(256, 2)
fsf_corr_b(const float2* __restrict__ scrG, const float2* __restrict__ scrV,
           float2* __restrict__ y, const float2* __restrict__ tabs, int N2) {
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  float2* tf = buf + 16 * kRowB;
  float2* accs = tf + kTabB;           // [8][kRowB] running sums of the dO threads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sig = lane & 15;
  const int j = 2 * warp + (lane >> 4);
  const int k2 = blockIdx.x % N2;
  const int bhl = blockIdx.x / N2;
  const float2* src = sig < 8 ? scrG : scrV;
  float2* row = buf + sig * kRowB;
  // This thread's 32 bins; rows kRowB apart put the 8 signals of a quarter
  // warp in distinct 16-byte bank groups.
  float2* acc = accs + (sig & 7) * kRowB + j * 32;
  {
    const int t = threadIdx.x;
    const float4* g4 = reinterpret_cast<const float4*>(tabs);
    float4* tf4 = reinterpret_cast<float4*>(tf);
    tf4[t] = __ldg(g4 + t);
    float4* a4 = reinterpret_cast<float4*>(accs);
    for (int i = t; i < 8 * kRowB / 2; i += 256) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  for (int r = 0; r < kFastPairs / 8; ++r) {
    const int pair = 8 * r + (sig & 7);
    float2 a[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) a[u] = src[scr_idx(bhl, N2, k2, j + 16 * u, pair)];
    dft<32, false, CxPaired>(a);
    __syncthreads();   // the previous round's reads of the rows are done
#pragma unroll
    for (int q = 0; q < 32; q += 2) st_sh2(row + 32 * j + q, a[q], a[q + 1]);
    __syncthreads();
    float2 c[2][16];
#pragma unroll
    for (int u = 0; u < 16; ++u) ld_sh2(row + 2 * j + 32 * u, c[0][u], c[1][u]);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2* tw = tf + (2 * j + e) * 16;
#pragma unroll
      for (int u = 2; u < 16; u += 2) {
        float2 w0, w1;
        ld_sh2(tw + u, w0, w1);
        c[e][u] = cmul(c[e][u], w0);
        c[e][u + 1] = cmul(c[e][u + 1], w1);
      }
      c[e][1] = cmul(c[e][1], tw[1]);
      dft<16, false, CxPaired>(c[e]);
    }
    __syncthreads();   // every thread has read its row
    if (sig >= 8) {
#pragma unroll
      for (int q = 0; q < 16; ++q) st_sh2(row + (j * 16 + q) * 2, c[0][q], c[1][q]);
    }
    __syncthreads();
    if (sig < 8) {
      const float2* vrow = buf + (sig + 8) * kRowB;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        float2 v0, v1, s0, s1;
        ld_sh2(vrow + (j * 16 + q) * 2, v0, v1);
        ld_sh2(acc + 2 * q, s0, s1);
        st_sh2(acc + 2 * q, cadd(s0, cmulc(c[0][q], v0)), cadd(s1, cmulc(c[1][q], v1)));
      }
    }
  }
  __syncthreads();
  // Sum of the 8 partial spectra, two bins a thread, into Y[m][q] (row
  // stride 17): bin k1 = m + 32q, m = 2j + e, sits at 32j + 2q + e in the
  // sums' rows.
  float2* ybuf = buf + 8 * kRowB;      // Y: 32 x 17
  float2* zbuf = buf + 10 * kRowB;     // Z: 16 x 33
  {
    const int t = threadIdx.x;
    float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      float2 v0, v1;
      ld_sh2(accs + g * kRowB + 2 * t, v0, v1);
      s0 = cadd(s0, v0);
      s1 = cadd(s1, v1);
    }
    const int m = 2 * (t >> 4), q = t & 15;
    ybuf[m * 17 + q] = s0;
    ybuf[(m + 1) * 17 + q] = s1;
  }
  __syncthreads();
  if (warp != 0) return;
  // The inverse 512-point DFT (pass B's steps I1, I2 with the same
  // twiddles) on one warp.  I1: lane m, the 16-point inverse over q.
  {
    float2 c[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) c[q] = ybuf[lane * 17 + q];
    dft<16, true, CxPaired>(c);
#pragma unroll
    for (int r = 0; r < 16; ++r) zbuf[r * 33 + lane] = c[r];
  }
  __syncwarp();
  // I2: for each r the twiddle conj(w_512^{m r}), then the 32-point inverse
  // over m, split in two halves: lane r + 16h transforms the m = 2i + h
  // terms, h = 1 scales by w_32^{-n}, and the lane pair adds/subtracts
  // through one shuffle per component.
  // ti and the output twiddles tx are read from the global tables: a lane's
  // entries are 32 apart, one bank in shared memory.
  const int r = lane & 15, h = lane >> 4;
  const float2* ti = tabs + kTabB;
  float2 x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int m = 2 * i + h;
    x[i] = cmulc(zbuf[r * 33 + m], __ldg(ti + r * 32 + m));
  }
  dft<16, true, CxPaired>(x);
  if (h) {
#pragma unroll
    for (int n = 1; n < 16; ++n) x[n] = cmulc(x[n], tf[16 * 16 + n]);
  }
  const float2* tz = tabs + (size_t)(2 + k2) * kTabB + r * 32 + 16 * h;
  float2* out = y + ((size_t)bhl * N2 + k2) * kFastN1 + r + 256 * h;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    float2 o;
    o.x = __shfl_xor_sync(0xffffffffu, x[n].x, 16);
    o.y = __shfl_xor_sync(0xffffffffu, x[n].y, 16);
    const float2 v = h ? csub(o, x[n]) : cadd(x[n], o);
    out[16 * n] = cmulc(v, __ldg(tz + n));
  }
}


// Backward correlation, pass C for N2 = 32: one thread per (b, h, n1), the
// inverse DFT over k2 of y[bhl][k2][n1] in registers; dz*[n1 + 512·n2] =
// Re / N.  Consecutive threads take consecutive n1, so loads and stores are
// contiguous runs.
__global__ void __launch_bounds__(128)
fsf_corr_c32(const float2* __restrict__ y, float* __restrict__ dzs, int N, int bh0, int nb) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nb * kFastN1) return;
  const int bhl = i / kFastN1, n1 = i - bhl * kFastN1;
  const float2* src = y + (size_t)bhl * 32 * kFastN1 + n1;
  float2 a[32];
#pragma unroll
  for (int k2 = 0; k2 < 32; ++k2) a[k2] = src[(size_t)k2 * kFastN1];
  dft<32, true, CxPaired>(a);
  const float invN = 1.0f / (float)N;
  float* out = dzs + (size_t)(bh0 + bhl) * N + n1;
#pragma unroll
  for (int n2 = 0; n2 < 32; ++n2) out[(size_t)n2 * kFastN1] = a[n2].x * invN;
}

// Builds pass B's twiddle tables [tf | ti | tx for k2 = 0..N2-1] and, for
// N2 = 32, the spectrum kernel's t1, from the plan's table
// W[e] = exp(-2πi e/N).
__global__ void fsf_build_tables(float2* __restrict__ tabs, const float2* __restrict__ W, int N,
                                 int N2) {
  const int wstep = N / kFastN1;
  const int total = 2 * kTabB + N2 * kTabB + (N2 == 32 ? 32 * kFastN1 : 0);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    float2 v;
    if (i < kTabB) {                       // tf[k][u]
      const int k = i / 16, u = i % 16;
      v = W[(size_t)(u * k) * wstep];
    } else if (i < 2 * kTabB) {            // ti[j][u]
      const int r = i - kTabB, jj = r / 32, u = r % 32;
      v = W[(size_t)(u * jj) * wstep];
    } else if (i < (2 + N2) * kTabB) {     // tx[k2][j][q]
      const int r = i - 2 * kTabB, kk = r / kTabB, r2 = r % kTabB;
      const int jj = r2 / 32, q = r2 % 32;
      v = W[(size_t)(jj + 16 * q) * kk];
    } else {                               // t1[k2][n1] (N2 = 32)
      const int r = i - (2 + N2) * kTabB, kk = r / kFastN1, n1 = r % kFastN1;
      v = W[(size_t)n1 * kk];
    }
    tabs[i] = v;
  }
}

// ---------------------------------------------------------------------------
// Spectrum of z* in pass B's order for N2 > 32 (rows longer than one CTA
// holds), with the same register transforms.
// zspec_a (per n1, over n2): applies the softmax itself — z* = exp(z - m)/S
// from the double-float scores and the row's chunk partials — then the DFT;
// lanes are consecutive n1 of one (b, h) row, so the strided reads are
// coalesced; z* enters as a complex signal with zero imaginary part.
// Result times w_N^{n1 k2} into zscr[row][k2][n1].
// zspec_b (per k2, over n1): 8 consecutive k2 per CTA laid out like pass B's
// signals (lane: signal l & 7, j = 4·warp + (l >> 3)); result /N stored
// where pass B's thread j reads it.
// ---------------------------------------------------------------------------
template <int N2>
__global__ void __launch_bounds__(256)
fsf_zspec_a(const float2* __restrict__ z2, const float2* __restrict__ part, int P,
            float2* __restrict__ zscr, const float2* __restrict__ W, int N,
            const float2* __restrict__ tf) {
  // tf[k][u] = w_512^{u·k} (k < 32, u < 16), the plan's first table: the
  // step-2 twiddle w_N2^{u·k} is tf[k][(16 / R2)·u], a 4 KB table that stays
  // in L1 (the full table W is N entries).
  __shared__ float stats[2];
  static_assert(N2 > 32, "N2 = 32 rows take fsf_zspec_row");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    constexpr int TS = N2 / 32;
    constexpr int R2 = N2 / 32;
    constexpr int PER = 32 / TS;
    constexpr int RS = N2 + 2;
    extern __shared__ float4 smem4[];
    float2* buf = reinterpret_cast<float2*>(smem4);
    const int j = warp;
    const int row = blockIdx.x / (kFastN1 / 32);
    const int n1 = (blockIdx.x % (kFastN1 / 32)) * 32 + lane;
    const float2* src = z2 + (size_t)row * N + n1;
    float2 zv[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) zv[u] = __ldg(src + (size_t)kFastN1 * (j + TS * u));
    row_softmax_stats(part + (size_t)row * P, P, stats);
    const float m = stats[0], inv = stats[1];
    float2 a[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) a[u] = make_float2(exp_shifted(zv[u], m) * inv, 0.f);
    dft<32, false>(a);
    float2* rb = buf + lane * RS;
#pragma unroll
    for (int s = 0; s < 32; s += 2) st_sh2(rb + 32 * j + s, a[s], a[s + 1]);
    __syncthreads();
    float2 c[PER][R2];
#pragma unroll
    for (int u = 0; u < R2; ++u)
#pragma unroll
      for (int e = 0; e < PER; e += 2) ld_sh2(rb + PER * j + e + 32 * u, c[e][u], c[e + 1][u]);
    float2* dst = zscr + (size_t)row * N + n1;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int k = PER * j + e;
#pragma unroll
      for (int u = 1; u < R2; ++u) c[e][u] = cmul(c[e][u], __ldg(&tf[k * 16 + (16 / R2) * u]));
      dft<R2, false>(c[e]);
#pragma unroll
      for (int s = 0; s < R2; ++s) {
        const int k2 = k + 32 * s;
        dst[(size_t)k2 * kFastN1] = cmul(c[e][s], __ldg(&W[(size_t)n1 * k2]));
      }
    }
  }
}

__global__ void __launch_bounds__(128)
fsf_zspec_b(const float2* __restrict__ zscr, float2* __restrict__ zft, const float2* __restrict__ tf,
            int N, int N2) {
  // tf[k][u] = w_512^{u·k}: the step-F2 twiddles, 16 a bin pair.
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pl = lane & 7;
  const int j = 4 * warp + (lane >> 3);
  const int per_row = N2 / 8;
  const int row = blockIdx.x / per_row;
  const int k2 = (blockIdx.x % per_row) * 8 + pl;
  float2* rb = buf + pl * kRowB;
  const float2* src = zscr + (size_t)row * N + (size_t)k2 * kFastN1;
  float2 a[32];
#pragma unroll
  for (int u = 0; u < 32; ++u) a[u] = src[j + 16 * u];
  dft<32, false>(a);
#pragma unroll
  for (int s = 0; s < 32; s += 2) st_sh2(rb + 32 * j + s, a[s], a[s + 1]);
  __syncthreads();
  float2 c[2][16];
#pragma unroll
  for (int u = 0; u < 16; ++u) ld_sh2(rb + 2 * j + 32 * u, c[0][u], c[1][u]);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float4* tw = reinterpret_cast<const float4*>(tf + (2 * j + e) * 16);
#pragma unroll
    for (int u = 0; u < 16; u += 2) {
      const float4 w = __ldg(tw + u / 2);
      if (u > 0) c[e][u] = cmul(c[e][u], make_float2(w.x, w.y));
      c[e][u + 1] = cmul(c[e][u + 1], make_float2(w.z, w.w));
    }
    dft<16, false>(c[e]);
  }
  const float invN = 1.0f / (float)N;
  float4* out = reinterpret_cast<float4*>(zft) + (((size_t)row * N2 + k2) * 16 + j) * 16;
#pragma unroll
  for (int s = 0; s < 16; ++s)
    out[s] = make_float4(c[0][s].x * invN, c[0][s].y * invN, c[1][s].x * invN, c[1][s].y * invN);
}

// ---------------------------------------------------------------------------
// Spectrum of z* for N = 16384 (N2 = 32) in one CTA per (b, h) row: the
// softmax and both DFT passes of the row without leaving the SM.  Thread t
// (of 512) loads the scores z[t + 512·u], u < 32 — the length-32 signal of
// n1 = t over n2 = u — so the row maximum and the sum of exp(z - m) are
// block reductions over registers, and the first pass (DFT over n2, times
// w_N^{n1 k2}) needs no exchange.  Its results go to shared memory as
// [k2][n1]; the second pass (DFT over n1 per k2, 16 threads per k2 exactly
// as pass B's forward steps) stores FFT(z*)/N in pass B's order.
// ---------------------------------------------------------------------------
constexpr int kZRowThreads = 512;
constexpr int kZRowStride = kRowB;        // shared row of one k2 signal (float2)
constexpr size_t kZRowBuf = (size_t)32 * kZRowStride * sizeof(float2);
constexpr size_t kSmemZRow = kZRowBuf + kTabB * sizeof(float2) + 16;

__global__ void __launch_bounds__(kZRowThreads, 1)
fsf_zspec_row(const float2* z2, float2* __restrict__ zft, const float2* __restrict__ tabs, int N,
              unsigned int* status, float* __restrict__ zs) {
  extern __shared__ float4 smem4[];
  float2* buf = reinterpret_cast<float2*>(smem4);
  float2* tfs = buf + 32 * kZRowStride;                        // tf[k][u] = w_512^{u·k}
  uint64_t* bar = reinterpret_cast<uint64_t*>(tfs + kTabB);
  __shared__ float red[32];
  const int t = threadIdx.x;
  const int row = blockIdx.x;
  // The first-pass twiddles t1[k2][n1] land in the row buffer itself, each
  // where the thread that multiplies by it will store its product; tf goes
  // after it.  Bulk copies, in flight while the scores load.
  if (t == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
    const float2* t1 = tabs + (size_t)(2 + 32) * kTabB;
    mbar_expect_tx(bar, (32 * kFastN1 + kTabB) * (uint32_t)sizeof(float2));
    for (int k2 = 0; k2 < 32; ++k2)
      bulk_g2s(buf + k2 * kZRowStride, t1 + k2 * kFastN1, kFastN1 * sizeof(float2), bar);
    bulk_g2s(tfs, tabs, kTabB * sizeof(float2), bar);
  }
  const float2* src = z2 + (size_t)row * N;
  float2 a[32];
  // Launched as the dependent of the score: the table copies above are in
  // flight while it finishes; the scores are read after the wait.
  pdl_wait();
#pragma unroll
  for (int u = 0; u < 32; ++u) a[u] = ld_dep(src + t + kFastN1 * u);
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < 32; ++u) m = fmaxf(m, a[u].x);
  m = block_reduce<true>(m, red);     // (its barriers also publish the mbarrier init)
  float S = 0.f;
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    const float e = exp_shifted(a[u], m);
    a[u] = make_float2(e, 0.f);
    S += e;
  }
  S = block_reduce<false>(S, red);
  const float inv = 1.0f / S;
#pragma unroll
  for (int u = 0; u < 32; ++u) a[u].x *= inv;
  if (zs) {   // z* itself (the backward's softmax backward reads it)
    float* zr = zs + (size_t)row * N + t;
#pragma unroll
    for (int u = 0; u < 32; ++u) zr[kFastN1 * u] = a[u].x;
  }
  dft<32, false, CxPaired>(a);
  const bool ok = __syncthreads_and(mbar_wait(bar, 0, status, 0x503));
  // Twiddle w_N^{n1·k2} (n1 = t) and store [k2][n1].
  if (ok) {
#pragma unroll
    for (int k2 = 0; k2 < 32; ++k2) {
      float2* e = buf + k2 * kZRowStride + t;
      *e = cmul(a[k2], *e);
    }
  }
  __syncthreads();
  if (!ok) return;

  // Second pass, lanes laid out as in pass B: signal k2 = (lane mod 16) +
  // 16·(warp mod 2), thread j = 2·(warp / 2) + lane / 16 of it.
  const int lane = t & 31, warp = t >> 5;
  const int k2 = (lane & 15) + 16 * (warp & 1), j = 2 * (warp >> 1) + (lane >> 4);
  float2* rb = buf + k2 * kZRowStride;
#pragma unroll
  for (int u = 0; u < 32; ++u) a[u] = rb[j + 16 * u];
  __syncthreads();
  dft<32, false, CxPaired>(a);
#pragma unroll
  for (int q = 0; q < 32; q += 2) st_sh2(rb + 32 * j + q, a[q], a[q + 1]);
  __syncthreads();
  float2 c[2][16];
#pragma unroll
  for (int u = 0; u < 16; ++u) ld_sh2(rb + 2 * j + 32 * u, c[0][u], c[1][u]);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float2* tw = tfs + (2 * j + e) * 16;
#pragma unroll
    for (int u = 2; u < 16; u += 2) {
      float2 w0, w1;
      ld_sh2(tw + u, w0, w1);
      c[e][u] = cmul(c[e][u], w0);
      c[e][u + 1] = cmul(c[e][u + 1], w1);
    }
    c[e][1] = cmul(c[e][1], tw[1]);
    dft<16, false, CxPaired>(c[e]);
  }
  const float invN = 1.0f / (float)N;
  float4* out = reinterpret_cast<float4*>(zft) + (((size_t)row * 32 + k2) * 16 + j) * 16;
#pragma unroll
  for (int q = 0; q < 16; ++q)
    out[q] = make_float4(c[0][q].x * invN, c[0][q].y * invN, c[1][q].x * invN, c[1][q].y * invN);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
size_t fast_smem_a(int N2) { return N2 == 32 ? 0 : (size_t)kFastPairs * (N2 + 2) * sizeof(float2); }
size_t fast_smem_b() { return (size_t)16 * kRowB * sizeof(float2); }   // zspec_b

template <typename T>
static cudaError_t setup_t(int N2) {
  cudaError_t e = cudaSuccess;
  switch (N2) {
    case 32: break;   // the pipelined passes and the row spectrum kernel, set below
#define CAT_N2(n)                                                   \
  case n:                                                           \
    e = allow_max_smem(fsf_pass_a<T, n>);                           \
    if (e == cudaSuccess) e = allow_max_smem(fsf_pass_a_tma<T, n>); \
    if (e == cudaSuccess) e = allow_max_smem(fsf_pass_c<T, n>);     \
    if (e == cudaSuccess) e = allow_max_smem(fsf_zspec_a<n>);       \
    break;
    CAT_N2(64) CAT_N2(128) CAT_N2(256)
#undef CAT_N2
    default: return cudaErrorInvalidValue;
  }
  if (e == cudaSuccess) e = allow_max_smem(fsf_pass_b);
  if (e == cudaSuccess) e = allow_max_smem(fsf_pass_a32<T>);
  if (e == cudaSuccess) e = allow_max_smem(fsf_pass_c32<T>);
  if (e == cudaSuccess) e = allow_max_smem(fsf_zspec_b);
  if (e == cudaSuccess) e = allow_max_smem(fsf_zspec_row);
  if (e == cudaSuccess) e = allow_max_smem(fsf_corr_b);
  return e;
}

// [tf | ti | tx for k2 < N2], then for N2 = 32 the spectrum kernel's
// first-pass twiddles t1[k2][n1] = w_N^{n1·k2}.
size_t fast_tables_bytes(int N2) {
  return ((size_t)(2 + N2) * kTabB + (N2 == 32 ? (size_t)32 * kFastN1 : 0)) * sizeof(float2);
}

// Resident CTAs per SM of the tensor-copy pass A at N2 (0 if it cannot run).
template <typename T>
static int pass_a_tma_per_sm(int N2) {
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (N2) {
    case 64:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fsf_pass_a_tma<T, 64>, 64,
                                                        PipeAT<T, 64>::kSmem);
      break;
    case 128:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fsf_pass_a_tma<T, 128>, 128,
                                                        PipeAT<T, 128>::kSmem);
      break;
    case 256:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fsf_pass_a_tma<T, 256>, 256,
                                                        PipeAT<T, 256>::kSmem);
      break;
    default: break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t setup_fast_kernels(cat_plan_s* p) {
  cudaError_t e = p->dtype == 1 ? setup_t<__nv_bfloat16>(p->fs.N2) : setup_t<float>(p->fs.N2);
  if (e != cudaSuccess) return e;
  // The tensor-copy pass A for N2 >= 128 (at N2 = 64 the plain one was
  // faster); CAT_PASS_A_TMA=0 / 1 forces the plain / tensor-copy one.
  p->fs.a_tma_per_sm = 0;
  const char* ea = std::getenv("CAT_PASS_A_TMA");
  const bool use_tma = ea ? ea[0] != '0' : p->fs.N2 >= 128;
  if (p->fs.N2 > 32 && use_tma)
    p->fs.a_tma_per_sm = p->dtype == 1 ? pass_a_tma_per_sm<__nv_bfloat16>(p->fs.N2)
                                       : pass_a_tma_per_sm<float>(p->fs.N2);
  fsf_build_tables<<<64, 256, 0, p->stream>>>(p->tabs, p->tw, p->N, p->fs.N2);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
  if (e != cudaSuccess) return e;
  // Each scratch slot viewed as fp32 [chunk_bh][N2 (k2)][512 (n1)][64 (32 pairs)].
  const unsigned long long row = (unsigned long long)kFastPairs * sizeof(float2);
  const unsigned long long dims[4] = {2ull * kFastPairs, (unsigned long long)kFastN1,
                                      (unsigned long long)p->fs.N2,
                                      (unsigned long long)p->fs.chunk_bh};
  const unsigned long long strides[3] = {row, row * kFastN1, row * kFastN1 * p->fs.N2};
  const unsigned int box_c[4] = {64, 1, 32, 1};      // 32 rows k2 of all pairs
  for (int slot = 0; slot < 2; ++slot) {
    const float2* base = p->scratch + (size_t)slot * (p->scratch_bytes / 2 / sizeof(float2));
    if (p->fs.N2 == 32 &&
        !encode_map_4d(&p->tm_c[slot], base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dims, strides, box_c))
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// Generic passes A and C (N2 > 32): a CTA of N2 threads per (b, h, n1).
// An ordinary launch, or (dep) one as the programmatic dependent of the
// kernel ahead on the stream.
template <typename... KArgs, typename... Args>
static cudaError_t fast_launch(bool dep, void (*kernel)(KArgs...), int grid, int block,
                               size_t smem, cudaStream_t st, Args... args) {
  if (dep) return launch_dependent(kernel, dim3(grid), dim3(block), smem, st, args...);
  kernel<<<grid, block, smem, st>>>(args...);
  return cudaGetLastError();
}

// V viewed as [B][N2 (n2)][512 (n1)][D]: the box is one head's 64 columns of
// the N2 rows n1 + 512·n2.
template <typename T>
static bool encode_v_map(const cat_plan_s* p, const T* V, CUtensorMap* tmV) {
  const unsigned long long es = sizeof(T);
  const unsigned long long dims[4] = {(unsigned long long)p->D, (unsigned long long)kFastN1,
                                      (unsigned long long)p->fs.N2, (unsigned long long)p->B};
  const unsigned long long strides[3] = {p->D * es, (unsigned long long)kFastN1 * p->D * es,
                                         (unsigned long long)p->N * p->D * es};
  const unsigned int box[4] = {64, 1, (unsigned int)p->fs.N2, 1};
  return encode_map_4d(tmV, V, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       dims, strides, box);
}

// Grid of the tensor-copy pass A over `items` items: every CTA takes the
// same number of items (the last ones possibly one fewer), at most the
// resident CTAs of all SMs.
static int pass_a_tma_grid(const cat_plan_s* p, int items) {
  const int slots = p->fs.a_tma_per_sm * p->sms;
  const int per_cta = (items + slots - 1) / slots;
  return (items + per_cta - 1) / per_cta;
}

template <typename T, int N2>
static cudaError_t launch_ac(const cat_plan_s* p, const T* V, T* O, float2* scr, int bh0,
                             int nb, bool pass_a, cudaStream_t st, bool dep) {
  static_assert(N2 > 32, "N2 = 32 takes the pipelined passes");
  const int grid = nb * kFastN1;
  const int threads = N2;
  const size_t smem = fast_smem_a(N2);
  const int early = p->fast_pdl == 2;
  CUtensorMap tm;
  if (pass_a && p->fs.a_tma_per_sm > 0 && encode_v_map(p, V, &tm)) {
    const int g = pass_a_tma_grid(p, grid);
    return fast_launch(dep, fsf_pass_a_tma<T, N2>, g, N2, PipeAT<T, N2>::kSmem, st, tm, scr,
                       (const float2*)p->tw, p->N, p->D, p->H, bh0, nb, p->status, tm, scr, 1,
                       early);
  }
  if (pass_a)
    return fast_launch(dep, fsf_pass_a<T, N2>, grid, threads, smem, st, V, scr, (const float2*)p->tw,
                       (const float2*)p->tabs, p->N, p->D, p->H, bh0, nb, (const T*)nullptr,
                       (float2*)nullptr, early);
  return fast_launch(dep, fsf_pass_c<T, N2>, grid, threads, smem, st, (const float2*)scr, O,
                     (const float2*)p->tabs, p->N, p->D, p->H, bh0, nb, early);
}

cudaError_t launch_fast_zspec(const cat_plan_s* p, int row0, int nrows, cudaStream_t st,
                              bool dependent, float* zs) {
  const int N2 = p->fs.N2;
  if (nrows <= 0) return cudaSuccess;
  if (N2 == 32)
    return fast_launch(dependent && p->fast_pdl != 0, fsf_zspec_row, nrows, kZRowThreads,
                       kSmemZRow, st, (const float2*)(p->z2 + (size_t)row0 * p->N),
                       p->zf + (size_t)row0 * p->N, (const float2*)p->tabs, p->N, p->status,
                       zs ? zs + (size_t)row0 * p->N : nullptr);
  if (zs) return cudaErrorInvalidValue;
  // Longer rows: the multi-CTA softmax's chunk partials, then the two passes
  // (as programmatic dependents their early CTAs held SMs the kernel ahead
  // still needed: long128k 541 against 552 us).
  Span sp;
  sp.b0 = row0 / p->H;
  sp.nbat = nrows / p->H;
  sp.st = st;
  sp.own = true;
  cudaError_t e0 = launch_softmax(p, sp, false);
  if (e0 != cudaSuccess) return e0;
  const int P = softmax_parts(p->N);
  const float2* z2 = p->z2 + (size_t)row0 * p->N;
  const float2* part = p->part + (size_t)row0 * P;
  float2* zscr = p->zscr + (size_t)row0 * p->N;
  float2* zf = p->zf + (size_t)row0 * p->N;
  switch (N2) {
#define CAT_ZA(n)                                                                      \
  case n:                                                                              \
    fsf_zspec_a<n><<<nrows * (kFastN1 / 32), n, fast_smem_a(n), st>>>(z2, part, P, zscr, \
                                                                      p->tw, p->N, p->tabs); \
    break;
    CAT_ZA(64) CAT_ZA(128) CAT_ZA(256)
#undef CAT_ZA
    default: return cudaErrorInvalidValue;
  }
  fsf_zspec_b<<<nrows * (N2 / 8), 128, fast_smem_b() / 2, st>>>(zscr, zf, p->tabs, p->N, N2);
  return cudaGetLastError();
}

// A chunk's passes on stream st.  With p->fast_pdl set, each pass whose
// stream predecessor is the pass before it (pass A after the previous
// chunk's pass C when dep_a, pass B after pass A unless an event wait sits
// between them, pass C after pass B) launches as that kernel's programmatic
// dependent: its launch and the work before its wait overlap the end of the
// pass ahead.  Stage timing (after != nullptr) keeps ordinary launches.
template <typename T>
static cudaError_t chunk_t(const cat_plan_s* p, const T* V, T* O, int bh0, int nb, int slot,
                           cudaStream_t st, const CUtensorMap* tmV, cudaEvent_t before_b,
                           cudaEvent_t* after, bool dep_a) {
  const int N2 = p->fs.N2;
  float2* scr = p->scratch + (size_t)slot * (p->scratch_bytes / 2 / sizeof(float2));
  const bool pdl = p->fast_pdl != 0 && after == nullptr;
  const int early = p->fast_pdl == 2;
  auto ac = [&](bool pass_a, bool dep) -> cudaError_t {
    switch (N2) {
      case 32: {
        const int items = nb * kFastN1;
        if (pass_a) {
          // Resident CTAs per SM: two when two tiles' stages fit.
          const int per_sm = PipeA<T>::kSmem <= (113u << 10) ? 2 : 1;
          int grid = (items + kPipeWarps - 1) / kPipeWarps;
          if (grid > per_sm * p->sms) grid = per_sm * p->sms;
          return fast_launch(dep, fsf_pass_a32<T>, grid, kPipeWarps * 32, PipeA<T>::kSmem, st,
                             *tmV, scr, (const float2*)p->tw, p->N, p->D, p->H, bh0, nb,
                             p->status, *tmV, scr, 1, early);
        }
        int grid = (items + PipeC::kWarps - 1) / PipeC::kWarps;
        if (grid > 2 * p->sms) grid = 2 * p->sms;
        return fast_launch(dep, fsf_pass_c32<T>, grid, PipeC::kWarps * 32, PipeC::kSmem, st,
                           p->tm_c[slot], (const float2*)scr, O, p->N, p->D, p->H, bh0, nb,
                           p->status, early, 0);
      }
      case 64: return launch_ac<T, 64>(p, V, O, scr, bh0, nb, pass_a, st, dep);
      case 128: return launch_ac<T, 128>(p, V, O, scr, bh0, nb, pass_a, st, dep);
      default: return launch_ac<T, 256>(p, V, O, scr, bh0, nb, pass_a, st, dep);
    }
  };
  cudaError_t e = ac(true, pdl && dep_a);
  if (e != cudaSuccess) return e;
  if (after) cudaEventRecord(after[0], st);
  if (before_b) {
    e = cudaStreamWaitEvent(st, before_b, 0);
    if (e != cudaSuccess) return e;
  }
  e = fast_launch(pdl && !before_b, fsf_pass_b, nb * N2 * (kFastPairs / kBPairs), kBPairs * 16,
                  kSmemB, st, scr, (const float2*)p->zf, (const float2*)p->tabs, N2, bh0, early,
                  0);
  if (e != cudaSuccess) return e;
  if (after) cudaEventRecord(after[1], st);
  e = ac(false, pdl);
  if (e != cudaSuccess) return e;
  if (after) cudaEventRecord(after[2], st);
  return cudaGetLastError();
}

cudaError_t launch_fast_chunk(const cat_plan_s* p, const void* V, void* O, int bh0, int nb,
                              int slot, cudaStream_t st, cudaEvent_t before_b,
                              cudaEvent_t* after, bool dep_a) {
  CUtensorMap tmV;
  if (p->dtype == 1) {
    if (p->fs.N2 == 32 && !encode_v_map(p, (const __nv_bfloat16*)V, &tmV))
      return cudaErrorInvalidValue;
    return chunk_t(p, (const __nv_bfloat16*)V, (__nv_bfloat16*)O, bh0, nb, slot, st, &tmV,
                   before_b, after, dep_a);
  }
  if (p->fs.N2 == 32 && !encode_v_map(p, (const float*)V, &tmV)) return cudaErrorInvalidValue;
  return chunk_t(p, (const float*)V, (float*)O, bh0, nb, slot, st, &tmV, before_b, after, dep_a);
}

// Passes B and C (N2 = 32) of the backward's dV = circ(z*)^T dO on rows
// [bh0, bh0 + nb) whose pass-A output is already at scr: rows row_off ..
// row_off + nb - 1 of scratch slot 0 (the correlation leaves dO's transform
// there).  circ(z*)^T = circ(r) with r[n] = z*[(-n) mod N], whose spectrum
// is conj(FFT(z*)) (z* is real): pass B multiplies by the spectrum in p->zf
// conjugated; pass C writes O.
template <typename T>
static cudaError_t bc32_t(const cat_plan_s* p, float2* scr, T* O, int bh0, int nb, int row_off,
                          cudaStream_t st) {
  const int early = p->fast_pdl == 2;
  fsf_pass_b<<<nb * 32 * (kFastPairs / kBPairs), kBPairs * 16, kSmemB, st>>>(
      scr, p->zf, p->tabs, 32, bh0, early, 1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int grid = (nb * kFastN1 + PipeC::kWarps - 1) / PipeC::kWarps;
  if (grid > 2 * p->sms) grid = 2 * p->sms;
  return fast_launch(p->fast_pdl != 0, fsf_pass_c32<T>, grid, PipeC::kWarps * 32, PipeC::kSmem,
                     st, p->tm_c[0], (const float2*)scr, O, p->N, p->D, p->H, bh0, nb, p->status,
                     early, row_off);
}

cudaError_t launch_fast_bc32(const cat_plan_s* p, float2* scr, void* O, int bh0, int nb,
                             int row_off, cudaStream_t st) {
  if (p->fs.N2 != 32 || row_off + nb > p->fs.chunk_bh) return cudaErrorInvalidValue;
  return p->dtype == 1 ? bc32_t(p, scr, (__nv_bfloat16*)O, bh0, nb, row_off, st)
                       : bc32_t(p, scr, (float*)O, bh0, nb, row_off, st);
}

int fast_chunks(const cat_plan_s* p) {
  const int rows = p->B * p->H;
  return (rows + p->fs.chunk_bh - 1) / p->fs.chunk_bh;
}

// Serialised fast path on the plan's stream (used when stage timing is on;
// the spectrum of z* is already in place): every chunk in turn on scratch
// slot 0.
cudaError_t launch_fast_conv(const cat_plan_s* p, const void* V, void* O, cudaEvent_t* ev) {
  const int rows = p->B * p->H;
  for (int bh0 = 0, c = 0; bh0 < rows; bh0 += p->fs.chunk_bh, ++c) {
    const int nb = rows - bh0 < p->fs.chunk_bh ? rows - bh0 : p->fs.chunk_bh;
    const cudaError_t e =
        launch_fast_chunk(p, V, O, bh0, nb, 0, p->stream, nullptr, ev ? ev + 3 * c : nullptr);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}


// Pass A alone (the backward correlation transforms dO and V with it): rows
// [bh0, bh0 + nb) of V into scratch slot `slot`, on stream st.
template <typename T>
static cudaError_t pass_a32_pair(const cat_plan_s* p, const T* A, const T* Bm, int bh0, int nb,
                                 float2* s0, float2* s1, cudaStream_t st) {
  CUtensorMap tmA, tmB;
  if (!encode_v_map(p, A, &tmA) || !encode_v_map(p, Bm, &tmB)) return cudaErrorInvalidValue;
  const int per_sm = PipeA<T>::kSmem <= (113u << 10) ? 2 : 1;
  int grid = (2 * nb * kFastN1 + kPipeWarps - 1) / kPipeWarps;
  if (grid > per_sm * p->sms) grid = per_sm * p->sms;
  fsf_pass_a32<T><<<grid, kPipeWarps * 32, PipeA<T>::kSmem, st>>>(
      tmA, s0, p->tw, p->N, p->D, p->H, bh0, nb, p->status, tmB, s1, 2, 0);
  return cudaGetLastError();
}

// The correlation's pass A for N2 > 32 on dO (into s0) and V (into s1) in
// one launch: the plain kernel on a doubled grid ...
template <typename T, int N2>
static cudaError_t corr_a_plain_t(const cat_plan_s* p, const T* g, const T* v, float2* s0,
                                  float2* s1, int bh0, int nb, cudaStream_t st) {
  fsf_pass_a<T, N2><<<2 * nb * kFastN1, N2, fast_smem_a(N2), st>>>(g, s0, p->tw, p->tabs, p->N, p->D,
                                                                   p->H, bh0, nb, v, s1);
  return cudaGetLastError();
}

// ... or the tensor-copy kernel over both tensors' items
// (cudaErrorNotSupported when it cannot run: off, or a map that does not
// encode).
template <typename T, int N2>
static cudaError_t corr_a_tma_t(const cat_plan_s* p, const T* g, const T* v, float2* s0,
                                float2* s1, int bh0, int nb, cudaStream_t st) {
  CUtensorMap tmA, tmB;
  if (p->fs.a_tma_per_sm <= 0 || !encode_v_map(p, g, &tmA) || !encode_v_map(p, v, &tmB))
    return cudaErrorNotSupported;
  const int grid = pass_a_tma_grid(p, 2 * nb * kFastN1);
  fsf_pass_a_tma<T, N2><<<grid, N2, PipeAT<T, N2>::kSmem, st>>>(
      tmA, s0, p->tw, p->N, p->D, p->H, bh0, nb, p->status, tmB, s1, 2, 0);
  return cudaGetLastError();
}

template <bool TMA, typename T>
static cudaError_t corr_a_t(const cat_plan_s* p, const T* g, const T* v, float2* s0, float2* s1,
                            int bh0, int nb, cudaStream_t st) {
  switch (p->fs.N2) {
#define CAT_CA(n)                                                              \
  case n:                                                                      \
    return TMA ? corr_a_tma_t<T, n>(p, g, v, s0, s1, bh0, nb, st)              \
               : corr_a_plain_t<T, n>(p, g, v, s0, s1, bh0, nb, st);
    CAT_CA(64) CAT_CA(128) CAT_CA(256)
#undef CAT_CA
    default: return cudaErrorInvalidValue;
  }
}

static cudaError_t corr_pass_a_tma(const cat_plan_s* p, const void* G, const void* V, float2* s0,
                                   float2* s1, int bh0, int nb, cudaStream_t st) {
  return p->dtype == 1 ? corr_a_t<true>(p, (const __nv_bfloat16*)G, (const __nv_bfloat16*)V, s0,
                                        s1, bh0, nb, st)
                       : corr_a_t<true>(p, (const float*)G, (const float*)V, s0, s1, bh0, nb, st);
}

static cudaError_t corr_pass_a_plain(const cat_plan_s* p, const void* G, const void* V,
                                     float2* s0, float2* s1, int bh0, int nb, cudaStream_t st) {
  return p->dtype == 1 ? corr_a_t<false>(p, (const __nv_bfloat16*)G, (const __nv_bfloat16*)V, s0,
                                         s1, bh0, nb, st)
                       : corr_a_t<false>(p, (const float*)G, (const float*)V, s0, s1, bh0, nb, st);
}

cudaError_t launch_fast_corr(const cat_plan_s* p, const void* G, const void* V, float2* y,
                             int bh0, int nb, cudaStream_t st, float2* s0, float2* s1) {
  if (!s0) s0 = p->scratch;
  if (!s1) s1 = p->scratch + p->scratch_bytes / 2 / sizeof(float2);
  if (p->fs.N2 != 32) {
    // dO into s0 and V into s1 as one launch (a doubled grid, or the
    // tensor-copy pass A over both tensors' items).
    cudaError_t e = corr_pass_a_tma(p, G, V, s0, s1, bh0, nb, st);
    if (e == cudaErrorNotSupported) e = corr_pass_a_plain(p, G, V, s0, s1, bh0, nb, st);
    if (e != cudaSuccess) return e;
    fsf_corr_b<<<nb * p->fs.N2, 256, kSmemCorrB, st>>>(s0, s1, y, p->tabs, p->fs.N2);
    return cudaGetLastError();
  }
  // N2 = 32: dO into s0 and V into s1 as one launch.
  cudaError_t e = p->dtype == 1
      ? pass_a32_pair(p, (const __nv_bfloat16*)G, (const __nv_bfloat16*)V, bh0, nb, s0, s1, st)
      : pass_a32_pair(p, (const float*)G, (const float*)V, bh0, nb, s0, s1, st);
  if (e != cudaSuccess) return e;
  fsf_corr_b<<<nb * p->fs.N2, 256, kSmemCorrB, st>>>(s0, s1, y, p->tabs, p->fs.N2);
  return cudaGetLastError();
}

cudaError_t launch_fast_corr_c32(const cat_plan_s* p, const float2* y, float* dzs, int bh0,
                                 int nb, cudaStream_t st) {
  const int items = nb * kFastN1;
  fsf_corr_c32<<<(items + 127) / 128, 128, 0, st>>>(y, dzs, p->N, bh0, nb);
  return cudaGetLastError();
}

}  // namespace cat
