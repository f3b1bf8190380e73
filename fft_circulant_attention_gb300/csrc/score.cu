// Score projection and softmax over tokens — the "circulant attention matrix
// construction" design of the notes page "CAT: Circular-Convolutional
// Attention for Sub-Quadratic Transformers" (section 关键设计):
//     z[b, h, n] = sum_d X[b, n, d] · W_A[d, h]
//     z*[b, h, :] = softmax over the N tokens of z[b, h, :]
// plus, for the shared-memory path, the spectrum of z* (the "FFT
// acceleration" design) fused into the softmax kernel.
#include <cuda_bf16.h>

#include <type_traits>

#include "bulk.cuh"
#include "cat_internal.h"
#include "elem.cuh"
#include "mma.cuh"

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

// The same for two accumulators at once with the paired fp32 instructions
// (each component rounds exactly as the scalar operation; x - y is formed as
// y·(-1) + x, exact in the product).
__device__ __forceinline__ float2 sub2(float2 x, float2 y) {
  return __ffma2_rn(y, make_float2(-1.f, -1.f), x);
}
__device__ __forceinline__ void two_sum_acc2(float2& hi, float2& lo, float2 p) {
  const float2 s = __fadd2_rn(hi, p);
  const float2 bp = sub2(s, hi);
  const float2 err = __fadd2_rn(sub2(hi, sub2(s, bp)), sub2(p, bp));
  hi = s;
  lo = __fadd2_rn(lo, err);
}

// W_A's columns [h0, h0 + HT) as fp32 [D][HP] in shared memory (columns HT
// to HP zero).  Eight loads per thread are in flight before any is stored,
// so the staging costs a few latencies rather than D·HP / blockDim of them.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Row d of the staged block starts at float d·HP, or with `pad` at
// d·HP + 4·(d / 4): one 16-byte slot after every fourth row, so that the
// split kernel's four lanes of a token, which read rows 4 (fp32) or 8
// (bf16) apart at the same time, fall in distinct bank groups.
__host__ __device__ inline int w_row(int d, int HP, bool pad) { return d * HP + (pad ? 4 * (d >> 2) : 0); }

template <typename T>
__device__ __forceinline__ void stage_w_f32(float* ws, const T* __restrict__ WA, int D, int H,
                                            int h0, int HT, int HP, bool wait = true,
                                            bool pad = false) {
  if constexpr (std::is_same<T, float>::value) {
    // fp32 W_A needs no conversion: every element goes by an asynchronous
    // copy (all of a thread's copies in flight at once, no registers held),
    // 16 bytes at a time when the staged block is W_A itself (all heads,
    // H a multiple of 4, 16-byte aligned), else 4; padding columns are zeroed.
    if (h0 == 0 && HT == H && HP == H && ((uintptr_t)WA % 16) == 0) {
      const int c4 = H / 4;   // 16-byte chunks a row
      for (int i = threadIdx.x; i < D * c4; i += blockDim.x) {
        const int d = i / c4, c = i - d * c4;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         smem_addr(ws + w_row(d, HP, pad) + 4 * c)),
                     "l"(__cvta_generic_to_global(WA + 4 * i))
                     : "memory");
      }
    } else {
      for (int i = threadIdx.x; i < D * HP; i += blockDim.x) {
        const int d = i / HP, h = i - d * HP;
        float* dst = ws + w_row(d, HP, pad) + h;
        if (h < HT)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)),
                       "l"(__cvta_generic_to_global(WA + (size_t)d * H + h0 + h))
                       : "memory");
        else
          *dst = 0.f;
      }
    }
    // Without `wait` the caller waits (cp_async_wait_all) before the
    // barrier that publishes the block.
    if (wait) cp_async_wait_all();
    return;
  }
  constexpr int kBatch = 8;
  const int total = D * HP;
  for (int i0 = threadIdx.x; i0 < total; i0 += kBatch * blockDim.x) {
    float v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * blockDim.x;
      const int d = i / HP, h = i - d * HP;
      v[j] = (i < total && h < HT) ? ld_elem(WA + (size_t)d * H + h0 + h) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * blockDim.x;
      const int d = i / HP, h = i - d * HP;
      if (i < total) ws[w_row(d, HP, pad) + h] = v[j];
    }
  }
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
             int N, int D, int H, int h0, int b0) {
  pdl_trigger();   // the softmax kernel behind may launch (it waits for the scores)
  constexpr int HP = (HT + 3) & ~3;
  constexpr int TP = kScoreTokPerThread;
  extern __shared__ float4 ws4[];
  float* ws = reinterpret_cast<float*>(ws4);
  const int b = b0 + blockIdx.y;
  stage_w_f32(ws, WA, D, H, h0, HT, HP);
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

// The same score with kSplit threads per token: thread q of a token takes
// the 16-byte vectors q, q + kSplit, q + 2·kSplit, … of the token's row, so
// a warp reads rows in contiguous kSplit·16-byte runs.  Each thread serves
// kSplitTok tokens (the W_A row it reads from shared memory feeds all of
// them) and loads a run's vectors for all of them before the first FMA.
// Each run of kChunk products per head is summed in a fresh fp32 register
// and added into the thread's double-float (hi, lo) by TwoSum; the kSplit
// partial double-floats of a token are then combined by TwoSum across the
// lanes.  Requires 16-byte vectors and D a multiple of kSplit vectors.
constexpr int kSplitTok = 2;
// Tokens per CTA with KS threads per token.
template <int KS>
constexpr int split_tokens() { return kScoreThreads / KS * kSplitTok; }

template <typename T, int HT, int kSplit>
__global__ void __launch_bounds__(kScoreThreads)
score_split_kernel(const T* __restrict__ X, const T* __restrict__ WA, float2* __restrict__ z,
                   int N, int D, int H, int h0, int b0) {
  pdl_trigger();   // the softmax kernel behind may launch (it waits for the scores)
  constexpr int HP = (HT + 3) & ~3;
  constexpr int V = Vec16<T>::n;
  constexpr int RUN = kChunk / V;   // vectors per fresh run
  constexpr int TT = kSplitTok;
  constexpr int kScoreSplitTok = split_tokens<kSplit>();
  extern __shared__ float4 ws4[];
  float* ws = reinterpret_cast<float*>(ws4);
  const int b = b0 + blockIdx.y;
  // W_A's copies are issued first and waited for after the first X loads,
  // so the two latencies overlap.
  stage_w_f32(ws, WA, D, H, h0, HT, HP, false, true);
  const int q = threadIdx.x % kSplit;
  const int slot = threadIdx.x / kSplit;              // 0 .. kScoreThreads/kSplit - 1
  int n[TT];
  bool ok[TT];
  const T* xr[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    n[t] = blockIdx.x * kScoreSplitTok + slot + t * (kScoreThreads / kSplit);
    ok[t] = n[t] < N;
    xr[t] = X + ((size_t)b * N + (ok[t] ? n[t] : 0)) * D;
  }
  float hi[TT][HT], lo[TT][HT];
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int h = 0; h < HT; ++h) hi[t][h] = lo[t][h] = 0.f;
  const int nvec = D / V;   // vectors per row; a multiple of kSplit
  constexpr int kStep = kSplit * RUN;   // vectors a run advances
  // One run: RUN vectors of each token, loaded before any FMA (two buffers,
  // the next run's loads in flight while this one is summed).
  auto load_run = [&](float (&xv)[TT][RUN][V], int v0) {
#pragma unroll
    for (int r = 0; r < RUN; ++r) {
      const int v = min(v0 + r * kSplit, nvec - 1);   // loads stay in the row
#pragma unroll
      for (int t = 0; t < TT; ++t) Vec16<T>::load(xr[t] + v * V, xv[t][r]);
    }
  };
  auto sum_run = [&](const float (&xv)[TT][RUN][V], int v0) {
    float part[TT][HT];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int h = 0; h < HT; ++h) part[t][h] = 0.f;
#pragma unroll
    for (int r = 0; r < RUN; ++r) {
      const int v = v0 + r * kSplit;
      if (v < nvec) {
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const float4* wrow = ws4 + w_row(v * V + j, HP, true) / 4;
#pragma unroll
          for (int c = 0; c < HP / 4; ++c) {
            const float4 w = wrow[c];
            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (c * 4 + e < HT) {
#pragma unroll
                for (int t = 0; t < TT; ++t)
                  part[t][c * 4 + e] = fmaf(xv[t][r][j], wv[e], part[t][c * 4 + e]);
              }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int h = 0; h < HT; ++h) two_sum_acc(hi[t][h], lo[t][h], part[t][h]);
  };
  float xa[TT][RUN][V], xb[TT][RUN][V];
  load_run(xa, q);
  cp_async_wait_all();
  __syncthreads();
  for (int v0 = q; v0 < nvec; v0 += 2 * kStep) {
    if (v0 + kStep < nvec) load_run(xb, v0 + kStep);
    sum_run(xa, v0);
    if (v0 + kStep >= nvec) break;
    if (v0 + 2 * kStep < nvec) load_run(xa, v0 + 2 * kStep);
    sum_run(xb, v0 + kStep);
  }
  // Combine each token's kSplit lanes (adjacent lanes of one warp).
#pragma unroll
  for (int o = 1; o < kSplit; o <<= 1) {
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int h = 0; h < HT; ++h) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi[t][h], o);
        const float ol = __shfl_xor_sync(0xffffffffu, lo[t][h], o);
        two_sum_acc(hi[t][h], lo[t][h], oh);
        lo[t][h] += ol;
      }
  }
  if (q == 0) {
#pragma unroll
    for (int t = 0; t < TT; ++t)
      if (ok[t]) {
#pragma unroll
        for (int h = 0; h < HT; ++h)
          z[((size_t)b * H + h0 + h) * N + n[t]] = make_float2(hi[t][h], lo[t][h]);
      }
  }
}

// ---------------------------------------------------------------------------
// bf16 score on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 out).
// Products of two bf16 values are exact in fp32, so each MMA pair sums 32
// exact products of one 32-wide slice of d into a fresh fp32 accumulator;
// the slice sums are then added into a double-float (hi, lo) with TwoSum,
// exactly as the CUDA-core kernel does with its 16-wide runs.
//
// The slice order inside an MMA is free (a dot product), so each lane feeds
// the MMAs from one 16-byte load per token row: lane (r = lane/4, c = lane%4)
// loads X[row][d0 + 8c .. d0 + 8c + 8) for rows r and r + 8 of a 16-token
// tile; words 0-1 of that load feed MMA 1 and words 2-3 MMA 2, and W_A^T
// rows in shared memory are read with the same map.  A warp owns two tiles
// (32 tokens); heads go in n-tiles of 8 (NT = 1 or 2).
// ---------------------------------------------------------------------------
// W_A^T staging for the tensor-core kernels: wt[hh·ws + d] = W_A[d, h0 + hh]
// for hh < rows (0 beyond HT), by threads tid, tid + nthr, ...  When W_A's
// rows split into 16-byte vectors (H a multiple of 8, W_A 16-byte aligned)
// the threads read consecutive vectors of W_A — one coalesced stream — and
// scatter their 8 heads into the transposed layout; otherwise each thread
// copies whole rows element by element.
// PAIRED: within each 16 columns the order 0 1 8 9 2 3 10 11 ..., so that a
// lane's two B-fragment words of an m16n8k16 MMA (k0, k0 + 1 and k0 + 8,
// k0 + 9, k0 = 2c) are one 8-byte load.
__device__ __forceinline__ int wt_col(int d, bool paired) {
  if (!paired) return d;
  const int r = d & 15;
  return (d & ~15) + ((r & 7) >> 1) * 4 + (r >> 3) * 2 + (r & 1);
}
template <bool PAIRED = false>
__device__ __forceinline__ void stage_wt(unsigned short* wt, int ws, const unsigned short* wa,
                                         int D, int H, int h0, int HT, int rows, int tid,
                                         int nthr) {
  for (int hh = HT; hh < rows; ++hh)
    for (int d = tid; d < D; d += nthr) wt[hh * ws + d] = 0;
  if (H % 8 == 0 && ((uintptr_t)wa & 15) == 0) {
    // kBatch vectors per thread are loaded before any is stored, so their
    // latencies overlap instead of adding up.
    constexpr int kBatch = 8;
    const int vpr = H / 8;                        // 16-byte vectors per row of W_A
    const int total = D * vpr;
    const uint4* wv = reinterpret_cast<const uint4*>(wa);
    for (int i0 = tid; i0 < total; i0 += kBatch * nthr) {
      uint4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * nthr;
        const int d = i / vpr, hb = (i - d * vpr) * 8 - h0;   // head of the vector's element 0
        v[j] = (i < total && hb + 8 > 0 && hb < HT) ? __ldg(wv + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * nthr;
        const int d = i / vpr, hb = (i - d * vpr) * 8 - h0;
        if (i >= total || hb + 8 <= 0 || hb >= HT) continue;
        const unsigned w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int hh = hb + q;
          if (hh >= 0 && hh < HT && hh < rows)
            wt[hh * ws + wt_col(d, PAIRED)] =
                (unsigned short)((q & 1) ? (w[q >> 1] >> 16) : (w[q >> 1] & 0xffffu));
        }
      }
    }
  } else {
    for (int d = tid; d < D; d += nthr) {
      const unsigned short* src = wa + (size_t)d * H + h0;
      unsigned short v[16];
#pragma unroll
      for (int hh = 0; hh < 16; ++hh) v[hh] = hh < HT ? __ldg(src + hh) : (unsigned short)0;
#pragma unroll
      for (int hh = 0; hh < 16; ++hh)
        if (hh < rows && hh < HT) wt[hh * ws + wt_col(d, PAIRED)] = v[hh];
    }
  }
}

constexpr int kMmaWarps = 4;
constexpr int kMmaTilesPerWarp = 2;
constexpr int kMmaTokPerCta = kMmaWarps * kMmaTilesPerWarp * 16;

// Row stride (bf16) of W_A^T in shared memory: D padded so that the eight
// head rows a quarter-warp reads fall in distinct bank groups.
__host__ __device__ inline int mma_wt_stride(int D) { return D + ((32 - D % 64) + 64) % 64; }

template <int NT>
__global__ void __launch_bounds__(kMmaWarps * 32)
score_mma_kernel(const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ WA,
                 float2* __restrict__ z, int N, int D, int H, int h0, int HT, int b0) {
  pdl_trigger();   // the softmax kernel behind may launch (it waits for the scores)
  extern __shared__ uint4 wsh4[];
  unsigned short* wt = reinterpret_cast<unsigned short*>(wsh4);
  const int ws = mma_wt_stride(D);
  const int b = b0 + blockIdx.y;
  stage_wt(wt, ws, reinterpret_cast<const unsigned short*>(WA), D, H, h0, HT, NT * 8, threadIdx.x,
           blockDim.x);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, c = lane & 3;
  const int tok0 = blockIdx.x * kMmaTokPerCta + warp * kMmaTilesPerWarp * 16;
  const uint4* xr[kMmaTilesPerWarp][2];
#pragma unroll
  for (int t = 0; t < kMmaTilesPerWarp; ++t)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      int n = min(tok0 + t * 16 + r + 8 * q, N - 1);
      xr[t][q] = reinterpret_cast<const uint4*>(X + ((size_t)b * N + n) * D + 8 * c);
    }
  const uint4* wrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
    wrow[nt] = reinterpret_cast<const uint4*>(wt + (nt * 8 + r) * ws + 8 * c);

  float hi[kMmaTilesPerWarp][NT][4], lo[kMmaTilesPerWarp][NT][4];
#pragma unroll
  for (int t = 0; t < kMmaTilesPerWarp; ++t)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) hi[t][nt][i] = lo[t][nt][i] = 0.f;

#pragma unroll 2
  for (int d0 = 0; d0 < D; d0 += 32) {
    uint4 xa[kMmaTilesPerWarp][2];
#pragma unroll
    for (int t = 0; t < kMmaTilesPerWarp; ++t)
#pragma unroll
      for (int q = 0; q < 2; ++q) xa[t][q] = __ldg(xr[t][q] + d0 / 8);
    uint4 wb[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) wb[nt] = wrow[nt][d0 / 8];
#pragma unroll
    for (int t = 0; t < kMmaTilesPerWarp; ++t) {
      const unsigned a1[4] = {xa[t][0].x, xa[t][1].x, xa[t][0].y, xa[t][1].y};
      const unsigned a2[4] = {xa[t][0].z, xa[t][1].z, xa[t][0].w, xa[t][1].w};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16(acc, a1, wb[nt].x, wb[nt].y);
        mma_bf16(acc, a2, wb[nt].z, wb[nt].w);
#pragma unroll
        for (int i = 0; i < 4; ++i) two_sum_acc(hi[t][nt][i], lo[t][nt][i], acc[i]);
      }
    }
  }
  // Accumulator i of a tile: token r + 8·(i >> 1), head 2c + (i & 1).
#pragma unroll
  for (int t = 0; t < kMmaTilesPerWarp; ++t)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = tok0 + t * 16 + r + 8 * (i >> 1);
        const int hh = nt * 8 + 2 * c + (i & 1);
        if (n < N && hh < HT)
          z[((size_t)b * H + h0 + hh) * N + n] = make_float2(hi[t][nt][i], lo[t][nt][i]);
      }
}

// ---------------------------------------------------------------------------
// TMA-fed bf16 score (the long workloads).  A persistent CTA streams tiles of
// 64 tokens × 64 d of X through an 8-stage shared-memory ring: one producer
// warp issues a 2-D tensor copy (128-byte swizzle) per stage, and 4·NT
// consumer warps, one per 16 tokens and n-tile of 8 heads, read their A
// fragments with ldmatrix and run the same slice-wise MMA + TwoSum as
// score_mma_kernel.  Loads thus run up to eight stages ahead of the math,
// independent of the consumer registers; a warp per n-tile halves each
// warp's chain of MMAs and TwoSums at NT = 2.
// ---------------------------------------------------------------------------
constexpr int kTsRows = 64, kTsCols = 64, kTsStages = 8;
template <int NT>
constexpr int ts_consumers() { return 4 * NT; }
template <int NT>
constexpr int ts_threads() { return (ts_consumers<NT>() + 1) * 32; }
constexpr int kTsStageBytes = kTsRows * kTsCols * 2;

// D + 16: a row is 8 words past a multiple of 32, so the 8-byte B-fragment
// loads of a half warp (4 rows × 4 lanes) fall in distinct banks.
__host__ __device__ inline int ts_wt_stride(int D) { return D + 16; }
static size_t score_tma_smem(int D) {
  return (size_t)kTsStages * kTsStageBytes + (size_t)16 * ts_wt_stride(D) * 2 + 2 * kTsStages * 8 +
         1024;
}

template <int NT>
__global__ void __launch_bounds__(ts_threads<NT>())
score_tma_kernel(const __grid_constant__ CUtensorMap tmX, const __nv_bfloat16* __restrict__ WA,
                 float2* __restrict__ z, int N, int D, int H, int h0, int HT, int row0,
                 int rows_total, unsigned int* status) {
  constexpr int kTsConsumers = ts_consumers<NT>();
  pdl_trigger();   // the softmax kernel behind may launch (it waits for the scores)
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* stages = sm;
  const int ws = ts_wt_stride(D);
  unsigned short* wt = reinterpret_cast<unsigned short*>(sm + kTsStages * kTsStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(wt + 16 * ws);
  uint64_t* empty = full + kTsStages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTsStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kTsConsumers);
    }
  }
  mbar_fence_init();
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // The producer starts streaming X at once; the consumer warps stage W_A^T
  // meanwhile and sync among themselves (named barrier 1) before using it.
  if (warp < kTsConsumers) {
    stage_wt<true>(wt, ws, reinterpret_cast<const unsigned short*>(WA), D, H, h0, HT, 16,
                   threadIdx.x, kTsConsumers * 32);
    asm volatile("bar.sync 1, %0;" ::"n"(kTsConsumers * 32) : "memory");
  }
  const int nkb = D / kTsCols;
  const int ntiles = (rows_total - row0 + kTsRows - 1) / kTsRows;

  if (warp == kTsConsumers) {   // producer
    if (lane == 0) {
      const uint64_t stream = policy_evict_first();
      int it = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x)
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kTsStages, use = it / kTsStages;
          if (use > 0) {
            if (!mbar_wait(empty + s, (use - 1) & 1, status, 0x601)) return;
            fence_proxy_async_smem();   // the consumers' ldmatrix reads come first
          }
          mbar_expect_tx(full + s, kTsStageBytes);
          tma_load_2d_hint(stages + s * kTsStageBytes, &tmX, kb * kTsCols, row0 + tile * kTsRows,
                           full + s, stream);
        }
    }
    return;
  }

  // Consumer warp: tokens 16·tg .. of the tile, heads 8·nt .. (n-tile nt).
  const int tg = warp & 3, nt = warp >> 2;
  const int c = lane & 3, mrow = lane >> 2;
  const int lm = lane >> 3, li = lane & 7;
  const int arow = tg * 16 + (lm & 1) * 8 + li;   // ldmatrix row this lane addresses
  const unsigned short* wrow = wt + (nt * 8 + mrow) * ws + 4 * c;   // paired columns
  int it = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    // Accumulators in pairs: [r] holds fragment elements 2r, 2r + 1.
    float2 hi[2], lo[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) hi[r] = lo[r] = make_float2(0.f, 0.f);
    for (int kb = 0; kb < nkb; ++kb, ++it) {
      const int s = it % kTsStages;
      if (!mbar_wait(full + s, (it / kTsStages) & 1, status, 0x602)) return;
      const uint32_t base = smem_addr(stages + s * kTsStageBytes) + arow * 128;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int t = 2 * half + q;            // 16-wide k step within the 64
          const int chunk = 2 * t + (lm >> 1);
          unsigned a[4];
          ldmatrix_x4(a, base + ((chunk ^ (arow & 7)) << 4));
          const uint2 bw = *reinterpret_cast<const uint2*>(wrow + kb * kTsCols + 16 * t);
          mma_bf16(acc, a, bw.x, bw.y);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
          two_sum_acc2(hi[r], lo[r], make_float2(acc[2 * r], acc[2 * r + 1]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = row0 + tile * kTsRows + tg * 16 + mrow + 8 * (i >> 1);
      const int hh = nt * 8 + 2 * c + (i & 1);
      if (r < rows_total && hh < HT) {
        const int b = r / N, n = r - b * N;
        const float2 hv = hi[i >> 1], lv = lo[i >> 1];
        z[((size_t)b * H + h0 + hh) * N + n] =
            (i & 1) ? make_float2(hv.y, lv.y) : make_float2(hv.x, lv.x);
      }
    }
  }
}

static bool score_tma_ok(const cat_plan_s* p, const void* X) {
  return p->dtype == 1 && p->D % 64 == 0 && ((uintptr_t)X % 16) == 0 &&
         score_tma_smem(p->D) <= (226u << 10);
}

static cudaError_t score_tma(const cat_plan_s* p, const void* X, const void* WA, bool setup,
                             const Span& sp = Span{}) {
  if (setup) {
    cudaError_t e = allow_max_smem(score_tma_kernel<1>);
    return e == cudaSuccess ? allow_max_smem(score_tma_kernel<2>) : e;
  }
  CUtensorMap tm;
  const unsigned long long rows = (unsigned long long)p->B * p->N;
  if (!encode_map_2d_sw128(&tm, X, (unsigned long long)p->D, rows, (unsigned long long)p->D * 2,
                           kTsCols, kTsRows))
    return cudaErrorInvalidValue;
  const int row0 = sp.b0 * p->N;
  const int row_end = (sp.b0 + sp.nb(p)) * p->N;
  const int ntiles = (row_end - row0 + kTsRows - 1) / kTsRows;
  if (ntiles <= 0) return cudaSuccess;
  const size_t smem = score_tma_smem(p->D);
  const int per_sm = smem <= (113u << 10) ? 2 : 1;
  // Every CTA takes the same number of tiles (the last one possibly fewer),
  // so no CTA runs a lone extra tile at the end.
  const int max_grid = per_sm * p->sms;
  const int per_cta = (ntiles + max_grid - 1) / max_grid;
  const int grid = (ntiles + per_cta - 1) / per_cta;
  const cudaStream_t st = sp.stream(p);
  for (int h0 = 0; h0 < p->H; h0 += 16) {
    const int ht = p->H - h0 < 16 ? p->H - h0 : 16;
    if (ht > 8)
      score_tma_kernel<2><<<grid, ts_threads<2>(), smem, st>>>(
          tm, (const __nv_bfloat16*)WA, p->z2, p->N, p->D, p->H, h0, ht, row0, row_end, p->status);
    else
      score_tma_kernel<1><<<grid, ts_threads<1>(), smem, st>>>(
          tm, (const __nv_bfloat16*)WA, p->z2, p->N, p->D, p->H, h0, ht, row0, row_end, p->status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

static size_t score_mma_smem(int D) { return (size_t)16 * mma_wt_stride(D) * 2; }

static bool score_mma_ok(const cat_plan_s* p, const void* X) {
  return p->dtype == 1 && p->D % 32 == 0 && ((uintptr_t)X % 16) == 0 &&
         score_mma_smem(p->D) <= (200u << 10);
}

static cudaError_t score_mma(const cat_plan_s* p, const void* X, const void* WA, bool setup,
                             const Span& sp = Span{}) {
  if (setup) {
    cudaError_t e = allow_max_smem(score_mma_kernel<1>);
    return e == cudaSuccess ? allow_max_smem(score_mma_kernel<2>) : e;
  }
  dim3 grid((p->N + kMmaTokPerCta - 1) / kMmaTokPerCta, sp.nb(p));
  const cudaStream_t st = sp.stream(p);
  for (int h0 = 0; h0 < p->H; h0 += 16) {
    const int ht = p->H - h0 < 16 ? p->H - h0 : 16;
    const size_t smem = score_mma_smem(p->D);
    if (ht > 8)
      score_mma_kernel<2><<<grid, kMmaWarps * 32, smem, st>>>(
          (const __nv_bfloat16*)X, (const __nv_bfloat16*)WA, p->z2, p->N, p->D, p->H, h0, ht,
          sp.b0);
    else
      score_mma_kernel<1><<<grid, kMmaWarps * 32, smem, st>>>(
          (const __nv_bfloat16*)X, (const __nv_bfloat16*)WA, p->z2, p->N, p->D, p->H, h0, ht,
          sp.b0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T>
static bool score_vec_ok(const cat_plan_s* p, const void* X) {
  const int V = 16 / (int)sizeof(T);
  return (p->D % V) == 0 && ((uintptr_t)X % 16) == 0;
}

template <typename T, int HT, bool VEC>
static cudaError_t run_score(const cat_plan_s* p, const T* X, const T* WA, int h0, bool setup,
                            const Span& sp) {
  constexpr int HP = (HT + 3) & ~3;
  size_t smem = (size_t)HP * p->D * sizeof(float);
  auto k = score_kernel<T, HT, VEC>;
  auto ks4 = score_split_kernel<T, HT, 4>;
  if (setup) {
    cudaError_t e = allow_max_smem(k);
    return (e == cudaSuccess && VEC) ? allow_max_smem(ks4) : e;
  }
  // Rows of whole 4-thread vector groups take the split kernel.
  if (VEC && p->D % (4 * Vec16<T>::n) == 0) {
    constexpr int tok = split_tokens<4>();
    dim3 grid((p->N + tok - 1) / tok, sp.nb(p));
    const size_t smem_split = (size_t)w_row(p->D, HP, true) * sizeof(float);   // padded rows
    ks4<<<grid, kScoreThreads, smem_split, sp.stream(p)>>>(X, WA, p->z2, p->N, p->D, p->H, h0,
                                                            sp.b0);
    return cudaGetLastError();
  }
  dim3 grid((p->N + kScoreTokPerCta - 1) / kScoreTokPerCta, sp.nb(p));
  k<<<grid, kScoreThreads, smem, sp.stream(p)>>>(X, WA, p->z2, p->N, p->D, p->H, h0, sp.b0);
  return cudaGetLastError();
}

template <typename T, bool VEC>
static cudaError_t score_heads(const cat_plan_s* p, const T* X, const T* WA, bool setup,
                               const Span& sp = Span{}) {
  const int hpp = score_heads_per_pass(p->D);
  for (int h0 = 0; h0 < p->H; h0 += hpp) {
    int ht = p->H - h0 < hpp ? p->H - h0 : hpp;
    cudaError_t e;
    switch (ht) {
#define CAT_HT(n) case n: e = run_score<T, n, VEC>(p, X, WA, h0, setup, sp); break;
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
static cudaError_t score_dispatch(const cat_plan_s* p, const T* X, const T* WA, bool setup,
                                 const Span& sp = Span{}) {
  if (setup) {
    cudaError_t e = score_heads<T, true>(p, X, WA, true);
    if (e != cudaSuccess) return e;
    return score_heads<T, false>(p, X, WA, true);
  }
  if (score_vec_ok<T>(p, X)) return score_heads<T, true>(p, X, WA, false, sp);
  return score_heads<T, false>(p, X, WA, false, sp);
}

cudaError_t launch_score(const cat_plan_s* p, const void* X, const void* WA, const Span& sp) {
  if (sp.nb(p) == 0) return cudaSuccess;
  if (!p->score_cuda_cores && p->score_path != 1 && score_tma_ok(p, X))
    return score_tma(p, X, WA, false, sp);
  if (score_mma_ok(p, X) && !p->score_cuda_cores) return score_mma(p, X, WA, false, sp);
  if (p->dtype == 1)
    return score_dispatch(p, (const __nv_bfloat16*)X, (const __nv_bfloat16*)WA, false, sp);
  return score_dispatch(p, (const float*)X, (const float*)WA, false, sp);
}


// Softmax over the N tokens of each (b, h) row, split over P CTAs per row
// (about 2048 tokens each).  softmax_partial: per chunk c, m_c = max of the
// scores and s_c = sum of exp(z - m_c).  softmax_finish: every CTA combines
// its row's partials into m = max m_c and S = sum s_c·exp(m_c - m), then
// writes z* = exp(z - m) / S for its chunk.
constexpr int kSoftmaxThreads = 256;

__device__ __forceinline__ void chunk_range(int N, int P, int c, int& n0, int& n1) {
  const int len = (N + P - 1) / P;
  n0 = min(N, c * len);
  n1 = min(N, n0 + len);
}

// Each thread owns at most 8 tokens of its chunk (chunks hold at most
// 2048 = 256·8 tokens); its loads are all issued before any use.
constexpr int kSoftmaxPer = 8;

__global__ void __launch_bounds__(kSoftmaxThreads)
softmax_partial(const float2* __restrict__ z, float2* __restrict__ part, int N, int P) {
  __shared__ float red[32];
  const int row = blockIdx.x / P, c = blockIdx.x % P;
  int n0, n1;
  chunk_range(N, P, c, n0, n1);
  const float2* zr = z + (size_t)row * N;
  float2 v[kSoftmaxPer];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < kSoftmaxPer; ++k) {
    const int n = n0 + threadIdx.x + k * kSoftmaxThreads;
    v[k] = n < n1 ? zr[n] : make_float2(-INFINITY, 0.f);
  }
#pragma unroll
  for (int k = 0; k < kSoftmaxPer; ++k) m = fmaxf(m, v[k].x);
  m = block_reduce<true>(m, red);
  float s = 0.f;
  if (m > -INFINITY) {
#pragma unroll
    for (int k = 0; k < kSoftmaxPer; ++k)
      if (n0 + threadIdx.x + k * kSoftmaxThreads < n1) s += exp_shifted(v[k], m);
  }
  s = block_reduce<false>(s, red);
  if (threadIdx.x == 0) part[blockIdx.x] = make_float2(m, s);
}

__global__ void __launch_bounds__(kSoftmaxThreads)
softmax_finish(const float2* __restrict__ z, const float2* __restrict__ part, float* __restrict__ zs,
               int N, int P) {
  __shared__ float red[32];
  const int row = blockIdx.x / P, c = blockIdx.x % P;
  int n0, n1;
  chunk_range(N, P, c, n0, n1);
  const float2* zr = z + (size_t)row * N;
  float2 v[kSoftmaxPer];
#pragma unroll
  for (int k = 0; k < kSoftmaxPer; ++k) {
    const int n = n0 + threadIdx.x + k * kSoftmaxThreads;
    v[k] = n < n1 ? zr[n] : make_float2(0.f, 0.f);
  }
  const float2* pr = part + (size_t)row * P;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < P; i += blockDim.x) m = fmaxf(m, pr[i].x);
  m = block_reduce<true>(m, red);
  float S = 0.f;
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    float2 q = pr[i];
    if (q.y > 0.f) S += q.y * expf(q.x - m);
  }
  S = block_reduce<false>(S, red);
  const float inv = 1.0f / S;
  float* out = zs + (size_t)row * N;
#pragma unroll
  for (int k = 0; k < kSoftmaxPer; ++k) {
    const int n = n0 + threadIdx.x + k * kSoftmaxThreads;
    if (n < n1) out[n] = exp_shifted(v[k], m) * inv;
  }
}

int softmax_parts(int N) { return (N + 2047) / 2048; }

cudaError_t launch_softmax(const cat_plan_s* p, const Span& sp, bool finish) {
  const int rows = sp.nb(p) * p->H;
  if (rows == 0) return cudaSuccess;
  const int P = softmax_parts(p->N);
  const size_t r0 = (size_t)sp.b0 * p->H;
  const cudaStream_t st = sp.stream(p);
  softmax_partial<<<rows * P, kSoftmaxThreads, 0, st>>>(p->z2 + r0 * p->N, p->part + r0 * P, p->N,
                                                        P);
  if (finish)
    softmax_finish<<<rows * P, kSoftmaxThreads, 0, st>>>(p->z2 + r0 * p->N, p->part + r0 * P,
                                                         p->zs + r0 * p->N, p->N, P);
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
  if (p->dtype == 1) {
    cudaError_t e0 = score_mma(p, nullptr, nullptr, true);
    if (e0 == cudaSuccess) e0 = score_tma(p, nullptr, nullptr, true);
    if (e0 != cudaSuccess) return e0;
  }
  cudaError_t e = p->dtype == 1
      ? score_dispatch<__nv_bfloat16>(p, nullptr, nullptr, true)
      : score_dispatch<float>(p, nullptr, nullptr, true);
  if (e != cudaSuccess) return e;
  if (p->path == PATH_SMEM) e = allow_max_smem(softmax_spectrum_kernel);
  return e;
}

cudaError_t launch_softmax_spectrum(const cat_plan_s* p) {
  if (p->sm.reg_m) return launch_softmax_spectrum_reg(p);
  int rows = p->B * p->H;
  if (rows == 0) return cudaSuccess;
  softmax_spectrum_kernel<<<rows, p->sm.spec_threads, p->sm.spec_smem, p->stream>>>(
      p->z2, p->zs, p->zf, p->rpN, p->tw, p->status);
  return cudaGetLastError();
}

}  // namespace cat
