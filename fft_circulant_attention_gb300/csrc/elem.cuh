// Element load/store helpers: fp32 or bf16 storage, fp32 arithmetic.
// bf16 -> fp32 is exact; fp32 -> bf16 rounds to nearest-even.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace cat {

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start before the kernel ahead of it in the stream has
// finished (once every CTA of that kernel has run pdl_trigger or exited);
// pdl_wait blocks until that kernel has completed and its memory is
// visible.  Launched the ordinary way, both are no-ops.  A kernel that is
// launched this way calls pdl_wait before it touches memory the kernels
// ahead of it write, and before it exits, so that completion stays
// transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// A load of the kernel ahead's output after pdl_wait.  A load through a
// const __restrict__ pointer may be compiled as an invariant (read-only
// cache) load and moved above the wait; this one is ordered after it.
__device__ __forceinline__ float2 ld_dep(const float2* p) {
  float2 v;
  asm volatile("ld.global.v2.f32 {%0, %1}, [%2];"
               : "=f"(v.x), "=f"(v.y)
               : "l"(__cvta_generic_to_global(p))
               : "memory");
  return v;
}

__device__ __forceinline__ float ld_elem(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p) {
  unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(p));
  return __uint_as_float(((unsigned int)u) << 16);
}
__device__ __forceinline__ void st_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Two adjacent elements (a packed column pair), 2·sizeof(T)-aligned.
__device__ __forceinline__ float2 ld_pair(const float* p) { return __ldg(reinterpret_cast<const float2*>(p)); }
__device__ __forceinline__ float2 ld_pair(const __nv_bfloat16* p) {
  unsigned int u = __ldg(reinterpret_cast<const unsigned int*>(p));
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ void st_pair(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void st_pair(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

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

// Warp and block reductions.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Block-wide reduction; `red` is >= 32 floats of shared memory.  All threads
// get the result.
template <bool MAX>
__device__ __forceinline__ float block_reduce(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = MAX ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : (MAX ? -INFINITY : 0.f);
  r = MAX ? warp_max(r) : warp_sum(r);
  return r;
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

// Softmax statistics of one (b, h) row from its P chunk partials (m_c, s_c):
// sh[0] = m = max m_c, sh[1] = 1 / S with S = sum s_c·exp(m_c - m).  Warp 0
// combines; every thread of the CTA must call it (it ends with
// __syncthreads).
__device__ __forceinline__ void row_softmax_stats(const float2* __restrict__ part, int P,
                                                  float* sh) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float m = -INFINITY;
    for (int i = lane; i < P; i += 32) m = fmaxf(m, part[i].x);
    m = warp_max(m);
    float S = 0.f;
    for (int i = lane; i < P; i += 32) {
      const float2 q = part[i];
      if (q.y > 0.f) S += q.y * expf(q.x - m);
    }
    S = warp_sum(S);
    if (lane == 0) {
      sh[0] = m;
      sh[1] = 1.0f / S;
    }
  }
  __syncthreads();
}

}  // namespace cat
