// Single-CTA circulant product for N up to 16384 — the "FFT acceleration"
// design of the notes page "CAT: Circular-Convolutional Attention for
// Sub-Quadratic Transformers" (section 关键设计):
//     O_h[:, c] = IFFT( FFT(z*_h) ⊙ FFT(V_h[:, c]) )
//
// Two real value columns (c, c+1) of one head are packed as one complex
// signal v = V[:, c] + i·V[:, c+1].  Because the kernel z* is real, the
// circular convolution maps real signals to real signals and is linear, so
// the real part of IFFT(Zf ⊙ FFT(v)) is column c's result and the imaginary
// part column c+1's.  The spectrum Zf is stored already divided by N.
//
// One CTA owns G pairs of one (b, h): it loads the N x 2G tile (rows of 2G
// contiguous elements), transforms the G signals in shared memory, multiplies
// by Zf, transforms back and stores.
#include <cuda_bf16.h>

#include "cat_internal.h"
#include "elem.cuh"

namespace cat {

template <typename T>
__global__ void __launch_bounds__(1024)
conv_smem_kernel(const T* __restrict__ V, T* __restrict__ O, const float2* __restrict__ zf,
                 const float2* __restrict__ W, RadixPlan rp, int D, int H, int dh, int npair,
                 int G, int groups, int tstride, unsigned int* status) {
  extern __shared__ float2 buf[];
  const int N = rp.L;
  const int bh = blockIdx.x / groups;
  const int grp = blockIdx.x - bh * groups;
  const int b = bh / H, h = bh - b * H;
  const int g0 = grp * G;
  const int gc = min(G, npair - g0);
  if (gc <= 0) return;
  if (gc * N > vals_capacity(rp) * (int)blockDim.x) {
    report(status, 0x201);
    return;
  }
  const int col0 = h * dh + 2 * g0;                 // first column of this CTA
  const bool full_pairs = (2 * (g0 + gc) <= dh);    // no half pair at the end
  // Pair loads need 2·sizeof(T) alignment in every row: an even column and
  // an even row length.
  const bool aligned = ((col0 & 1) == 0) && ((D & 1) == 0);
  const T* Vb = V + (size_t)b * N * D;
  T* Ob = O + (size_t)b * N * D;

  // Load: consecutive threads walk the 2·gc contiguous columns of a row.
  const int total = gc * N;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int n = idx / gc, g = idx - n * gc;
    const T* src = Vb + (size_t)n * D + col0 + 2 * g;
    float2 v;
    if (full_pairs && aligned) {
      v = ld_pair(src);
    } else {
      v.x = ld_elem(src);
      v.y = (2 * (g0 + g) + 1 < dh) ? ld_elem(src + 1) : 0.f;
    }
    buf[g * tstride + n] = v;
  }
  __syncthreads();

  block_fft<false>(buf, rp, gc, tstride, W, 1);

  const float2* zrow = zf + (size_t)bh * N;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int g = idx / N, k = idx - g * N;
    buf[g * tstride + k] = cmul(buf[g * tstride + k], __ldg(&zrow[k]));
  }
  __syncthreads();

  block_fft<true>(buf, rp, gc, tstride, W, 1);

  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int n = idx / gc, g = idx - n * gc;
    T* dst = Ob + (size_t)n * D + col0 + 2 * g;
    float2 v = buf[g * tstride + n];
    if (full_pairs && aligned) {
      st_pair(dst, v);
    } else {
      st_elem(dst, v.x);
      if (2 * (g0 + g) + 1 < dh) st_elem(dst + 1, v.y);
    }
  }
}

cudaError_t setup_smem_kernels(const cat_plan_s* p) {
  if (p->sm.reg_m) return setup_conv_reg(p);
  if (p->dtype == 1) return allow_max_smem(conv_smem_kernel<__nv_bfloat16>);
  return allow_max_smem(conv_smem_kernel<float>);
}

cudaError_t launch_conv_smem(const cat_plan_s* p, const void* V, void* O) {
  if (p->sm.reg_m) return launch_conv_reg(p, V, O);
  const int ctas = p->B * p->H * p->sm.groups;
  if (ctas == 0) return cudaSuccess;
  if (p->dtype == 1)
    conv_smem_kernel<__nv_bfloat16><<<ctas, p->sm.threads, p->sm.smem, p->stream>>>(
        (const __nv_bfloat16*)V, (__nv_bfloat16*)O, p->zf, p->tw, p->rpN, p->D, p->H, p->dh,
        p->npair, p->sm.G, p->sm.groups, p->sm.tstride, p->status);
  else
    conv_smem_kernel<float><<<ctas, p->sm.threads, p->sm.smem, p->stream>>>(
        (const float*)V, (float*)O, p->zf, p->tw, p->rpN, p->D, p->H, p->dh, p->npair, p->sm.G,
        p->sm.groups, p->sm.tstride, p->status);
  return cudaGetLastError();
}

}  // namespace cat
