// Long-sequence circulant product (N above the single-CTA limit): the
// "FFT acceleration" design of the notes page "CAT: Circular-Convolutional
// Attention for Sub-Quadratic Transformers" (section 关键设计),
//     O_h[:, c] = IFFT( FFT(z*_h) ⊙ FFT(V_h[:, c]) ),
// evaluated with the four-step split N = N1·N2, n = n1 + N1·n2,
// k = N2·k1 + k2:
//     FFT(x)[N2 k1 + k2] = sum_n1 w_N1^{n1 k1} · w_N^{n1 k2} · A[n1, k2],
//     A[n1, k2]          = sum_n2 w_N2^{n2 k2} · x[n1 + N1 n2].
// Pass A (per n1): length-N2 DFTs of V's column pairs and of z*, times the
//   twiddle w_N^{n1 k2}, into scratch.
// Pass B (per k2): length-N1 DFTs give both spectra at bins N2 k1 + k2; the
//   pair spectra are multiplied by FFT(z*)/N, transformed back over k1 and
//   multiplied by the conjugate twiddle.  The spectrum is never reordered:
//   the product is taken in the order the forward pass leaves it.
// Pass C (per n1): inverse length-N2 DFTs over k2 give the output rows
//   n1 + N1 n2.
// Column pairs (c, c+1) are packed as one complex signal, exactly as in the
// shared-memory path: the kernel z* is real, so the real and imaginary parts
// stay separate through the whole product.
// Without the twiddles (template flag TW = false) the same passes compute
// the 2-D DFT over an h x w token grid (N1 = w, N2 = h, n = x + w·y): the
// BCCB product of the page "Vision Transformers are Circulant Attention
// Learners", O = σ(a) ⊛ V, a 2-D circular convolution.
#include <cuda_bf16.h>

#include "cat_internal.h"
#include "elem.cuh"

namespace cat {

// Pass A.  blockIdx.x = (bhl · (N1/TA) + tile) · groups + grp.
// Shared layout: signal (t, s) at buf[(t·S + s)·N2]; s < gc are the CTA's
// pairs, s = gc is z* (only in group 0).
template <typename T, bool TW>
__global__ void __launch_bounds__(1024)
fs_pass_a(const T* __restrict__ V, const float* __restrict__ zs, float2* __restrict__ scr,
          const float2* __restrict__ W, RadixPlan rp2, int N, int N1, int D, int H, int dh,
          int npair, int G, int groups, int TA, int P, int bh0, unsigned int* status) {
  extern __shared__ float2 buf[];
  const int N2 = rp2.L;
  const int ntile = N1 / TA;
  int r = blockIdx.x;
  const int grp = r % groups; r /= groups;
  const int tile = r % ntile;
  const int bhl = r / ntile;
  const int bh = bh0 + bhl;
  const int b = bh / H, h = bh - b * H;
  const int g0 = grp * G;
  const int gc = min(G, npair - g0);
  const bool with_z = (grp == 0);
  const int S = gc + (with_z ? 1 : 0);
  const int count = TA * S;
  if (gc <= 0) return;
  if (count * N2 > vals_capacity(rp2) * (int)blockDim.x) {
    report(status, 0x301);
    return;
  }
  const int n1_0 = tile * TA;
  const int col0 = h * dh + 2 * g0;
  const bool full_pairs = (2 * (g0 + gc) <= dh);
  const bool aligned = ((col0 & 1) == 0) && ((D & 1) == 0);   // even column, even row length
  const T* Vb = V + (size_t)b * N * D;
  const float* zrow = zs + (size_t)bh * N;

  // Load: s fastest (contiguous pairs of one row), then t, then n2.
  const int total = count * N2;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int s = idx % S, q = idx / S;
    int t = q % TA, n2 = q / TA;
    int n = n1_0 + t + N1 * n2;
    float2 v;
    if (s < gc) {
      const T* src = Vb + (size_t)n * D + col0 + 2 * s;
      if (full_pairs && aligned) {
        v = ld_pair(src);
      } else {
        v.x = ld_elem(src);
        v.y = (2 * (g0 + s) + 1 < dh) ? ld_elem(src + 1) : 0.f;
      }
    } else {
      v = make_float2(__ldg(zrow + n), 0.f);
    }
    buf[(t * S + s) * N2 + n2] = v;
  }
  __syncthreads();
  block_fft<false>(buf, rp2, count, N2, W, N1);

  // Twiddle and store: scratch[bhl][k2][n1][p].
  float2* srow = scr + (size_t)bhl * N * P;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int s = idx % S, q = idx / S;
    int t = q % TA, k2 = q / TA;
    int n1 = n1_0 + t;
    float2 v = buf[(t * S + s) * N2 + k2];
    if (TW) v = cmul(v, __ldg(&W[(size_t)n1 * k2]));
    int pidx = (s < gc) ? g0 + s : npair;
    srow[((size_t)k2 * N1 + n1) * P + pidx] = v;
  }
}

// Pass B.  blockIdx.x = (bhl · (N2/TB) + tile) · groups + grp.
// Shared layout: pair signal (t, s) at buf[(t·gc + s)·N1], z* of k2-slot t
// at buf[(TB·gc + t)·N1].
template <bool TW>
__global__ void __launch_bounds__(1024)
fs_pass_b(float2* __restrict__ scr, const float2* __restrict__ W, RadixPlan rp1, int N,
          int N2, int npair, int G, int groups, int TB, int P, unsigned int* status) {
  extern __shared__ float2 buf[];
  const int N1 = rp1.L;
  const int ntile = N2 / TB;
  int r = blockIdx.x;
  const int grp = r % groups; r /= groups;
  const int tile = r % ntile;
  const int bhl = r / ntile;
  const int g0 = grp * G;
  const int gc = min(G, npair - g0);
  if (gc <= 0) return;
  const int S = gc + 1;
  const int count = TB * S;
  if (count * N1 > vals_capacity(rp1) * (int)blockDim.x) {
    report(status, 0x302);
    return;
  }
  const int k2_0 = tile * TB;
  float2* srow = scr + (size_t)bhl * N * P;

  const int total = count * N1;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int s = idx % S, q = idx / S;
    int n1 = q % N1, t = q / N1;
    int k2 = k2_0 + t;
    int pidx = (s < gc) ? g0 + s : npair;
    float2 v = srow[((size_t)k2 * N1 + n1) * P + pidx];
    int slot = (s < gc) ? (t * gc + s) : (TB * gc + t);
    buf[slot * N1 + n1] = v;
  }
  __syncthreads();
  block_fft<false>(buf, rp1, count, N1, W, N2);

  // Product with the spectrum of z* (divided by N).
  const float invN = 1.0f / (float)N;
  const int npts = TB * N1;
  for (int idx = threadIdx.x; idx < npts; idx += blockDim.x) {
    int k1 = idx % N1, t = idx / N1;
    float2 zf = cscale(buf[(TB * gc + t) * N1 + k1], invN);
    for (int s = 0; s < gc; ++s) {
      float2* e = &buf[(t * gc + s) * N1 + k1];
      *e = cmul(*e, zf);
    }
  }
  __syncthreads();
  block_fft<true>(buf, rp1, TB * gc, N1, W, N2);

  // Conjugate twiddle w_N^{-n1 k2} and store the pairs back.
  const int tot2 = TB * gc * N1;
  for (int idx = threadIdx.x; idx < tot2; idx += blockDim.x) {
    int s = idx % gc, q = idx / gc;
    int n1 = q % N1, t = q / N1;
    int k2 = k2_0 + t;
    float2 v = buf[(t * gc + s) * N1 + n1];
    if (TW) v = cmulc(v, __ldg(&W[(size_t)n1 * k2]));
    srow[((size_t)k2 * N1 + n1) * P + g0 + s] = v;
  }
}

// Pass C.  Same grid as pass A.  Shared layout: signal (t, s) at
// buf[(t·gc + s)·N2].
template <typename T>
__global__ void __launch_bounds__(1024)
fs_pass_c(const float2* __restrict__ scr, T* __restrict__ O, const float2* __restrict__ W,
          RadixPlan rp2, int N, int N1, int D, int H, int dh, int npair, int G, int groups,
          int TA, int P, int bh0, unsigned int* status) {
  extern __shared__ float2 buf[];
  const int N2 = rp2.L;
  const int ntile = N1 / TA;
  int r = blockIdx.x;
  const int grp = r % groups; r /= groups;
  const int tile = r % ntile;
  const int bhl = r / ntile;
  const int bh = bh0 + bhl;
  const int b = bh / H, h = bh - b * H;
  const int g0 = grp * G;
  const int gc = min(G, npair - g0);
  if (gc <= 0) return;
  const int count = TA * gc;
  if (count * N2 > vals_capacity(rp2) * (int)blockDim.x) {
    report(status, 0x303);
    return;
  }
  const int n1_0 = tile * TA;
  const int col0 = h * dh + 2 * g0;
  const bool full_pairs = (2 * (g0 + gc) <= dh);
  const bool aligned = ((col0 & 1) == 0) && ((D & 1) == 0);   // even column, even row length
  const float2* srow = scr + (size_t)bhl * N * P;

  const int total = count * N2;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int s = idx % gc, q = idx / gc;
    int t = q % TA, k2 = q / TA;
    buf[(t * gc + s) * N2 + k2] = srow[((size_t)k2 * N1 + n1_0 + t) * P + g0 + s];
  }
  __syncthreads();
  block_fft<true>(buf, rp2, count, N2, W, N1);

  T* Ob = O + (size_t)b * N * D;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    int s = idx % gc, q = idx / gc;
    int t = q % TA, n2 = q / TA;
    int n = n1_0 + t + N1 * n2;
    float2 v = buf[(t * gc + s) * N2 + n2];
    T* dst = Ob + (size_t)n * D + col0 + 2 * s;
    if (full_pairs && aligned) {
      st_pair(dst, v);
    } else {
      st_elem(dst, v.x);
      if (2 * (g0 + s) + 1 < dh) st_elem(dst + 1, v.y);
    }
  }
}

template <typename T>
static cudaError_t setup_t(const cat_plan_s* p) {
  cudaError_t e = p->twod ? allow_max_smem(fs_pass_a<T, false>) : allow_max_smem(fs_pass_a<T, true>);
  if (e == cudaSuccess) e = allow_max_smem(fs_pass_c<T>);
  if (e == cudaSuccess) e = p->twod ? allow_max_smem(fs_pass_b<false>) : allow_max_smem(fs_pass_b<true>);
  return e;
}

cudaError_t setup_fourstep_kernels(const cat_plan_s* p) {
  return p->dtype == 1 ? setup_t<__nv_bfloat16>(p) : setup_t<float>(p);
}

template <typename T, bool TW>
static cudaError_t run_t(const cat_plan_s* p, const T* V, T* O) {
  const FourStepCfg& f = p->fs;
  const int rows = p->B * p->H;
  for (int bh0 = 0; bh0 < rows; bh0 += f.chunk_bh) {
    int nb = rows - bh0 < f.chunk_bh ? rows - bh0 : f.chunk_bh;
    int ga = nb * (f.N1 / f.TA) * f.groups;
    fs_pass_a<T, TW><<<ga, f.threadsA, f.smemA, p->stream>>>(
        V, p->zs, p->scratch, p->tw, f.rp2, p->N, f.N1, p->D, p->H, p->dh, p->npair, f.G,
        f.groups, f.TA, f.P, bh0, p->status);
    int gb = nb * (f.N2 / f.TB) * f.groups;
    fs_pass_b<TW><<<gb, f.threadsB, f.smemB, p->stream>>>(p->scratch, p->tw, f.rp1, p->N, f.N2,
                                                           p->npair, f.G, f.groups, f.TB, f.P,
                                                           p->status);
    fs_pass_c<T><<<ga, f.threadsC, f.smemC, p->stream>>>(
        p->scratch, O, p->tw, f.rp2, p->N, f.N1, p->D, p->H, p->dh, p->npair, f.G, f.groups,
        f.TA, f.P, bh0, p->status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_fourstep_conv(const cat_plan_s* p, const void* V, void* O) {
  if (p->B == 0) return cudaSuccess;
  // A 2-D plan (N1 = w, N2 = h) takes the passes without the inter-pass
  // twiddle: their two DFTs are then the 2-D DFT over the token grid.
  if (p->twod) {
    if (p->dtype == 1) return run_t<__nv_bfloat16, false>(p, (const __nv_bfloat16*)V, (__nv_bfloat16*)O);
    return run_t<float, false>(p, (const float*)V, (float*)O);
  }
  if (p->dtype == 1) return run_t<__nv_bfloat16, true>(p, (const __nv_bfloat16*)V, (__nv_bfloat16*)O);
  return run_t<float, true>(p, (const float*)V, (float*)O);
}

}  // namespace cat
