// Device-side FFT building blocks: complex helpers, small DFTs of radix
// 2, 3, 4, 5, 7, 8, and a block-cooperative Stockham (self-sorting) pass
// over shared memory.
//
// The method these serve is the "FFT acceleration" design of the notes page
// "CAT: Circular-Convolutional Attention for Sub-Quadratic Transformers"
// (section 关键设计): circ(z*)·v = IFFT(FFT(z*) ⊙ FFT(v)).  Conventions:
// forward kernel exp(-2πi kn/L), inverse exp(+2πi kn/L) without 1/L (the
// 1/N factor is folded into the stored spectrum of z*).
//
// Stockham pass (radix R, sub-transform span Ls -> R·Ls, transform length L,
// M = L / (R·Ls)); for task i in [0, L/R), k = i mod Ls, p = i / Ls:
//     a_u  = x[i + u·L/R] · w_{R·Ls}^{u·k}          u = 0..R-1
//     y[p·R·Ls + k + Ls·s] = sum_u a_u · w_R^{u·s}   s = 0..R-1
// Starting from natural order with Ls = 1 and ending with Ls = L, the result
// is the DFT in natural order.  Twiddles w_{R·Ls}^{u·k} = W[u·k·M·(Ntab/L)]
// come from a table W[j] = exp(-2πi j/Ntab) built on the host in fp64.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace cat {

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cscale(float2 a, float s) { return make_float2(a.x * s, a.y * s); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
// a · conj(b)
__device__ __forceinline__ float2 cmulc(float2 a, float2 b) {
  return make_float2(fmaf(a.x, b.x, a.y * b.y), fmaf(a.y, b.x, -a.x * b.y));
}
// multiply by -i (forward quarter turn) or +i (inverse quarter turn)
template <bool INV>
__device__ __forceinline__ float2 rot90(float2 a) {
  return INV ? make_float2(-a.y, a.x) : make_float2(a.y, -a.x);
}

// Complex add and subtract for the register transforms: ordinary fp32
// component pairs, or the paired fp32 instructions of sm_100 and later (one
// instruction per complex add or subtract, the same rounding per component;
// a - b is b·(-1) + a, exact).
struct CxScalar {
  static __device__ __forceinline__ float2 add(float2 a, float2 b) { return cadd(a, b); }
  static __device__ __forceinline__ float2 sub(float2 a, float2 b) { return csub(a, b); }
};
struct CxPaired {
  static __device__ __forceinline__ float2 add(float2 a, float2 b) { return __fadd2_rn(a, b); }
  static __device__ __forceinline__ float2 sub(float2 a, float2 b) {
    return __ffma2_rn(b, make_float2(-1.f, -1.f), a);
  }
};

// Twiddle w or its conjugate.
template <bool INV>
__device__ __forceinline__ float2 twmul(float2 a, float2 w) {
  return INV ? cmulc(a, w) : cmul(a, w);
}

// ---------------------------------------------------------------------------
// Small DFTs on registers: b[s] = sum_u a[u] w_R^{±u s}, in place.
// Constants are cos/sin of 2πk/R.
// ---------------------------------------------------------------------------
template <bool INV, class Ops = CxScalar>
__device__ __forceinline__ void dft2(float2* a) {
  float2 t = a[0];
  a[0] = Ops::add(t, a[1]);
  a[1] = Ops::sub(t, a[1]);
}

template <bool INV>
__device__ __forceinline__ void dft3(float2* a) {
  const float S3 = 0.8660254037844386f;  // sin(2π/3)
  float2 t = cadd(a[1], a[2]);
  float2 d = csub(a[1], a[2]);
  float2 m = make_float2(fmaf(-0.5f, t.x, a[0].x), fmaf(-0.5f, t.y, a[0].y));
  float2 r = rot90<INV>(cscale(d, S3));  // ∓i·sin·d
  a[0] = cadd(a[0], t);
  a[1] = cadd(m, r);
  a[2] = csub(m, r);
}

template <bool INV, class Ops = CxScalar>
__device__ __forceinline__ void dft4(float2* a) {
  float2 t0 = Ops::add(a[0], a[2]), t1 = Ops::sub(a[0], a[2]);
  float2 t2 = Ops::add(a[1], a[3]), t3 = rot90<INV>(Ops::sub(a[1], a[3]));
  a[0] = Ops::add(t0, t2);
  a[2] = Ops::sub(t0, t2);
  a[1] = Ops::add(t1, t3);
  a[3] = Ops::sub(t1, t3);
}

template <bool INV>
__device__ __forceinline__ void dft5(float2* a) {
  const float C1 = 0.30901699437494745f, C2 = -0.8090169943749473f;
  const float S1 = 0.9510565162951535f, S2 = 0.5877852522924732f;
  float2 t1 = cadd(a[1], a[4]), d1 = csub(a[1], a[4]);
  float2 t2 = cadd(a[2], a[3]), d2 = csub(a[2], a[3]);
  float2 a0 = a[0];
  float2 m1 = make_float2(a0.x + C1 * t1.x + C2 * t2.x, a0.y + C1 * t1.y + C2 * t2.y);
  float2 m2 = make_float2(a0.x + C2 * t1.x + C1 * t2.x, a0.y + C2 * t1.y + C1 * t2.y);
  float2 r1 = rot90<INV>(make_float2(S1 * d1.x + S2 * d2.x, S1 * d1.y + S2 * d2.y));
  float2 r2 = rot90<INV>(make_float2(S2 * d1.x - S1 * d2.x, S2 * d1.y - S1 * d2.y));
  a[0] = cadd(a0, cadd(t1, t2));
  a[1] = cadd(m1, r1);
  a[4] = csub(m1, r1);
  a[2] = cadd(m2, r2);
  a[3] = csub(m2, r2);
}

template <bool INV>
__device__ __forceinline__ void dft7(float2* a) {
  const float C1 = 0.6234898018587336f, C2 = -0.22252093395631434f, C3 = -0.900968867902419f;
  const float S1 = 0.7818314824680298f, S2 = 0.9749279121818236f, S3 = 0.43388373911755823f;
  float2 t1 = cadd(a[1], a[6]), d1 = csub(a[1], a[6]);
  float2 t2 = cadd(a[2], a[5]), d2 = csub(a[2], a[5]);
  float2 t3 = cadd(a[3], a[4]), d3 = csub(a[3], a[4]);
  float2 a0 = a[0];
  // s = 1: cos(2πk/7), sin(2πk/7) for k = 1, 2, 3
  float2 m1 = make_float2(a0.x + C1 * t1.x + C2 * t2.x + C3 * t3.x,
                          a0.y + C1 * t1.y + C2 * t2.y + C3 * t3.y);
  float2 r1 = rot90<INV>(make_float2(S1 * d1.x + S2 * d2.x + S3 * d3.x,
                                     S1 * d1.y + S2 * d2.y + S3 * d3.y));
  // s = 2: angles 2, 4, 6 (·2π/7): cos c2, c3, c1; sin s2, -s3, -s1
  float2 m2 = make_float2(a0.x + C2 * t1.x + C3 * t2.x + C1 * t3.x,
                          a0.y + C2 * t1.y + C3 * t2.y + C1 * t3.y);
  float2 r2 = rot90<INV>(make_float2(S2 * d1.x - S3 * d2.x - S1 * d3.x,
                                     S2 * d1.y - S3 * d2.y - S1 * d3.y));
  // s = 3: angles 3, 6, 2: cos c3, c1, c2; sin s3, -s1, s2
  float2 m3 = make_float2(a0.x + C3 * t1.x + C1 * t2.x + C2 * t3.x,
                          a0.y + C3 * t1.y + C1 * t2.y + C2 * t3.y);
  float2 r3 = rot90<INV>(make_float2(S3 * d1.x - S1 * d2.x + S2 * d3.x,
                                     S3 * d1.y - S1 * d2.y + S2 * d3.y));
  a[0] = cadd(a0, cadd(t1, cadd(t2, t3)));
  a[1] = cadd(m1, r1);
  a[6] = csub(m1, r1);
  a[2] = cadd(m2, r2);
  a[5] = csub(m2, r2);
  a[3] = cadd(m3, r3);
  a[4] = csub(m3, r3);
}

template <bool INV, class Ops = CxScalar>
__device__ __forceinline__ void dft8(float2* a) {
  const float R2 = 0.7071067811865476f;  // cos(π/4)
  float2 e[4] = {a[0], a[2], a[4], a[6]};
  float2 o[4] = {a[1], a[3], a[5], a[7]};
  dft4<INV, Ops>(e);
  dft4<INV, Ops>(o);
  // o[k] *= w8^{±k}
  float2 o1 = o[1], o3 = o[3];
  if (!INV) {
    o[1] = make_float2(R2 * (o1.x + o1.y), R2 * (o1.y - o1.x));
    o[3] = make_float2(R2 * (o3.y - o3.x), -R2 * (o3.x + o3.y));
  } else {
    o[1] = make_float2(R2 * (o1.x - o1.y), R2 * (o1.x + o1.y));
    o[3] = make_float2(-R2 * (o3.x + o3.y), R2 * (o3.x - o3.y));
  }
  o[2] = rot90<INV>(o[2]);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a[k] = Ops::add(e[k], o[k]);
    a[k + 4] = Ops::sub(e[k], o[k]);
  }
}

template <int R, bool INV>
__device__ __forceinline__ void dft_small(float2* a) {
  if constexpr (R == 2) dft2<INV>(a);
  else if constexpr (R == 3) dft3<INV>(a);
  else if constexpr (R == 4) dft4<INV>(a);
  else if constexpr (R == 5) dft5<INV>(a);
  else if constexpr (R == 7) dft7<INV>(a);
  else if constexpr (R == 8) dft8<INV>(a);
  else static_assert(R == 2, "unsupported radix");
}

// ---------------------------------------------------------------------------
// Radix plan for one transform length: up to 24 passes, each radix in
// {2, 3, 4, 5, 7, 8}; product of radices = L.
// ---------------------------------------------------------------------------
constexpr int kMaxPasses = 24;
struct RadixPlan {
  int L;                    // transform length
  int npass;                // number of passes
  int radix[kMaxPasses];
};

// Values each thread may hold in registers during one pass.
constexpr int kMaxValsPerThread = 32;

// Largest count·L one thread can cover in every pass of `rp`: a pass of
// radix R holds floor(32/R) tasks of R values per thread.
__host__ __device__ inline int vals_capacity(const RadixPlan& rp) {
  int cap = kMaxValsPerThread;
  for (int s = 0; s < rp.npass; ++s) {
    int c = (kMaxValsPerThread / rp.radix[s]) * rp.radix[s];
    if (c < cap) cap = c;
  }
  return cap;
}

// One in-place Stockham pass of radix R over `count` transforms of length L
// stored at buf[t·tstride + j].  Every thread first loads all of its tasks,
// the block synchronises, then each thread writes its results; so the pass
// is safe in place.  Requires count·L/R <= (kMaxValsPerThread/R)·blockDim.
template <int R, bool INV>
__device__ __forceinline__ void stockham_pass(float2* buf, int L, int Ls, int count, int tstride,
                                              const float2* __restrict__ W, int wstep) {
  constexpr int TMAX = kMaxValsPerThread / R;
  const int per = L / R;            // tasks per transform
  const int ntask = count * per;
  const int M = per / Ls;           // = L / (R·Ls)
  float2 a[TMAX][R];
#pragma unroll
  for (int j = 0; j < TMAX; ++j) {
    int task = threadIdx.x + j * blockDim.x;
    if (task < ntask) {
      int t = task / per, i = task - t * per;
      const float2* src = buf + (size_t)t * tstride + i;
#pragma unroll
      for (int u = 0; u < R; ++u) a[j][u] = src[u * per];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < TMAX; ++j) {
    int task = threadIdx.x + j * blockDim.x;
    if (task < ntask) {
      int t = task / per, i = task - t * per;
      int k = i % Ls, p = i / Ls;
      if (Ls > 1) {
#pragma unroll
        for (int u = 1; u < R; ++u) {
          float2 w = __ldg(&W[(size_t)(u * k * M) * wstep]);
          a[j][u] = twmul<INV>(a[j][u], w);
        }
      }
      dft_small<R, INV>(a[j]);
      float2* dst = buf + (size_t)t * tstride + p * R * Ls + k;
#pragma unroll
      for (int s = 0; s < R; ++s) dst[s * Ls] = a[j][s];
    }
  }
  __syncthreads();
}

// Full transform: all passes of `rp` over `count` transforms in shared memory.
// W is a table of Ntab = L·wstep entries.
template <bool INV>
__device__ void block_fft(float2* buf, const RadixPlan& rp, int count, int tstride,
                          const float2* __restrict__ W, int wstep) {
  int Ls = 1;
  for (int s = 0; s < rp.npass; ++s) {
    int R = rp.radix[s];
    switch (R) {
      case 2: stockham_pass<2, INV>(buf, rp.L, Ls, count, tstride, W, wstep); break;
      case 3: stockham_pass<3, INV>(buf, rp.L, Ls, count, tstride, W, wstep); break;
      case 4: stockham_pass<4, INV>(buf, rp.L, Ls, count, tstride, W, wstep); break;
      case 5: stockham_pass<5, INV>(buf, rp.L, Ls, count, tstride, W, wstep); break;
      case 7: stockham_pass<7, INV>(buf, rp.L, Ls, count, tstride, W, wstep); break;
      default: stockham_pass<8, INV>(buf, rp.L, Ls, count, tstride, W, wstep); break;
    }
    Ls *= R;
  }
}

// Device status word helpers: kernels record the first failed internal check
// here instead of trapping.
__device__ __forceinline__ void report(unsigned int* status, unsigned int code) {
  if (status) atomicCAS(status, 0u, code);
}

}  // namespace cat
