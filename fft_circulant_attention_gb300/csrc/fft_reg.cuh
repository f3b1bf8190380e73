// Register-resident DFT building blocks for lengths 1, 2, 3, 4, 7, 8, 12, 14,
// 16, 32 and 64.
//
// The method they serve is the "FFT acceleration" design of the notes page
// "CAT: Circular-Convolutional Attention for Sub-Quadratic Transformers"
// (section 关键设计): circ(z*)·v = IFFT(FFT(z*) ⊙ FFT(v)).  Forward kernel
// exp(-2πi kn/R), inverse exp(+2πi kn/R), neither scaled.
//
// dft<R, INV>(a) transforms R values held in registers, in place, natural
// order in and out.  Lengths 12, 14, 16, 32 and 64 are split R = P·Q with
// n = P·n1 + n2 and k = Q·k2 + k1:
//     X[Q k2 + k1] = sum_n2 w_P^{n2 k2} · w_R^{n2 k1} · sum_n1 a[P n1 + n2] w_Q^{n1 k1},
// i.e. P DFTs of length Q, a twiddle per (n2, k1), Q DFTs of length P.
// Every index and twiddle angle is a compile-time constant, so the whole
// transform unrolls into straight-line code with immediate constants; the
// constants come from a constexpr Taylor series on the reduced angle.
#pragma once
#include <cuda_runtime.h>

#include <type_traits>

#include "fft_device.cuh"

namespace cat {

// ---------------------------------------------------------------------------
// Compile-time trigonometry: cos and sin of 2π·e/R for integers e, R.
// The angle is reduced by the symmetries of the circle to [0, π/4] and the
// Taylor series is summed in double (error below 2e-16 there).
// ---------------------------------------------------------------------------
struct CS {
  double c, s;
};

constexpr double kTwoPi = 6.283185307179586476925286766559;

constexpr CS taylor_cs(double x) {
  double c = 1.0, s = x, tc = 1.0, ts = x;
  for (int k = 1; k < 14; ++k) {
    tc *= -x * x / ((2.0 * k - 1.0) * (2.0 * k));
    ts *= -x * x / ((2.0 * k) * (2.0 * k + 1.0));
    c += tc;
    s += ts;
  }
  return CS{c, s};
}

// cos, sin of 2π·e/R (R > 0).
constexpr CS turn_cs(long e, long R) {
  e %= R;
  if (e < 0) e += R;
  if (2 * e >= R) {                      // θ = π + θ'
    CS t = turn_cs(e * 2 - R, 2 * R);
    return CS{-t.c, -t.s};
  }
  if (4 * e >= R) {                      // θ = π/2 + θ'
    CS t = turn_cs(e * 4 - R, 4 * R);
    return CS{-t.s, t.c};
  }
  if (8 * e > R) {                       // θ = π/2 - θ'
    CS t = turn_cs(R - 4 * e, 4 * R);
    return CS{t.s, t.c};
  }
  return taylor_cs(kTwoPi * (double)e / (double)R);
}

template <int I, int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for<I + 1, N>(f);
  }
}

// a · w_R^{±E} with w_R = exp(-2πi/R): forward multiplies by
// cos(2πE/R) - i sin(2πE/R), inverse by its conjugate.
template <int R, int E, bool INV>
__device__ __forceinline__ float2 twc(float2 a) {
  constexpr int e = ((E % R) + R) % R;
  if constexpr (e == 0) {
    return a;
  } else if constexpr (2 * e == R) {
    return make_float2(-a.x, -a.y);
  } else if constexpr (4 * e == R) {
    return rot90<INV>(a);               // forward: ·(-i)
  } else if constexpr (4 * e == 3 * R) {
    return rot90<!INV>(a);              // forward: ·(+i)
  } else {
    constexpr CS cs = turn_cs(e, R);
    constexpr float wr = (float)cs.c;
    constexpr float wi = INV ? (float)cs.s : (float)-cs.s;
    return make_float2(fmaf(a.x, wr, -a.y * wi), fmaf(a.x, wi, a.y * wr));
  }
}

// Ops: the complex add/subtract policy (CxScalar, or CxPaired for the paired
// fp32 instructions).
template <int R, bool INV, class Ops = CxScalar>
__device__ __forceinline__ void dft(float2* a);

// R = P·Q split (see the file comment).
template <int P, int Q, bool INV, class Ops>
__device__ __forceinline__ void dft_pq(float2* a) {
  constexpr int R = P * Q;
  float2 y[P][Q];
  static_for<0, P>([&](auto n2c) {
    constexpr int n2 = decltype(n2c)::value;
    float2 t[Q];
#pragma unroll
    for (int n1 = 0; n1 < Q; ++n1) t[n1] = a[P * n1 + n2];
    dft<Q, INV, Ops>(t);
    static_for<0, Q>([&](auto k1c) {
      constexpr int k1 = decltype(k1c)::value;
      y[n2][k1] = twc<R, n2 * k1, INV>(t[k1]);
    });
  });
#pragma unroll
  for (int k1 = 0; k1 < Q; ++k1) {
    float2 t[P];
#pragma unroll
    for (int n2 = 0; n2 < P; ++n2) t[n2] = y[n2][k1];
    dft<P, INV, Ops>(t);
#pragma unroll
    for (int k2 = 0; k2 < P; ++k2) a[Q * k2 + k1] = t[k2];
  }
}

template <int R, bool INV, class Ops>
__device__ __forceinline__ void dft(float2* a) {
  if constexpr (R == 1) {
  } else if constexpr (R == 2) {
    dft2<INV, Ops>(a);
  } else if constexpr (R == 3) {
    dft3<INV>(a);
  } else if constexpr (R == 4) {
    dft4<INV, Ops>(a);
  } else if constexpr (R == 7) {
    dft7<INV>(a);
  } else if constexpr (R == 8) {
    dft8<INV, Ops>(a);
  } else if constexpr (R == 12) {
    dft_pq<4, 3, INV, Ops>(a);
  } else if constexpr (R == 14) {
    dft_pq<2, 7, INV, Ops>(a);
  } else if constexpr (R == 16) {
    dft_pq<4, 4, INV, Ops>(a);
  } else if constexpr (R == 32) {
    dft_pq<4, 8, INV, Ops>(a);
  } else if constexpr (R == 64) {
    dft_pq<8, 8, INV, Ops>(a);
  } else {
    static_assert(R == 2, "dft: unsupported length");
  }
}

// Complex multiply by a runtime twiddle, forward (w) or inverse (conj w).
template <bool INV>
__device__ __forceinline__ float2 twr(float2 a, float2 w) {
  return INV ? cmulc(a, w) : cmul(a, w);
}

}  // namespace cat
