// df.cuh -- double-float arithmetic on the fp32 pipes of sm_103a.
//
// A double-float value is the unevaluated sum hi + lo of two fp32 numbers
// (float2 {x = hi, y = lo}), which carries about 44-48 significant bits.
// GB300 has only a token FP64 rate, while the BaKron error feedback needs
// far more than fp32's 24 bits to reproduce the exact rounding decisions
// (a single near-tie flipped by fp32 error cascades through the factors),
// so all solver state is kept in this form.
//
// Building blocks (Dekker 1971; Knuth TAOCP vol. 2, 4.2.2):
//   two_sum       s + e = a + b exactly (6 adds)
//   fast_two_sum  the same when |a| >= |b| (3 adds)
//   two_prod      p + e = a * b exactly (mul + fma)
// and the offset accumulator below.
//
// Offset accumulator (after Rump, Ogita and Oishi, "Accurate floating-point
// summation, part I: faithful rounding", SIAM J. Sci. Comput. 2008, whose
// ExtractScalar splits a number against a power-of-two offset sigma):
// the running sum S is held as H = sigma + S plus a low word L.  Adding a
// product x*y is
//     Hn = fma(x, y, H);  d = H - Hn;  r = fma(x, y, d);  L += r;  H = Hn
// where d is exact (Sterbenz: H and Hn are within a factor 2 of each other
// while |S| < sigma/2 and every term is small against sigma) and r is the
// exact rounding error of the first fma (itself rounded once, a relative
// 2^-24 of an already tiny number).  With the low word of a double-float
// operand folded into L by one more fma, one double-float MAC costs 5 fp32
// instructions and loses nothing but the rounding of L, about
// 2^-48 * sigma * sqrt(#terms).
#pragma once

#include <cuda_runtime.h>

namespace bakron {

__device__ __forceinline__ float2 two_sum(float a, float b) {
  float s = a + b;
  float bb = s - a;
  float e = (a - (s - bb)) + (b - bb);
  return make_float2(s, e);
}

__device__ __forceinline__ float2 fast_two_sum(float a, float b) {
  float s = a + b;
  float e = b - (s - a);
  return make_float2(s, e);
}

// Normalized sum of two double-floats.
__device__ __forceinline__ float2 df_add(float2 a, float2 b) {
  float2 s = two_sum(a.x, b.x);
  float2 t = two_sum(a.y, b.y);
  s.y += t.x;
  s = fast_two_sum(s.x, s.y);
  s.y += t.y;
  return fast_two_sum(s.x, s.y);
}

__device__ __forceinline__ float2 df_neg(float2 a) { return make_float2(-a.x, -a.y); }

__device__ __forceinline__ float2 df_sub(float2 a, float2 b) { return df_add(a, df_neg(b)); }

// Exact product of two fp32 numbers as a double-float.
__device__ __forceinline__ float2 two_prod(float a, float b) {
  float p = a * b;
  return make_float2(p, fmaf(a, b, -p));
}

// Double-float product (normalized), about 2^-46 relative error.
__device__ __forceinline__ float2 df_mul(float2 a, float2 b) {
  float p = a.x * b.x;
  float e = fmaf(a.x, b.x, -p);
  e = fmaf(a.x, b.y, e);
  e = fmaf(a.y, b.x, e);
  return fast_two_sum(p, e);
}

// Double-float quotient a / b (normalized).
__device__ __forceinline__ float2 df_div(float2 a, float2 b) {
  float q1 = __fdiv_rn(a.x, b.x);
  float2 r = df_sub(a, df_mul(make_float2(q1, 0.f), b));
  float q2 = __fdiv_rn(r.x, b.x);
  return fast_two_sum(q1, q2);
}

// Offset accumulator: value = (H - sigma) + L.
struct OffsetAcc {
  float H, L;

  __device__ __forceinline__ void init(float sigma) {
    H = sigma;
    L = 0.f;
  }
  // += x * y   (x fp32, y fp32)
  __device__ __forceinline__ void mac(float x, float y) {
    float Hn = fmaf(x, y, H);
    float d = H - Hn;
    L += fmaf(x, y, d);
    H = Hn;
  }
  // += x * (y.hi + y.lo)   (x fp32, y double-float)
  __device__ __forceinline__ void mac(float x, float2 y) {
    float Hn = fmaf(x, y.x, H);
    float d = H - Hn;
    L += fmaf(x, y.x, d);
    L = fmaf(x, y.y, L);
    H = Hn;
  }
  // += (x.hi + x.lo) * (y.hi + y.lo)   (both double-float; lo*lo dropped)
  __device__ __forceinline__ void mac(float2 x, float2 y) {
    float Hn = fmaf(x.x, y.x, H);
    float d = H - Hn;
    L += fmaf(x.x, y.x, d);
    L = fmaf(x.x, y.y, L);
    L = fmaf(x.y, y.x, L);
    H = Hn;
  }
  // Normalized double-float value.
  __device__ __forceinline__ float2 value(float sigma) const { return two_sum(H - sigma, L); }
};

// Power-of-two offset sigma in (4 * bound, 8 * bound] for sums bounded by `bound`.
__host__ __device__ __forceinline__ float offset_for_bound(float bound) {
  float b = bound > 1e-30f ? bound : 1e-30f;
  int e;
  frexpf(4.0f * b, &e);  // 4b = f * 2^e with f in [0.5, 1)
  return ldexpf(1.0f, e);
}

}  // namespace bakron
