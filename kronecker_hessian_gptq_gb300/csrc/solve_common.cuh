// solve_common.cuh -- pieces shared by the two BaKron solve schedules
// (the launch-per-step tile wavefront in quantize.cu and the persistent
// band sweep in sweep.cu): the workspace header, the input check and the
// accumulator offset, the fixed-point form of the chunk planes, the bf16
// digit split of solver values, and the per-(row, chunk) exponents and
// packed bf16 digits of the factors that the tensor-core products read.
//
// "BaKron: Efficient Quantization with Kronecker-Factored Hessians":
// the products L_B E L_A^T of App. B eq. (1), computed exactly on the
// tensor cores through integer digits (see the chunk products' comment in
// quantize.cu), need the factors and the solver values split into bf16
// digits on known exponents; this header holds those splits.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "bakron.h"
#include "df.cuh"

namespace bakron {
namespace {

constexpr int T = 32;            // tile edge
constexpr int B = 4;             // tiles per chunk
constexpr int CK = B * T;        // chunk depth (128)
constexpr int kDigF = 5;         // digits of a factor element
constexpr int kDigD = 6;         // digits of a solver value
constexpr int kLevels = 6;       // levels 0 .. kDigD - 1 of the digit products
constexpr int kSlab = 32;        // k per slab of factor digits

struct Header {
  unsigned maxw_bits;  // max |W| as ordered uint bits
  unsigned maxs_bits;  // max row (or group) scale
  unsigned maxc_bits;  // max column scale
  float sigma;         // offset of the offset accumulators
  int abort;           // set by a bounded wait that gave up (persistent sweep)
  unsigned queue_head; // persistent sweep: next ready-queue position to serve
  unsigned queue_tail; // persistent sweep: next ready-queue position to fill
  int pad[57];
};
static_assert(sizeof(Header) == 256, "header is one alignment unit");

// The inputs the prepass checks.
struct InputDesc {
  const float* W;
  const float* scales;   // m x ngroups row (group) scales, or null
  const float* cscales;  // n column scales, or null
  int ngroups, m, n, bits, lo, hi;
  Header* hdr;
  int32_t* status;
};

__device__ __forceinline__ unsigned warp_max(unsigned v) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Checks the inputs and finds max |W| and max scale.
__global__ void prepass_kernel(InputDesc P) {
  const size_t total = (size_t)P.m * P.n;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  unsigned wmax = 0, smax = 0, cmax = 0;
  int bad = 0;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const float w = P.W[idx];
    if (!isfinite(w)) {
      bad |= BAKRON_DEV_NONFINITE_W;
    } else {
      wmax = max(wmax, __float_as_uint(fabsf(w)));
    }
  }
  if (P.scales) {
    const size_t ns = (size_t)P.m * P.ngroups;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < ns; i += stride) {
      const float s = P.scales[i];
      if (!(s > 0.f) || !isfinite(s)) {
        bad |= BAKRON_DEV_BAD_SCALE;
      } else {
        smax = max(smax, __float_as_uint(s));
      }
    }
  }
  if (P.cscales) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)P.n; i += stride) {
      const float t = P.cscales[i];
      if (!(t > 0.f) || !isfinite(t)) {
        bad |= BAKRON_DEV_BAD_SCALE;
      } else {
        cmax = max(cmax, __float_as_uint(t));
      }
    }
  }
  wmax = warp_max(wmax);
  smax = warp_max(smax);
  cmax = warp_max(cmax);
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&P.hdr->maxw_bits, wmax);
    atomicMax(&P.hdr->maxs_bits, smax);
    atomicMax(&P.hdr->maxc_bits, cmax);
  }
  if (bad) atomicOr(P.status, bad);
}

__global__ void sigma_kernel(InputDesc P) {
  const float maxw = __uint_as_float(P.hdr->maxw_bits);
  // Every entry's scale is at most (max row scale) (max column scale), up to
  // one fp32 rounding, far inside the margin below.
  const float maxs = (P.scales ? __uint_as_float(P.hdr->maxs_bits) : 1.f) *
                     (P.cscales ? __uint_as_float(P.hdr->maxc_bits) : 1.f);
  const float levels = P.bits ? (float)max(-P.lo, P.hi) : 1.f;
  // Every value rounded or accumulated stays within a few alphabet steps of
  // the weights; the offset leaves a wide margin above that.
  P.hdr->sigma = offset_for_bound(16.f * (maxw + maxs * (levels + 2.f)));
}

// Exponent e with |x| < 2^e for every |x| <= mx, kept >= -100 so that every
// scale 2^(7 - e) below is a normal float (smaller values are negligible
// against the offset of the accumulators).
__device__ __forceinline__ int bound_exp(float mx) {
  if (!(mx > 0.f)) return -100;
  int e;
  frexpf(mx, &e);  // mx = f 2^e, f in [0.5, 1)
  return max(e, -100);
}

// 2^k as a float, -126 <= k <= 127.
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((k + 127) << 23); }


// Source digits (the B operand of the chunk products, see the tensor-core
// section below): six bf16 integer digits of a double-float value x on the
// global exponent eD of the solve (2^eD = 2 sigma exceeds every value the
// solve holds, since the offset accumulators rely on that bound):
//   x ~ 2^(eD-7) sum_{b<6} d_b 256^-b,  |d_b| <= 128, error <= 2^(eD-48).
__device__ __forceinline__ void put_digits(__nv_bfloat16* planes, size_t pstride, size_t o, float2 x, float sc) {
  float2 u = make_float2(x.x * sc, x.y * sc);
#pragma unroll
  for (int b = 0; b < kDigD; ++b) {
    const float dg = rintf(u.x);
    planes[b * pstride + o] = __float2bfloat16_rn(dg);
    const float2 rem = two_sum(u.x - dg, u.y);
    u = make_float2(rem.x * 256.f, rem.y * 256.f);
  }
}

// The two chunk planes (Xc, Gc) hold 64-bit two's-complement fixed point in
// units of 2^(eDc - 54), eDc = max(eD, -60) (2^eD = 2 sigma): 2^-53 sigma, 32
// times finer than double-float, with range 2^63 units = 1024 sigma (every
// value the solve holds is below sigma; partial sums of the chunk products
// would have to exceed the final values a thousandfold to wrap).  The chunk
// products add into them with integer reductions in L2 (exact, so the sums
// do not depend on their order), and no fp64 arithmetic is needed anywhere
// (GB300's fp64 rate is 1/64 of its fp32 rate).
__device__ __forceinline__ int fixed_unit_exp(float sigma) { return max(bound_exp(sigma), -60) - 54; }

// Double-float value x * 2^-unit_exp (|x| * 2^-unit_exp < 2^63) rounded to the
// fixed-point grid.
__device__ __forceinline__ long long df_to_fixed(float2 x, float to_units) {
  return __float2ll_rn(x.x * to_units) + __float2ll_rn(x.y * to_units);
}

// Nearest double-float to a fixed-point value v * 2^unit_exp: hi is the
// nearest float to v (an integer when |v| >= 2^24), the remainder v - hi is
// exact in 64 bits and rounded once more for lo.
__device__ __forceinline__ float2 df_from_fixed(long long v, float from_units) {
  const float hi = __ll2float_rn(v);
  const float lo = __ll2float_rn(v - __float2ll_rn(hi));
  return make_float2(hi * from_units, lo * from_units);
}

// Exponent of every (row, chunk) block of a d x d factor: out[r * nch + c]
// bounds row r over columns [c*CK, (c+1)*CK).  One warp per block.
__global__ void __launch_bounds__(256) factor_exp_kernel(const float* F, int d, int nch, signed char* out) {
  const size_t wid = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (size_t)d * nch) return;
  const int r = (int)(wid / nch), c = (int)(wid % nch);
  float mx = 0.f;
  for (int k = lane; k < CK; k += 32) {
    const int gk = c * CK + k;
    if (gk < d) mx = fmaxf(mx, fabsf(F[(size_t)r * d + gk]));
  }
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) out[wid] = (signed char)bound_exp(mx);
}

// Factor digits, computed once per solve (the factors and their block
// exponents are fixed for the whole solve): element (row gr, column gk) of a
// d x d factor, x = F[gr][gk] 2^(7 - e) with e = the block exponent of (gr,
// chunk gk / CK), is split into kDigF integer digits
//     x = d_0 + d_1 / 256 + d_2 / 256^2 + ... (each |d_a| <= 128, exact in bf16)
// by rounding to the nearest integer (ties to even: adding and subtracting
// 1.5 * 2^23, exact for |u| <= 128.5) and scaling the remainder by 256.
// Layout: for chunk c, slab s (32 columns), digit a and tile row t (32 rows)
// one 2 KB block in the tcgen05 core-matrix order of the chunk products'
// shared memory, offset (r/8) 512 + (k/8) 128 + (r%8) 16 + (k%8) 2, blocks
// ordered [c][s][a][t]: the four tiles of a target group are 8 contiguous
// KB, one bulk copy per digit.  Entries outside the matrix are zero.
// One thread per (c, s, t, row, 8 columns).
__global__ void __launch_bounds__(256) factor_digits_kernel(const float* F, int d, int nch, int nt,
                                                            const signed char* fexp, __nv_bfloat16* Fd) {
  const size_t items = (size_t)nch * (CK / kSlab) * nt * T * (kSlab / 8);
  for (size_t it = (size_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (size_t)gridDim.x * blockDim.x) {
    const int k8 = 8 * (int)(it % (kSlab / 8));
    const int r = (int)((it / (kSlab / 8)) % T);
    const int t = (int)((it / (kSlab / 8 * T)) % nt);
    const size_t cs = it / ((size_t)kSlab / 8 * T * nt);  // c * (CK / kSlab) + s
    const int c = (int)(cs / (CK / kSlab)), sl = (int)(cs % (CK / kSlab));
    const int gr = t * T + r, gk = c * CK + sl * kSlab + k8;
    float u[8];
    const float sc = gr < d ? pow2f(7 - fexp[(size_t)gr * nch + c]) : 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) u[e] = (gr < d && gk + e < d) ? F[(size_t)gr * d + gk + e] * sc : 0.f;
    const int off = (r / 8) * 512 + (k8 / 8) * 128 + (r % 8) * 16;
#pragma unroll
    for (int a = 0; a < kDigF; ++a) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float d0 = (u[2 * e] + 0x1.8p23f) - 0x1.8p23f;
        const float d1 = (u[2 * e + 1] + 0x1.8p23f) - 0x1.8p23f;
        w[e] = __byte_perm(__float_as_uint(d0), __float_as_uint(d1), 0x7632);  // bf16 patterns, low half: smaller k
        u[2 * e] = (u[2 * e] - d0) * 256.f;  // exact: |u - d| <= 1/2, u has <= 24 significant bits
        u[2 * e + 1] = (u[2 * e + 1] - d1) * 256.f;
      }
      unsigned char* blk = reinterpret_cast<unsigned char*>(Fd) + ((cs * kDigF + a) * nt + t) * 2048;
      *reinterpret_cast<uint4*>(blk + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace
}  // namespace bakron
