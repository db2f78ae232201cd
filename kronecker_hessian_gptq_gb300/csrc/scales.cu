// scales.cu -- per-row scale choice and packed codes (base-quantizer variants
// of "BaKron: Efficient Quantization with Kronecker-Factored Hessians",
// App. D: scales per row = max |W_ij| / l, optionally shrunk by up to 2x by
// an MSE search; Sec. 3.1: alphabets of b+1 bits).
//
// Scale search, as the C ABI defines it (include/bakron.h):
//   s0 = fp32(max_j |W_ij| / hi)  (correctly rounded fp32 division);
//   candidates s_g = fp32(s0 f_g), f_g = fp32(1 - g / (2 (G - 1))), g < G;
//   error(s) = sum_j (W_ij - s v_ij)^2, v_ij = clamp(rne(fp32(W_ij) / s), lo, hi);
//   the chosen scale is the candidate of least error, the smallest g among
//   equals; G = 1: s0; a row of zeros: 1.
// Each error term is formed exactly (two_prod and two_sum) on the row scaled
// by a power of two; the sum is double-float.
#include <algorithm>

#include "bakron.h"
#include "df.cuh"
#include "internal.h"

namespace bakron {
namespace {

constexpr int kScaleThreads = 256;
constexpr int kMaxGrid = BAKRON_MAX_SCALE_GRID;
constexpr size_t kMaxStagedBytes = 192 * 1024;

struct ShrinkTable {
  float f[kMaxGrid];
};

// Round half to even of the fp32 quotient x / s (the decision of the solve:
// x * (1/s) is within 2 ulp of the correctly rounded quotient, which is used
// whenever the product is near a tie or large).
// A reciprocal that overflows (s below 2^-128) gives an infinite or NaN
// product, which also takes the division.
__device__ __forceinline__ float rne_quotient(float x, float s, float rcp) {
  float y = x * rcp;
  if (!(fabsf(y) <= 256.f) || fabsf(y - floorf(y) - 0.5f) < 1e-3f) y = __fdiv_rn(x, s);
  return rintf(y);
}

// x 2^k for -160 <= k <= 160, in two steps of normal powers of two (exact
// unless the result is subnormal).
__device__ __forceinline__ float scale_pow2(float x, int k) {
  const int k1 = k / 2, k2 = k - k1;
  return x * __int_as_float((k1 + 127) << 23) * __int_as_float((k2 + 127) << 23);
}

__device__ __forceinline__ float2 df_block_sum(float2 v, float2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o; o >>= 1) {
    const float2 w = make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
    v = df_add(v, w);
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  if (threadIdx.x == 0)
    for (int i = 0; i < kScaleThreads / 32; ++i) t = df_add(t, red[i]);
  __syncthreads();
  return t;  // valid in thread 0
}

// One CTA per run of `group` columns of a row (blockIdx.x = row * runs +
// run); the run is staged in dynamic shared memory.
__global__ void __launch_bounds__(kScaleThreads) row_scales_kernel(const float* W, int n, int group, int runs, int lo,
                                                                    int hi, int grid, bool staged, ShrinkTable tab,
                                                                    float* scales) {
  extern __shared__ float srow[];
  __shared__ float2 red[kScaleThreads / 32];
  __shared__ float smax[kScaleThreads / 32];
  const int row = blockIdx.x / runs, run = blockIdx.x % runs;
  const float* w = W + (size_t)row * n + (size_t)run * group;
  const int len = min(group, n - run * group);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float mx = 0.f;
  for (int j = threadIdx.x; j < len; j += kScaleThreads) {
    const float x = w[j];
    if (staged) srow[j] = x;
    mx = fmaxf(mx, fabsf(x));
  }
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) smax[warp] = mx;
  __syncthreads();
  float amax = 0.f;
  for (int i = 0; i < kScaleThreads / 32; ++i) amax = fmaxf(amax, smax[i]);
  if (!(amax > 0.f)) {
    if (threadIdx.x == 0) scales[blockIdx.x] = 1.f;
    return;
  }
  const float s0 = __fdiv_rn(amax, (float)hi);
  if (grid <= 1) {
    if (threadIdx.x == 0) scales[blockIdx.x] = s0;
    return;
  }
  const float* src = staged ? srow : w;  // rows too long for shared memory are re-read through L1/L2
  const float flo = (float)lo, fhi = (float)hi;
  // The errors are formed on the row scaled by 2^k, max |x| 2^k in [1/2, 1):
  // every candidate's errors scale alike, so the argmin is unchanged, and no
  // product underflows or overflows (entries below 2^-126 of the row's
  // maximum may lose bits, far below the sum's resolution).
  int ex;
  frexpf(amax, &ex);
  const int k = -ex;
  int best = 0;
  float2 best_err = make_float2(0.f, 0.f);
  for (int g = 0; g < grid; ++g) {
    const float s = __fmul_rn(s0, tab.f[g]);
    const float rcp = __frcp_rn(s);
    const float sk = scale_pow2(s, k);
    float2 acc = make_float2(0.f, 0.f);
    for (int j = threadIdx.x; j < len; j += kScaleThreads) {
      const float x = src[j];
      const float v = fminf(fmaxf(rne_quotient(x, s, rcp), flo), fhi);  // the decision on the unscaled row
      const float2 sv = two_prod(sk, v);               // s v 2^k exactly
      const float2 h = two_sum(scale_pow2(x, k), -sv.x);
      const float2 e = two_sum(h.x, h.y - sv.y);       // (x - s v) 2^k to double-float
      const float2 e2 = two_prod(e.x, e.x);
      acc = df_add(acc, make_float2(e2.x, e2.y + 2.f * e.x * e.y));
    }
    const float2 tot = df_block_sum(acc, red);
    // Strictly less (the double-float sums are normalized, so comparing the
    // high parts first is exact): the first minimum is kept.
    if (threadIdx.x == 0 && (g == 0 || tot.x < best_err.x || (tot.x == best_err.x && tot.y < best_err.y))) {
      best = g;
      best_err = tot;
    }
  }
  if (threadIdx.x == 0) scales[blockIdx.x] = __fmul_rn(s0, tab.f[best]);
}

// One thread per output byte: codes j = byte * (8 / bits) + t.
__global__ void pack_codes_kernel(const int32_t* V, int m, int n, int bits, int rowbytes, uint8_t* out) {
  const size_t total = (size_t)m * rowbytes;
  const int per = 8 / bits;
  const unsigned mask = (1u << bits) - 1u;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(idx / rowbytes), byte = (int)(idx % rowbytes);
    unsigned b = 0;
    for (int t = 0; t < per; ++t) {
      const int j = byte * per + t;
      if (j < n) b |= ((unsigned)V[(size_t)i * n + j] & mask) << (t * bits);
    }
    out[idx] = (uint8_t)b;
  }
}

}  // namespace

cudaError_t row_scales_launch(const float* W, int m, int n, int group, Alphabet al, int grid, float* scales,
                              cudaStream_t stream) {
  if (group <= 0 || group > n) group = n;
  const int runs = (n + group - 1) / group;
  ShrinkTable tab;
  for (int g = 0; g < kMaxGrid; ++g)
    tab.f[g] = g < grid ? (grid > 1 ? (float)(1.0 - (double)g / (2.0 * (grid - 1))) : 1.f) : 0.f;
  const bool staged = (size_t)group * sizeof(float) <= kMaxStagedBytes;
  const size_t smem = staged ? (size_t)group * sizeof(float) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(row_scales_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  row_scales_kernel<<<(unsigned)((size_t)m * runs), kScaleThreads, smem, stream>>>(W, n, group, runs, al.lo, al.hi,
                                                                                  grid, staged, tab, scales);
  return cudaGetLastError();
}

cudaError_t pack_codes_launch(const int32_t* V, int m, int n, int bits, uint8_t* out, cudaStream_t stream) {
  const int rowbytes = (n * bits + 7) / 8;
  const size_t total = (size_t)m * rowbytes;
  const int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 16);
  pack_codes_kernel<<<blocks, 256, 0, stream>>>(V, m, n, bits, rowbytes, out);
  return cudaGetLastError();
}

}  // namespace bakron
