// prep.cu -- the normalized inverse Cholesky factor L-hat on sm_103a.
//
// "BaKron: Efficient Quantization with Kronecker-Factored Hessians", Sec. 3.2
// Algorithm 1 prologue: L = Cholesky(H^-1), columns divided by their
// diagonal entries.  Sec. 3.1 defines RevCholesky(H) = R (lower, R^T R = H).
//
// Route taken (derived from those definitions, no inverse of H formed):
// Cholesky(H^-1) = R^-1 because H^-1 = R^-1 R^-T with R^-1 lower, so
// L-hat = R^-1 diag(R).  With J the reversal permutation, factor
// H' = J H J = C~ D C~^T (LDL^T, C~ unit lower); then R = J (C~ D^1/2)^T J and
// L-hat = J C~^-T J, i.e.  L-hat[i][j] = (C~^-1)[d-1-j][d-1-i].
// Steps: (1) blocked right-looking LDL^T of H' in 32-column panels
// (diagonal block, panel solve, trailing update), (2) blocked inverse of the
// unit lower C~ (diagonal blocks, then block sub-diagonals s = 1, 2, ...),
// (3) the index flip and one rounding to fp32.
//
// All arithmetic is double-float (df.cuh).  A pivot d_j <= 0 writes
// 1 + (index of that pivot in H) to *info (first failure only) and the
// computation carries on with garbage; nothing traps.
#include <algorithm>
#include <cmath>

#include "df.cuh"
#include "internal.h"

namespace bakron {
namespace {

constexpr int NB = 32;  // panel width

struct FParams {
  const float* H;
  float* Lhat;
  float2* M;  // d x d: LDL^T of the flipped matrix (strict lower: C~, diagonal: D)
  float2* X;  // d x d: C~^-1
  float2* P;  // d x NB: panel of C~ D (current panel)
  int32_t* info;
  int d, nb;  // order, number of panels
};

__global__ void init_kernel(FParams F) {
  const size_t total = (size_t)F.d * F.d;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(e / F.d), j = (int)(e % F.d);
    float2 v = make_float2(0.f, 0.f);
    if (i >= j) {  // H'[i][j] = H[d-1-i][d-1-j] = H[d-1-j][d-1-i] (lower triangle of H)
      v.x = F.H[(size_t)(F.d - 1 - j) * F.d + (F.d - 1 - i)];
    }
    F.M[e] = v;
    F.X[e] = make_float2(0.f, 0.f);
  }
}

// LDL^T of the diagonal block kb in place (one CTA of NB x NB threads).
__global__ void __launch_bounds__(NB* NB) diag_factor_kernel(FParams F, int kb) {
  __shared__ float2 blk[NB][NB + 1];
  __shared__ float2 col[NB];   // l_ij = a_ij / d_j for the current j
  __shared__ float2 wcol[NB];  // a_ij (= l_ij d_j) for the current j
  const int i = threadIdx.y, l = threadIdx.x;
  const int base = kb * NB;
  const int bs = min(NB, F.d - base);
  if (i < bs && l < bs) blk[i][l] = F.M[(size_t)(base + i) * F.d + base + l];
  __syncthreads();
  for (int j = 0; j < bs; ++j) {
    const float2 dj = blk[j][j];
    if (i == 0 && l == 0 && !(dj.x > 0.f)) atomicCAS(F.info, 0, 1 + (F.d - 1 - (base + j)));
    if (l == j && i > j && i < bs) {
      wcol[i] = blk[i][j];
      col[i] = df_div(blk[i][j], dj);
    }
    __syncthreads();
    if (i > j && i < bs && l > j && l <= i) blk[i][l] = df_sub(blk[i][l], df_mul(col[i], wcol[l]));
    __syncthreads();
    if (l == j && i > j && i < bs) blk[i][j] = col[i];
    __syncthreads();
  }
  if (i < bs && l < bs && l <= i) F.M[(size_t)(base + i) * F.d + base + l] = blk[i][l];
}

// Panel below the diagonal block: row r gets x = a_r C~_kk^-T (forward
// substitution), stores x in P (= C~_rk D_k) and x D_k^-1 in M (= C~_rk).
__global__ void __launch_bounds__(128) panel_kernel(FParams F, int kb) {
  __shared__ float2 Ckk[NB][NB + 1];
  const int base = kb * NB;
  const int bs = min(NB, F.d - base);
  for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
    const int a = e / NB, b = e % NB;
    Ckk[a][b] = (a < bs && b < bs) ? F.M[(size_t)(base + a) * F.d + base + b] : make_float2(0.f, 0.f);
  }
  __syncthreads();
  const int r = base + bs + blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= F.d) return;
  float2 x[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) x[j] = (j < bs) ? F.M[(size_t)r * F.d + base + j] : make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < NB; ++j) {
#pragma unroll
    for (int t = 0; t < j; ++t) x[j] = df_sub(x[j], df_mul(x[t], Ckk[j][t]));
  }
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    if (j < bs) {
      F.P[(size_t)r * NB + j] = x[j];
      F.M[(size_t)r * F.d + base + j] = df_div(x[j], Ckk[j][j]);
    }
  }
}

__device__ __forceinline__ void tri_decode(int t, int& a, int& b) {
  // t -> (a, b) with 0 <= b <= a, t = a(a+1)/2 + b
  int aa = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
  while ((aa + 1) * (aa + 2) / 2 <= t) ++aa;
  while (aa * (aa + 1) / 2 > t) --aa;
  a = aa;
  b = t - aa * (aa + 1) / 2;
}

__device__ __forceinline__ unsigned warp_max_u(unsigned v) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide max of two non-negative values (256 threads); result to all.
__device__ __forceinline__ float2 block_max2(float a, float b, unsigned* red) {
  unsigned ua = warp_max_u(__float_as_uint(a)), ub = warp_max_u(__float_as_uint(b));
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = ua;
    red[8 + (threadIdx.x >> 5)] = ub;
  }
  __syncthreads();
  unsigned ma = 0, mb = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    ma = max(ma, red[w]);
    mb = max(mb, red[8 + w]);
  }
  __syncthreads();
  return make_float2(__uint_as_float(ma), __uint_as_float(mb));
}

// Trailing update M[ib][jb] -= P[ib] C~[jb][kb]^T for kb < jb <= ib.
__global__ void __launch_bounds__(256) trailing_kernel(FParams F, int kb) {
  __shared__ float2 sA[NB][NB + 1];  // P rows of block ib
  __shared__ float2 sB[NB][NB + 1];  // C~ rows of block jb (panel kb)
  __shared__ unsigned red[16];
  int a, b;
  tri_decode(blockIdx.x, a, b);
  const int ib = kb + 1 + a, jb = kb + 1 + b;
  const int base = kb * NB;
  const int bs = min(NB, F.d - base);
  float amax = 0.f, bmax = 0.f;
  for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
    const int u = e / NB, v = e % NB;
    const int ra = ib * NB + u, rb = jb * NB + u;
    float2 va = (ra < F.d && v < bs) ? F.P[(size_t)ra * NB + v] : make_float2(0.f, 0.f);
    float2 vb = (rb < F.d && v < bs) ? F.M[(size_t)rb * F.d + base + v] : make_float2(0.f, 0.f);
    sA[u][v] = va;
    sB[u][v] = vb;
    amax = fmaxf(amax, fabsf(va.x));
    bmax = fmaxf(bmax, fabsf(vb.x));
  }
  const float2 mx = block_max2(amax, bmax, red);
  const float sigma = offset_for_bound(2.f * NB * mx.x * mx.y);
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  OffsetAcc acc[4];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) acc[rr].init(sigma);
  for (int t = 0; t < NB; ++t) {
    const float2 bv = sB[tx][t];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) acc[rr].mac(sA[ty + 8 * rr][t], bv);
  }
  const int gc = jb * NB + tx;
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int gr = ib * NB + ty + 8 * rr;
    if (gr < F.d && gc < F.d && gc <= gr) {
      const size_t o = (size_t)gr * F.d + gc;
      F.M[o] = df_sub(F.M[o], acc[rr].value(sigma));
    }
  }
}

// X_kk = C~_kk^-1 for every diagonal block (unit lower), one CTA per block,
// one thread per column.
__global__ void __launch_bounds__(NB) inv_diag_kernel(FParams F) {
  __shared__ float2 C[NB][NB + 1];
  const int kb = blockIdx.x;
  const int base = kb * NB;
  const int bs = min(NB, F.d - base);
  for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
    const int a = e / NB, b = e % NB;
    C[a][b] = (a < bs && b < bs) ? F.M[(size_t)(base + a) * F.d + base + b] : make_float2(0.f, 0.f);
  }
  __syncthreads();
  const int c = threadIdx.x;
  if (c >= bs) return;
  float2 x[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) x[i] = make_float2(i == c ? 1.f : 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    if (i > c) {
      float2 s = make_float2(0.f, 0.f);
#pragma unroll
      for (int t = 0; t < i; ++t)
        if (t >= c) s = df_add(s, df_mul(C[i][t], x[t]));
      x[i] = df_neg(s);
    }
  }
#pragma unroll
  for (int i = 0; i < NB; ++i)
    if (i < bs) F.X[(size_t)(base + i) * F.d + base + c] = x[i];
}

// Block sub-diagonal s of X = C~^-1: for jb, ib = jb + s,
//   X[ib][jb] = -X[ib][ib] * sum_{kb=jb}^{ib-1} C~[ib][kb] X[kb][jb].
__global__ void __launch_bounds__(256) inv_offdiag_kernel(FParams F, int s) {
  __shared__ float2 sA[NB][NB + 1];
  __shared__ float2 sB[NB][NB + 1];
  __shared__ float2 sS[NB][NB + 1];
  __shared__ unsigned red[16];
  const int jb = blockIdx.x, ib = jb + s;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  float2 sum[4];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) sum[rr] = make_float2(0.f, 0.f);
  for (int kb = jb; kb < ib; ++kb) {
    float amax = 0.f, bmax = 0.f;
    for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
      const int u = e / NB, v = e % NB;
      const int ra = ib * NB + u, ca = kb * NB + v;  // C~[ib][kb]
      const int rb = kb * NB + u, cb = jb * NB + v;  // X[kb][jb]
      float2 va = (ra < F.d && ca < F.d && ca < ra) ? F.M[(size_t)ra * F.d + ca] : make_float2(0.f, 0.f);
      float2 vb = (rb < F.d && cb < F.d) ? F.X[(size_t)rb * F.d + cb] : make_float2(0.f, 0.f);
      sA[u][v] = va;
      sB[u][v] = vb;
      amax = fmaxf(amax, fabsf(va.x));
      bmax = fmaxf(bmax, fabsf(vb.x));
    }
    const float2 mx = block_max2(amax, bmax, red);
    const float sigma = offset_for_bound(2.f * NB * mx.x * mx.y);
    OffsetAcc acc[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) acc[rr].init(sigma);
    for (int t = 0; t < NB; ++t) {
      const float2 bv = sB[t][tx];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) acc[rr].mac(sA[ty + 8 * rr][t], bv);
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) sum[rr] = df_add(sum[rr], acc[rr].value(sigma));
    __syncthreads();
  }
  // X[ib][jb] = -X[ib][ib] * S
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) sS[ty + 8 * rr][tx] = sum[rr];
  for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
    const int u = e / NB, v = e % NB;
    const int ra = ib * NB + u, ca = ib * NB + v;
    sA[u][v] = (ra < F.d && ca < F.d) ? F.X[(size_t)ra * F.d + ca] : make_float2(0.f, 0.f);
  }
  __syncthreads();
  float2 out[4];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) out[rr] = make_float2(0.f, 0.f);
  for (int t = 0; t < NB; ++t) {
    const float2 bv = sS[t][tx];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) out[rr] = df_add(out[rr], df_mul(sA[ty + 8 * rr][t], bv));
  }
  const int gc = jb * NB + tx;
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int gr = ib * NB + ty + 8 * rr;
    if (gr < F.d && gc < F.d) F.X[(size_t)gr * F.d + gc] = df_neg(out[rr]);
  }
}

// L-hat[i][j] = X[d-1-j][d-1-i] for i > j, 1 on the diagonal, 0 above.
__global__ void finalize_kernel(FParams F) {
  const size_t total = (size_t)F.d * F.d;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(e / F.d), j = (int)(e % F.d);
    float v = 0.f;
    if (i == j) {
      v = 1.f;
    } else if (i > j) {
      const float2 x = F.X[(size_t)(F.d - 1 - j) * F.d + (F.d - 1 - i)];
      v = x.x + x.y;  // one rounding of the double-float value
    }
    F.Lhat[e] = v;
  }
}

}  // namespace

size_t factor_workspace_bytes(int64_t d) {
  const size_t sq = align_up((size_t)d * (size_t)d * sizeof(float2));
  const size_t pan = align_up((size_t)d * NB * sizeof(float2));
  return 2 * sq + pan;
}

cudaError_t factor_launch(const float* H, int d, float* Lhat, void* ws, int32_t* info, cudaStream_t stream) {
  const size_t sq = align_up((size_t)d * (size_t)d * sizeof(float2));
  char* base = static_cast<char*>(ws);
  FParams F;
  F.H = H;
  F.Lhat = Lhat;
  F.M = reinterpret_cast<float2*>(base);
  F.X = reinterpret_cast<float2*>(base + sq);
  F.P = reinterpret_cast<float2*>(base + 2 * sq);
  F.info = info;
  F.d = d;
  F.nb = (d + NB - 1) / NB;
  cudaError_t err = cudaMemsetAsync(info, 0, sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  const size_t total = (size_t)d * d;
  const int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 8);
  init_kernel<<<blocks, 256, 0, stream>>>(F);
  for (int kb = 0; kb < F.nb; ++kb) {
    diag_factor_kernel<<<1, dim3(NB, NB), 0, stream>>>(F, kb);
    const int rows = d - std::min(d, (kb + 1) * NB);
    if (rows > 0) {
      panel_kernel<<<(rows + 127) / 128, 128, 0, stream>>>(F, kb);
      const int nr = F.nb - kb - 1;
      trailing_kernel<<<nr * (nr + 1) / 2, 256, 0, stream>>>(F, kb);
    }
  }
  inv_diag_kernel<<<F.nb, NB, 0, stream>>>(F);
  for (int s = 1; s < F.nb; ++s) inv_offdiag_kernel<<<F.nb - s, 256, 0, stream>>>(F, s);
  finalize_kernel<<<blocks, 256, 0, stream>>>(F);
  return cudaGetLastError();
}

}  // namespace bakron
