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
// (diagonal block and its inverse, panel as a product with that inverse,
// trailing update), (2) inverse of the unit lower C~ (block doubling from
// the diagonal blocks' inverses: 32 -> 64 -> ... rows),
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

// LDL^T of the diagonal block kb in place (one CTA of NB x NB threads), then
// the inverse W = C~_kk^-1 of its unit lower factor into X's diagonal block
// (the panel below uses it, and it is the leaf of the inverse of C~).
__global__ void __launch_bounds__(NB* NB) diag_factor_kernel(FParams F, int kb) {
  __shared__ float2 blk[NB][NB + 1];
  __shared__ float2 Ws[NB][NB + 1];
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
  // Column c of W by forward substitution (one thread per column, each
  // touching only its own column of Ws): W[c][c] = 1,
  // W[r][c] = -sum_{t = c}^{r-1} C~[r][t] W[t][c].
  if (i == 0 && l < bs) {
    const int c = l;
    for (int r = 0; r < NB; ++r) Ws[r][c] = make_float2(r == c ? 1.f : 0.f, 0.f);
    for (int r = c + 1; r < bs; ++r) {
      float2 acc = make_float2(0.f, 0.f);
      for (int t = c; t < r; ++t) acc = df_add(acc, df_mul(blk[r][t], Ws[t][c]));
      Ws[r][c] = df_neg(acc);
    }
  }
  __syncthreads();
  if (i < bs && l < bs) F.X[(size_t)(base + i) * F.d + base + l] = Ws[i][l];
}

// Panel below the diagonal block: row r's entries a (after the trailing
// updates of the earlier panels) satisfy C~_kk x = a with x = C~_rk D_k, so
// x = W a with W = C~_kk^-1 (written by diag_factor_kernel):
//     x_j = sum_{t <= j} W[j][t] a_t,
// one double-float dot product per (row, j), all in parallel.  Stores x in
// P (= C~_rk D_k) and x D_k^-1 in M (= C~_rk).  8 rows per CTA.
constexpr int kPanelRows = 8;
__global__ void __launch_bounds__(kPanelRows * NB) panel_kernel(FParams F, int kb) {
  __shared__ float2 Wk[NB][NB + 1];
  __shared__ float2 arow[kPanelRows][NB + 1];
  __shared__ float2 dk[NB];
  const int base = kb * NB;
  const int bs = min(NB, F.d - base);
  for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
    const int a = e / NB, b = e % NB;
    Wk[a][b] = (a < bs && b < bs) ? F.X[(size_t)(base + a) * F.d + base + b] : make_float2(0.f, 0.f);
  }
  if (threadIdx.x < NB)
    dk[threadIdx.x] = threadIdx.x < bs ? F.M[(size_t)(base + threadIdx.x) * F.d + base + threadIdx.x]
                                       : make_float2(1.f, 0.f);
  const int rr = threadIdx.x / NB, j = threadIdx.x % NB;
  const int r = base + bs + blockIdx.x * kPanelRows + rr;
  arow[rr][j] = (r < F.d && j < bs) ? F.M[(size_t)r * F.d + base + j] : make_float2(0.f, 0.f);
  __syncthreads();
  if (r >= F.d || j >= bs) return;
  float2 x = make_float2(0.f, 0.f);
  for (int t = 0; t <= j; ++t) x = df_add(x, df_mul(Wk[j][t], arow[rr][t]));
  F.P[(size_t)r * NB + j] = x;
  F.M[(size_t)r * F.d + base + j] = df_div(x, dk[j]);
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

// Trailing update M[ib][jb] -= P[ib] C~[jb][kb]^T for kb < jb <= ib, in
// 64 x 64 tiles (2 x 2 blocks of NB): CTA (A, Bs) of the lower tile
// triangle updates block rows kb+1+2A, kb+2+2A and block columns
// kb+1+2Bs, kb+2+2Bs (entries with column <= row only).  Each thread holds
// 16 outputs (rows ty + 8 rr, columns tx + 32 cc), so that every operand
// value loaded from shared memory feeds 8 or 2 multiply-adds.
constexpr int kTrail = 2 * NB;
__global__ void __launch_bounds__(256) trailing_kernel(FParams F, int kb) {
  __shared__ float2 sA[kTrail][NB + 1];  // P rows of the tile's two block rows
  __shared__ float2 sB[kTrail][NB + 1];  // C~ rows of its two block columns (panel kb)
  __shared__ unsigned red[16];
  int a, b;
  tri_decode(blockIdx.x, a, b);
  const int r0 = (kb + 1 + 2 * a) * NB, c0 = (kb + 1 + 2 * b) * NB;  // first row, first column
  const int base = kb * NB;
  const int bs = min(NB, F.d - base);
  float amax = 0.f, bmax = 0.f;
  for (int e = threadIdx.x; e < kTrail * NB; e += blockDim.x) {
    const int u = e / NB, v = e % NB;
    const int ra = r0 + u, rb = c0 + u;
    const float2 va = (ra < F.d && v < bs) ? F.P[(size_t)ra * NB + v] : make_float2(0.f, 0.f);
    const float2 vb = (rb < F.d && v < bs) ? F.M[(size_t)rb * F.d + base + v] : make_float2(0.f, 0.f);
    sA[u][v] = va;
    sB[u][v] = vb;
    amax = fmaxf(amax, fabsf(va.x));
    bmax = fmaxf(bmax, fabsf(vb.x));
  }
  const float2 mx = block_max2(amax, bmax, red);
  const float sigma = offset_for_bound(2.f * NB * mx.x * mx.y);
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  OffsetAcc acc[8][2];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    acc[rr][0].init(sigma);
    acc[rr][1].init(sigma);
  }
#pragma unroll 4
  for (int t = 0; t < NB; ++t) {
    const float2 b0 = sB[tx][t], b1 = sB[tx + NB][t];
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const float2 av = sA[ty + 8 * rr][t];
      acc[rr][0].mac(av, b0);
      acc[rr][1].mac(av, b1);
    }
  }
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int gr = r0 + ty + 8 * rr;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int gc = c0 + tx + NB * cc;
      if (gr < F.d && gc < F.d && gc <= gr) {
        const size_t o = (size_t)gr * F.d + gc;
        F.M[o] = df_sub(F.M[o], acc[rr][cc].value(sigma));
      }
    }
  }
}

// X = C~^-1 by block doubling.  For two consecutive diagonal blocks of b
// rows whose inverses X11, X22 are known (lower triangular),
//     X21 = -X22 C~21 X11,
// so the inverses of blocks of 2b follow from those of b in two products.
// Level b (32, 64, ...) runs every pair of blocks at once, as two launches:
//   stage 0:  T = C~21 X11     (stored transposed in the unused upper
//             triangle of X, at rows r1 .., columns r2 .., i.e. X[r1 + j][r2 + i])
//   stage 1:  X21 = -X22 T.
// The triangular operand is read with its upper part masked (that part of X
// holds the scratch T of inner levels), and its zero half skipped: stage 0
// sums over k >= the tile's first column, stage 1 over k <= its last row.
// blockIdx.y: pair t (r1 = 2 t b, r2 = r1 + b); blockIdx.x: 32 x 32 output
// tile (ti, tj), ti over the rows of the second block, tj over the columns
// of the first.  Each 32-deep chunk is summed on an offset of its own and
// folded into a double-float total.
__global__ void __launch_bounds__(256) inv_level_kernel(FParams F, int b, int stage) {
  __shared__ float2 sA[NB][NB + 1];
  __shared__ float2 sB[NB][NB + 1];
  __shared__ unsigned red[16];
  const int r1 = 2 * blockIdx.y * b, r2 = r1 + b;
  if (r2 >= F.d) return;
  const int n1 = b, n2 = min(b, F.d - r2);  // r2 < d, so the first block is whole
  const int per = b / NB;
  const int ti = blockIdx.x / per, tj = blockIdx.x % per;
  if (ti * NB >= n2) return;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  float2 sum[4];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) sum[rr] = make_float2(0.f, 0.f);
  const int kc0 = stage == 0 ? tj : 0;
  const int kc1 = stage == 0 ? (n1 + NB - 1) / NB : ti + 1;
  for (int kc = kc0; kc < kc1; ++kc) {
    float amax = 0.f, bmax = 0.f;
    for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
      const int u = e / NB, v = e % NB;
      const int ia = ti * NB + u, ka = kc * NB + v;  // A[ia][ka]
      const int kb = kc * NB + u, jb = tj * NB + v;  // B[kb][jb]
      float2 va = make_float2(0.f, 0.f), vb = make_float2(0.f, 0.f);
      if (stage == 0) {
        if (ia < n2 && ka < n1) va = F.M[(size_t)(r2 + ia) * F.d + (r1 + ka)];               // C~21
        if (kb < n1 && kb >= jb) vb = F.X[(size_t)(r1 + kb) * F.d + (r1 + jb)];              // X11
      } else {
        if (ia < n2 && ka <= ia) va = F.X[(size_t)(r2 + ia) * F.d + (r2 + ka)];              // X22
        if (kb < n2 && jb < n1) vb = F.X[(size_t)(r1 + jb) * F.d + (r2 + kb)];               // T (transposed)
      }
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
  const int j = tj * NB + tx;
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int i = ti * NB + ty + 8 * rr;
    if (i < n2 && j < n1) {
      if (stage == 0) F.X[(size_t)(r1 + j) * F.d + (r2 + i)] = sum[rr];
      else F.X[(size_t)(r2 + i) * F.d + (r1 + j)] = df_neg(sum[rr]);
    }
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
      panel_kernel<<<(rows + kPanelRows - 1) / kPanelRows, kPanelRows * NB, 0, stream>>>(F, kb);
      const int nr = F.nb - kb - 1;         // trailing block rows
      const int nt = (nr + 1) / 2;          // 64-row tiles
      trailing_kernel<<<nt * (nt + 1) / 2, 256, 0, stream>>>(F, kb);
    }
  }
  for (int b = NB; b < F.d; b *= 2) {
    const dim3 grid((unsigned)((b / NB) * (b / NB)), (unsigned)((F.d + 2 * b - 1) / (2 * b)));
    inv_level_kernel<<<grid, 256, 0, stream>>>(F, b, 0);
    inv_level_kernel<<<grid, 256, 0, stream>>>(F, b, 1);
  }
  finalize_kernel<<<blocks, 256, 0, stream>>>(F);
  return cudaGetLastError();
}

}  // namespace bakron
