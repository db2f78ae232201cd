// quantize.cu -- the BaKron core on sm_103a: a tile wavefront with delayed,
// batched propagation on three streams; all solver state in double-float.
//
// "BaKron: Efficient Quantization with Kronecker-Factored Hessians":
//   App. B eq. (2): W~ = W0 + L_B (sum of earlier errors) L_A^T on every
//     anti-diagonal, v = round(W~), E = v - W~.
//   Sec. 3.3: entry (i, j) only affects entries (p, q) with i <= p, j <= q,
//     so the entries of one anti-diagonal are rounded in parallel.
//   Sec. 3.4 / 3.5 and App. B eq. (1): the updates from a finished set of
//     entries to a later set are one dense product L_B E L_A^T restricted to
//     the later set; they can be delayed and batched, which is what turns
//     the quartic work of Alg. 3 into the cubic work of Alg. 5 and 6.
//
// Decomposition.  With G = E L_A^T (row transform: G[i, q] depends only on
// row i's errors in columns <= q) and L_B unit lower triangular,
//     W~[p, q] = W0[p, q] + sum_{i < p} L_B[p, i] G[i, q] + (G[p, q] - E[p, q]).
// The matrix is cut into T x T tiles; tile (I, J) depends on the tiles
// (I', J') with I' <= I, J' <= J, so the tiles of one tile anti-diagonal
// K = I + J are independent.  Tile (I, J) receives
//   column part  sum_{I' < I} L_B[I, I'] G[I', J]            (same tile column)
//   row part     L_B[I, I] sum_{J' < J} E[I, J'] L_A[J, J']^T  (same tile row)
// split by the distance d between source and target tile:
//   d = 1   pulled by the tile's own solve (right after its neighbours finish);
//   d >= 2  pushed by "mid" products from one source tile (K = T), or by
//           "chunk" products that batch the B source tiles of one chunk
//           (K = B*T; tile rows/columns are grouped in chunks of B).  A source
//           in chunk c pushes itself to the targets before chunk c+2; the
//           chunk product covers the targets from chunk c+2 on, so it has
//           B+1 tile anti-diagonals of slack and runs off the critical path.
// Streams: the caller's stream runs the tile solves, a second one the mid
// pushes, a third one the chunk products; events order
//   solve(K) -> mid(K) -> solve(K+2)   and   solve(K) -> chunk(K) -> solve(K+B+1).
// Mid and chunk pushes accumulate into separate planes, so the two streams
// never write the same element.
//
// Inside a tile each thread owns two entries of one tile row, placed so that
// the entries of one anti-diagonal sit in one warp.  At in-tile step k that
// warp rounds anti-diagonal k; after one barrier every
// later entry folds in the one new term of its row sum (E[p, k-p] L_A[q, k-p])
// and of its column sum (L_B[p, k-q] Gin[k-q, q], Gin = in-tile row sum + error).
//
// Precision: every accumulation is double-float (df.cuh); the rounding
// decision is the fp32 quotient fp32(W~) / s_i rounded half to even, with the
// correctly rounded division used whenever the quotient is near a tie.
#include <algorithm>
#include <mutex>
#include <vector>

#include "bakron.h"
#include "df.cuh"
#include "internal.h"

namespace bakron {
namespace {

constexpr int T = 32;  // tile edge
constexpr int B = 4;   // tiles per chunk
constexpr int U = 4;   // target tiles per push CTA

struct Header {
  unsigned maxw_bits;  // max |W| as ordered uint bits
  unsigned maxs_bits;  // max scale
  float sigma;         // offset of the offset accumulators
  int pad[61];
};
static_assert(sizeof(Header) == 256, "header is one alignment unit");

constexpr int kPlanes = 6;  // Xm, Xc, Gm, Gc, G, E

struct QParams {
  const float* W;
  const float* LA;
  const float* LB;
  const float* scales;
  int32_t* V;
  float* Wq;
  float2* Xm;  // column pushes from single tiles (mid)
  float2* Xc;  // column pushes from chunks
  float2* Gm;  // row pushes from single tiles (mid)
  float2* Gc;  // row pushes from chunks
  float2* G;   // full row transform of each solved entry
  float2* E;   // errors at rounding time
  Header* hdr;
  int32_t* status;
  int m, n, Mt, Nt, bits, lo, hi;
};

__device__ __forceinline__ unsigned warp_max(unsigned v) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Checks the inputs and finds max |W| and max scale.
__global__ void prepass_kernel(QParams P) {
  const size_t total = (size_t)P.m * P.n;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  unsigned wmax = 0, smax = 0;
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
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)P.m; i += stride) {
      const float s = P.scales[i];
      if (!(s > 0.f) || !isfinite(s)) {
        bad |= BAKRON_DEV_BAD_SCALE;
      } else {
        smax = max(smax, __float_as_uint(s));
      }
    }
  }
  wmax = warp_max(wmax);
  smax = warp_max(smax);
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&P.hdr->maxw_bits, wmax);
    atomicMax(&P.hdr->maxs_bits, smax);
  }
  if (bad) atomicOr(P.status, bad);
}

__global__ void sigma_kernel(QParams P) {
  const float maxw = __uint_as_float(P.hdr->maxw_bits);
  const float maxs = P.scales ? __uint_as_float(P.hdr->maxs_bits) : 1.f;
  const float levels = P.bits ? (float)(1 << (P.bits - 1)) : 1.f;
  // Every value rounded or accumulated stays within a few alphabet steps of
  // the weights; the offset leaves a wide margin above that.
  P.hdr->sigma = offset_for_bound(16.f * (maxw + maxs * (levels + 2.f)));
}

// Source tile index s lies in chunk s / B; it pushes itself to the targets
// s + 2 .. mid_end(s) - 1; the chunk product covers targets >= mid_end(s).
__host__ __device__ __forceinline__ int mid_end(int s) { return (s / B + 2) * B; }

// Solves every tile (I, K - I), I = I0 + blockIdx.x, of tile anti-diagonal K.
// 512 threads; lane p owns the two entries (p, q_j) of tile row p with
// p + q_j = 2 w + j (mod 32), j = 0, 1, w the warp: the entries of one
// anti-diagonal sit in one warp and one slot j, so only that warp runs the
// rounding step while the others accumulate.
constexpr int kSolveThreads = 512;
constexpr int kPer = T * T / kSolveThreads;  // entries per thread (2)
constexpr int kRows = kSolveThreads / T;     // rows per pass of the natural mapping (16)

__global__ void __launch_bounds__(kSolveThreads) tile_solve_kernel(QParams P, int K, int I0) {
  const int I = I0 + blockIdx.x;
  const int J = K - I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2 zero = make_float2(0.f, 0.f);

  // Strides are chosen so that every access pattern below is free of shared
  // memory bank conflicts (at most the two wavefronts of a 64-bit access).
  __shared__ float sLB[T][T + 2];   // L_B[I, I] (unit diagonal, zeros above)
  __shared__ float sLA[T][T + 2];   // L_A[J, J]
  __shared__ float sLBo[T][T + 1];  // L_B[I, I-1]
  __shared__ float sLAo[T][T + 1];  // L_A[J, J-1]
  __shared__ float2 sA[T][T + 2];   // G[I-1, J]; later the in-tile row sums
  __shared__ float2 sB[T][T + 2];   // E[I, J-1]; later W0 + X; later the tile's errors
  __shared__ float2 sGx[T][T + 1];  // full row-external sum of every entry
  const float sigma = P.hdr->sigma;

  // Loads in the natural mapping: rows a = warp + kRows t, column b = lane.
  const int b = lane;
  const int cb = J * T + b;
  const bool vb = cb < P.n;
  float2 c0[kPer], gf[kPer];
#pragma unroll
  for (int t = 0; t < kPer; ++t) {
    const int a = warp + kRows * t;
    const int ra = I * T + a;
    const bool va = ra < P.m;
    const int gc = I * T + b;
    sLB[a][b] = (va && gc < P.m) ? (b < a ? P.LB[(size_t)ra * P.m + gc] : (b == a ? 1.f : 0.f)) : 0.f;
    sLBo[a][b] = (I > 0 && va) ? P.LB[(size_t)ra * P.m + (I - 1) * T + b] : 0.f;
    const int rr = J * T + a, cc = J * T + b;
    sLA[a][b] = (rr < P.n && cc < P.n) ? (b < a ? P.LA[(size_t)rr * P.n + cc] : (b == a ? 1.f : 0.f)) : 0.f;
    sLAo[a][b] = (J > 0 && rr < P.n) ? P.LA[(size_t)rr * P.n + (J - 1) * T + b] : 0.f;
    sA[a][b] = (I > 0 && vb) ? P.G[(size_t)((I - 1) * T + a) * P.n + cb] : zero;
    sB[a][b] = (J > 0 && va) ? P.E[(size_t)ra * P.n + (J - 1) * T + b] : zero;
    c0[t] = zero;
    gf[t] = zero;
    if (va && vb) {
      const size_t o = (size_t)ra * P.n + cb;
      c0[t] = df_add(df_add(make_float2(P.W[o], 0.f), P.Xm[o]), P.Xc[o]);
      gf[t] = df_add(P.Gm[o], P.Gc[o]);
    }
  }
  __syncthreads();
  // Row-external sum: far pushes plus the distance-1 neighbour (I, J-1).
#pragma unroll
  for (int t = 0; t < kPer; ++t) {
    const int a = warp + kRows * t;
    OffsetAcc g;
    g.init(sigma);
    g.mac(1.f, gf[t]);
#pragma unroll 8
    for (int j = 0; j < T; ++j) g.mac(sLAo[b][j], sB[a][j]);
    gf[t] = g.value(sigma);
  }
  __syncthreads();
#pragma unroll
  for (int t = 0; t < kPer; ++t) {
    sGx[warp + kRows * t][b] = gf[t];
    sB[warp + kRows * t][b] = c0[t];
  }
  __syncthreads();

  // Skewed mapping.  acc: the whole value to round (tile input plus every
  // in-tile term); racc: the in-tile row terms alone (needed for the row
  // transform Gin = racc + e).
  const int p = lane;
  const int r = I * T + p;
  const bool vr = r < P.m;
  int qj[kPer];
  OffsetAcc acc[kPer], racc[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    qj[j] = (kPer * warp + j - p) & (T - 1);
    acc[j].init(sigma);
    racc[j].init(sigma);
    acc[j].mac(1.f, sB[p][qj[j]]);
  }
#pragma unroll 4
  for (int i = 0; i < T; ++i) {  // distance-1 neighbour (I-1, J)
    const float l = sLBo[p][i];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j].mac(l, sA[i][qj[j]]);
  }
  for (int i = 0; i <= p; ++i) {  // L_B[I, I] times the row-external sums
    const float l = sLB[p][i];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j].mac(l, sGx[i][qj[j]]);
  }
  const float s = (P.scales != nullptr && vr) ? P.scales[r] : 1.f;
  const float rcp = __frcp_rn(s);
  const float flo = (float)P.lo, fhi = (float)P.hi;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    sA[p][qj[j]] = zero;
    sB[p][qj[j]] = zero;
  }
  float vkeep[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) vkeep[j] = 0.f;
  __syncthreads();

  // Iteration k: first fold in the terms of anti-diagonal k-1 (published
  // before the barrier); the warp owning anti-diagonal k does this first for
  // the entries it rounds, rounds them and publishes; then every warp folds
  // the same terms into its other entries.
  for (int k = 0; k < 2 * T - 1; ++k) {
    const int ks = k - 1;    // source anti-diagonal of this iteration's terms
    const int jj = ks - p;   // row term: source column (the same for both entries)
    const float2 et = (jj >= 0 && jj < T) ? sB[p][jj] : zero;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int q = qj[j];
        const bool rounds_now = (p + q == k);
        if (rounds_now != (pass == 0)) continue;
        if (p + q > ks && ks >= 0) {
          if (jj >= 0 && jj < q) {
            const float l = sLA[q][jj];
            acc[j].mac(l, et);
            racc[j].mac(l, et);
          }
          const int i = ks - q;
          if (i >= 0 && i < p) {  // column term L_B[p, i] Gin[i, q], Gin = row sum + error
            const float l = sLB[p][i];
            acc[j].mac(l, sA[i][q]);
            acc[j].mac(l, sB[i][q]);
          }
        }
        if (rounds_now && vr && J * T + q < P.n) {
          const float2 x = acc[j].value(sigma);
          // fp32 decision: x.x == fp32(x); x.x * rcp is within 2 ulp of the
          // correctly rounded quotient, which is used near a rounding tie.
          float y = x.x * rcp;
          if (fabsf(y) > 256.f || fabsf(y - floorf(y) - 0.5f) < 1e-3f) y = __fdiv_rn(x.x, s);
          float v = rintf(y);
          if (P.bits) v = fminf(fmaxf(v, flo), fhi);
          // e = s v - x: exact high-word difference, then the low words
          const float2 sv = two_prod(s, v);
          const float2 h = two_sum(sv.x, -x.x);
          const float2 e = fast_two_sum(h.x, (sv.y - x.y) + h.y);
          sB[p][q] = e;
          sA[p][q] = racc[j].value(sigma);
          vkeep[j] = v;
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int c = J * T + qj[j];
    if (vr && c < P.n) {
      const size_t o = (size_t)r * P.n + c;
      P.V[o] = (int32_t)vkeep[j];
      P.Wq[o] = s * vkeep[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int t = 0; t < kPer; ++t) {  // natural mapping again: coalesced stores of E and G
    const int a = warp + kRows * t;
    const int ra = I * T + a;
    if (ra < P.m && vb) {
      const size_t o = (size_t)ra * P.n + cb;
      const float2 e = sB[a][b];
      P.E[o] = e;
      P.G[o] = df_add(sGx[a][b], df_add(sA[a][b], e));
    }
  }
}

// ---- asynchronous global -> shared copies (cp.async, zero-filled past the end)
__device__ __forceinline__ void cp_async(void* smem, const void* gmem, int src_bytes, int cp_bytes) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  if (cp_bytes == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
  } else if (cp_bytes == 8) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

// Shared memory of one push CTA (dynamic): NS stages of the factor block of
// up to U*T target rows by T source columns in its natural [row][k] layout
// (float4 reads along k) and of one source tile.  Mid pushes use one stage
// (a small footprint that fits beside the other kernels), chunk products two
// (the next source tile is copied in while the current one is used).
template <int NS>
struct PushSmem {
  float L[NS][U * T][T + 4];
  float2 S[NS][T][T + 2];
};

// Stages factor block rows [r0, r0 + U*T) x columns [k0, k0 + T) of the
// row-major d x d factor F (rows >= rows_valid or >= d, columns >= d: zero).
__device__ __forceinline__ void stage_factor(float (*dst)[T + 4], const float* F, int d, int r0, int rows_valid,
                                             int k0) {
  if ((d % 4) == 0) {  // 16-byte aligned rows
    for (int e = threadIdx.x; e < U * T * (T / 4); e += blockDim.x) {
      const int rr = e / (T / 4), k = 4 * (e % (T / 4));
      const int gr = r0 + rr, gk = k0 + k;
      const bool ok = rr < rows_valid && gr < d && gk < d;
      cp_async(&dst[rr][k], ok ? (const void*)(F + (size_t)gr * d + gk) : (const void*)F,
               ok ? 4 * min(4, d - gk) : 0, 16);
    }
  } else {
    for (int e = threadIdx.x; e < U * T * T; e += blockDim.x) {
      const int rr = e / T, k = e % T;
      const int gr = r0 + rr, gk = k0 + k;
      const bool ok = rr < rows_valid && gr < d && gk < d;
      cp_async(&dst[rr][k], ok ? (const void*)(F + (size_t)gr * d + gk) : (const void*)F, ok ? 4 : 0, 4);
    }
  }
}

// Stages the T x T double-float tile rows [r0, r0+T) x columns [c0, c0+T) of
// the m x n plane M (outside the matrix: zero).
__device__ __forceinline__ void stage_tile(float2 (*dst)[T + 2], const float2* M, int m, int n, int r0, int c0) {
  for (int e = threadIdx.x; e < T * T; e += blockDim.x) {
    const int rr = e / T, cc = e % T;
    const int gr = r0 + rr, gc = c0 + cc;
    const bool ok = gr < m && gc < n;
    cp_async(&dst[rr][cc], ok ? (const void*)(M + (size_t)gr * n + gc) : (const void*)M, ok ? 8 : 0, 8);
  }
}

// Column push: X[tiles tr0 .. tr0+ntr-1, column tile J] +=
//   L_B[those rows, source tile rows sr0 .. sr0+nsr-1] * G[source rows, column tile J].
// Lane l owns column l; warp w owns the 16 rows 16w .. 16w+15 (coalesced
// read-modify-write of 32 consecutive double-floats per row).
template <int NS>
__device__ void column_push(const QParams& P, PushSmem<NS>& sm, float2* X, int J, int tr0, int ntr, int sr0,
                            int nsr, float sigma) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int R = U * T / 8;  // rows per warp (16)
  const int rbase = R * warp;
  OffsetAcc acc[R];
#pragma unroll
  for (int u = 0; u < R; ++u) acc[u].init(sigma);
  const int rows = ntr * T;
  for (int st = 0; st < nsr; ++st) {
    const int buf = NS == 1 ? 0 : (st & 1);
    if (NS == 1 || st == 0) {
      stage_factor(sm.L[buf], P.LB, P.m, tr0 * T, rows, (sr0 + st) * T);
      stage_tile(sm.S[buf], P.G, P.m, P.n, (sr0 + st) * T, J * T);
      cp_async_commit();
    }
    if (NS == 2 && st + 1 < nsr) {
      stage_factor(sm.L[buf ^ 1], P.LB, P.m, tr0 * T, rows, (sr0 + st + 1) * T);
      stage_tile(sm.S[buf ^ 1], P.G, P.m, P.n, (sr0 + st + 1) * T, J * T);
      cp_async_commit();
      cp_async_wait_all_but_one();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < T; k += 4) {
      const float2 g0 = sm.S[buf][k][lane], g1 = sm.S[buf][k + 1][lane];
      const float2 g2 = sm.S[buf][k + 2][lane], g3 = sm.S[buf][k + 3][lane];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const float4 a = *reinterpret_cast<const float4*>(&sm.L[buf][rbase + u][k]);
        acc[u].mac(a.x, g0);
        acc[u].mac(a.y, g1);
        acc[u].mac(a.z, g2);
        acc[u].mac(a.w, g3);
      }
    }
    __syncthreads();
  }
  const int gc = J * T + lane;
  if (gc >= P.n) return;
#pragma unroll
  for (int u = 0; u < R; ++u) {
    const int gr = tr0 * T + rbase + u;
    if (rbase + u < rows && gr < P.m) {
      const size_t o = (size_t)gr * P.n + gc;
      X[o] = df_add(X[o], acc[u].value(sigma));
    }
  }
}

// Row push: Gp[row tile I, tiles tc0 .. tc0+ntc-1] +=
//   E[row tile I, source tile columns sc0 .. sc0+nsc-1] * L_A[target rows, source columns]^T.
// Lane l owns the columns l, l+32, l+64, l+96; warp w owns rows 4w .. 4w+3.
template <int NS>
__device__ void row_push(const QParams& P, PushSmem<NS>& sm, float2* Gp, int I, int tc0, int ntc, int sc0,
                         int nsc, float sigma) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int p0 = 4 * warp;
  OffsetAcc acc[4][U];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < U; ++v) acc[u][v].init(sigma);
  const int cols = ntc * T;
  for (int st = 0; st < nsc; ++st) {
    const int buf = NS == 1 ? 0 : (st & 1);
    if (NS == 1 || st == 0) {
      stage_factor(sm.L[buf], P.LA, P.n, tc0 * T, cols, (sc0 + st) * T);
      stage_tile(sm.S[buf], P.E, P.m, P.n, I * T, (sc0 + st) * T);
      cp_async_commit();
    }
    if (NS == 2 && st + 1 < nsc) {
      stage_factor(sm.L[buf ^ 1], P.LA, P.n, tc0 * T, cols, (sc0 + st + 1) * T);
      stage_tile(sm.S[buf ^ 1], P.E, P.m, P.n, I * T, (sc0 + st + 1) * T);
      cp_async_commit();
      cp_async_wait_all_but_one();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < T; k += 4) {
      float4 lv[U];
#pragma unroll
      for (int v = 0; v < U; ++v) lv[v] = *reinterpret_cast<const float4*>(&sm.L[buf][lane + T * v][k]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 e01 = *reinterpret_cast<const float4*>(&sm.S[buf][p0 + u][k]);
        const float4 e23 = *reinterpret_cast<const float4*>(&sm.S[buf][p0 + u][k + 2]);
        const float2 e0 = make_float2(e01.x, e01.y), e1 = make_float2(e01.z, e01.w);
        const float2 e2 = make_float2(e23.x, e23.y), e3 = make_float2(e23.z, e23.w);
#pragma unroll
        for (int v = 0; v < U; ++v) {
          acc[u][v].mac(lv[v].x, e0);
          acc[u][v].mac(lv[v].y, e1);
          acc[u][v].mac(lv[v].z, e2);
          acc[u][v].mac(lv[v].w, e3);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int gr = I * T + p0 + u;
    if (gr >= P.m) continue;
#pragma unroll
    for (int v = 0; v < U; ++v) {
      const int cc = lane + T * v;
      const int gc = tc0 * T + cc;
      if (cc < cols && gc < P.n) {
        const size_t o = (size_t)gr * P.n + gc;
        Gp[o] = df_add(Gp[o], acc[u][v].value(sigma));
      }
    }
  }
}

// Mid pushes of the sources of tile anti-diagonal K (blockIdx.x: source
// I = I0 + blockIdx.x; blockIdx.y: group of U targets, column targets first).
__global__ void __launch_bounds__(256) mid_push_kernel(QParams P, int K, int I0) {
  extern __shared__ __align__(16) unsigned char push_smem[];
  PushSmem<1>& sm = *reinterpret_cast<PushSmem<1>*>(push_smem);
  const int I = I0 + blockIdx.x, J = K - I;
  const int c_first = I + 2, c_end = min(P.Mt, mid_end(I));
  const int r_first = J + 2, r_end = min(P.Nt, mid_end(J));
  const int ncu = c_end > c_first ? (c_end - c_first + U - 1) / U : 0;
  const int nru = r_end > r_first ? (r_end - r_first + U - 1) / U : 0;
  const int u = blockIdx.y;
  const float sigma = P.hdr->sigma;
  if (u < ncu) {
    const int t0 = c_first + u * U;
    column_push(P, sm, P.Xm, J, t0, min(U, c_end - t0), I, 1, sigma);
  } else if (u < ncu + nru) {
    const int t0 = r_first + (u - ncu) * U;
    row_push(P, sm, P.Gm, I, t0, min(U, r_end - t0), J, 1, sigma);
  }
}

// (At most 85 registers per thread: three chunk CTAs fit in the register
// file.)
// Chunk products launched once tile anti-diagonal K is solved: for every
// column J whose tile (K - J, J) closes a chunk of B tile rows, and every row
// I whose tile (I, K - I) closes a chunk of B tile columns.  blockIdx.x:
// candidate (columns first, J = K - (B-1) - B*t, then rows likewise);
// blockIdx.y: group of U targets.
__global__ void __launch_bounds__(256, 3) chunk_push_kernel(QParams P, int K, int ncand_col) {
  extern __shared__ __align__(16) unsigned char push_smem[];
  PushSmem<2>& sm = *reinterpret_cast<PushSmem<2>*>(push_smem);
  const float sigma = P.hdr->sigma;
  const int t = blockIdx.x, u = blockIdx.y;
  if (t < ncand_col) {
    const int J = K - (B - 1) - B * t;      // the chunk's last tile row is K - J = B - 1 + B t
    const int last = K - J;
    if (J < 0 || J >= P.Nt || last >= P.Mt) return;
    const int c = last / B;
    const int first = (c + 2) * B;
    const int ntiles = P.Mt - first;
    if (ntiles <= 0 || u * U >= ntiles) return;
    column_push(P, sm, P.Xc, J, first + u * U, min(U, ntiles - u * U), c * B, B, sigma);
  } else {
    const int I = K - (B - 1) - B * (t - ncand_col);
    const int last = K - I;
    if (I < 0 || I >= P.Mt || last >= P.Nt) return;
    const int c = last / B;
    const int first = (c + 2) * B;
    const int ntiles = P.Nt - first;
    if (ntiles <= 0 || u * U >= ntiles) return;
    row_push(P, sm, P.Gc, I, first + u * U, min(U, ntiles - u * U), c * B, B, sigma);
  }
}

// Event pairs around launches when a KernelTimer is given (diagnostics).
class LaunchClock {
 public:
  explicit LaunchClock(KernelTimer* t) : t_(t) {
    if (t_) {
      for (int c = 0; c < kKernelClasses; ++c) {
        t_->ms[c] = 0.0;
        t_->launches[c] = 0;
        t_->flops[c] = 0.0;
      }
    }
  }
  ~LaunchClock() {
    for (auto& r : recs_) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
  }
  void begin(int cls, cudaStream_t s) {
    if (!t_) return;
    Rec r;
    r.cls = cls;
    r.s = s;
    cudaEventCreate(&r.a);
    cudaEventCreate(&r.b);
    cudaEventRecord(r.a, s);
    recs_.push_back(r);
  }
  void end(double flops) {
    if (!t_) return;
    Rec& r = recs_.back();
    cudaEventRecord(r.b, r.s);
    t_->launches[r.cls] += 1;
    t_->flops[r.cls] += flops;
  }
  cudaError_t finish(cudaStream_t s) {
    if (!t_) return cudaSuccess;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    for (auto& r : recs_) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, r.a, r.b);
      if (e != cudaSuccess) return e;
      t_->ms[r.cls] += ms;
    }
    return cudaSuccess;
  }

 private:
  struct Rec {
    int cls;
    cudaStream_t s;
    cudaEvent_t a, b;
  };
  KernelTimer* t_;
  std::vector<Rec> recs_;
};

// Two side streams and the ordering events, one set per device, reused by
// every call.  Streams and events are driver objects, not device memory.
// Calls that share a set serialize their side work on its streams, which
// is correct: each call's main stream waits only on its own events' records.
// Dynamic shared memory: a mid push CTA holds one stage, a chunk CTA two
// (53 KB: three chunk CTAs fit in an SM's shared memory, as in its register
// file).  Capping chunk CTAs at two per SM with unused extra space, to keep
// room for the other kernels, was measured slower: 22.6 against 22.3 ms on a
// 4096 x 4096 layer, 146.6 against 136.0 ms on 14336 x 4096.
constexpr int kMidSmem = (int)sizeof(PushSmem<1>);
constexpr int kChunkSmem = (int)sizeof(PushSmem<2>);

struct StreamSet {
  bool ready = false;
  cudaStream_t mid = nullptr, chunk = nullptr;
  std::vector<cudaEvent_t> ev;
};
constexpr int kMaxDevices = 128;
StreamSet g_sets[kMaxDevices];
std::mutex g_set_mutex;

cudaError_t prepare_set(StreamSet& S, size_t nev) {
  cudaError_t e;
  if (!S.ready) {
    int lo = 0, hi = 0;
    e = cudaDeviceGetStreamPriorityRange(&lo, &hi);  // hi is the most urgent (numerically lowest)
    if (e != cudaSuccess) return e;
    // Both side streams get the highest priority: the chunk products are
    // the largest block of work and their stream sets the pace (measured on
    // c3: 23.3 ms with the chunk stream at the lowest priority, 22.6 ms here).
    (void)lo;
    e = cudaStreamCreateWithPriority(&S.mid, cudaStreamNonBlocking, hi);
    if (e != cudaSuccess) return e;
    e = cudaStreamCreateWithPriority(&S.chunk, cudaStreamNonBlocking, hi);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chunk_push_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kChunkSmem);
    if (e != cudaSuccess) return e;
    S.ready = true;
  }
  while (S.ev.size() < nev) {
    cudaEvent_t x;
    e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    S.ev.push_back(x);
  }
  return cudaSuccess;
}

}  // namespace

size_t quantize_workspace_bytes(int64_t m, int64_t n) {
  const size_t plane = align_up((size_t)m * (size_t)n * sizeof(float2));
  return sizeof(Header) + kPlanes * plane;
}

cudaError_t quantize_launch(const float* W, const float* LA, const float* LB, const float* scales,
                            int bits, int m, int n, int32_t* V, float* Wq, void* ws,
                            int32_t* status_dev, cudaStream_t stream, KernelTimer* timer) {
  const size_t plane = align_up((size_t)m * (size_t)n * sizeof(float2));
  char* base = static_cast<char*>(ws);
  float2* planes = reinterpret_cast<float2*>(base + sizeof(Header));
  const size_t pstride = plane / sizeof(float2);
  QParams P;
  P.W = W;
  P.LA = LA;
  P.LB = LB;
  P.scales = scales;
  P.V = V;
  P.Wq = Wq;
  P.hdr = reinterpret_cast<Header*>(base);
  P.Xm = planes;
  P.Xc = planes + pstride;
  P.Gm = planes + 2 * pstride;
  P.Gc = planes + 3 * pstride;
  P.G = planes + 4 * pstride;
  P.E = planes + 5 * pstride;
  P.status = status_dev;
  P.m = m;
  P.n = n;
  P.Mt = (m + T - 1) / T;
  P.Nt = (n + T - 1) / T;
  P.bits = bits;
  P.lo = bits ? -(1 << (bits - 1)) : 0;
  P.hi = bits ? (1 << (bits - 1)) - 1 : 0;
  const int Kmax = P.Mt + P.Nt - 2;

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_set_mutex);
  StreamSet& S = g_sets[dev];
  const size_t nev = 3 * (size_t)(Kmax + 1) + 1;
  err = prepare_set(S, nev);
  if (err != cudaSuccess) return err;
  cudaEvent_t* ev_solve = S.ev.data();
  cudaEvent_t* ev_mid = ev_solve + (Kmax + 1);
  cudaEvent_t* ev_chunk = ev_mid + (Kmax + 1);
  cudaEvent_t ev_start = ev_chunk[Kmax + 1];
  // With a timer every kernel runs on the caller's stream, one after the
  // other, so that each event pair brackets one kernel alone.
  cudaStream_t s_mid = timer ? stream : S.mid;
  cudaStream_t s_chunk = timer ? stream : S.chunk;

  LaunchClock clock(timer);
  err = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(P.hdr, 0, sizeof(Header), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(planes, 0, 4 * plane, stream);  // Xm, Xc, Gm, Gc
  if (err != cudaSuccess) return err;
  const size_t total = (size_t)m * n;
  const int pre_blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 8);
  clock.begin(0, stream);
  prepass_kernel<<<pre_blocks, 256, 0, stream>>>(P);
  sigma_kernel<<<1, 1, 0, stream>>>(P);
  clock.end(0.0);
  cudaEventRecord(ev_start, stream);
  cudaStreamWaitEvent(s_mid, ev_start, 0);
  cudaStreamWaitEvent(s_chunk, ev_start, 0);

  const double t3 = (double)T * T * T;
  std::vector<char> mid_on(Kmax + 1, 0), chunk_on(Kmax + 1, 0);
  int last_mid = -1, last_chunk = -1;
  for (int K = 0; K <= Kmax; ++K) {
    const int I0 = std::max(0, K - (P.Nt - 1));
    const int I1 = std::min(K, P.Mt - 1);
    const int nsrc = I1 - I0 + 1;
    if (K >= 2 && mid_on[K - 2]) cudaStreamWaitEvent(stream, ev_mid[K - 2], 0);
    // Stream order makes one wait enough: mid(K-2) and chunk(K-B-1) follow
    // every earlier launch of their streams, and a missing launch was covered
    // by the wait of an earlier solve.
    if (K >= B + 1 && chunk_on[K - B - 1]) cudaStreamWaitEvent(stream, ev_chunk[K - B - 1], 0);
    clock.begin(1, stream);
    tile_solve_kernel<<<nsrc, kSolveThreads, 0, stream>>>(P, K, I0);
    clock.end(2.0 * 3.5 * t3 * nsrc);  // in-tile sums, L_B[I,I] row part, two distance-1 pulls
    cudaEventRecord(ev_solve[K], stream);

    // mid pushes from the sources of K
    double mid_tiles = 0;
    for (int I = I0; I <= I1; ++I) {
      const int J = K - I;
      mid_tiles += std::max(0, std::min(P.Mt, mid_end(I)) - (I + 2));
      mid_tiles += std::max(0, std::min(P.Nt, mid_end(J)) - (J + 2));
    }
    if (mid_tiles > 0) {
      cudaStreamWaitEvent(s_mid, ev_solve[K], 0);
      const int units = 2 * ((2 * B - 2 + U - 1) / U);
      clock.begin(2, s_mid);
      mid_push_kernel<<<dim3(nsrc, units), 256, kMidSmem, s_mid>>>(P, K, I0);
      clock.end(2.0 * t3 * mid_tiles);
      cudaEventRecord(ev_mid[K], s_mid);
      mid_on[K] = 1;
      last_mid = K;
    }

    // chunk products closed by K
    const int ncc = std::min(K, P.Mt - 1) >= B - 1 ? (std::min(K, P.Mt - 1) - (B - 1)) / B + 1 : 0;
    const int ncr = std::min(K, P.Nt - 1) >= B - 1 ? (std::min(K, P.Nt - 1) - (B - 1)) / B + 1 : 0;
    double chunk_tiles = 0;
    for (int t = 0; t < ncc; ++t) {
      const int J = K - (B - 1) - B * t, last = K - J;
      if (J >= 0 && J < P.Nt && last < P.Mt) chunk_tiles += std::max(0, P.Mt - (last / B + 2) * B);
    }
    for (int t = 0; t < ncr; ++t) {
      const int I = K - (B - 1) - B * t, last = K - I;
      if (I >= 0 && I < P.Mt && last < P.Nt) chunk_tiles += std::max(0, P.Nt - (last / B + 2) * B);
    }
    if (chunk_tiles > 0) {
      cudaStreamWaitEvent(s_chunk, ev_solve[K], 0);
      const int units = (std::max(P.Mt, P.Nt) + U - 1) / U;
      clock.begin(3, s_chunk);
      chunk_push_kernel<<<dim3(ncc + ncr, units), 256, kChunkSmem, s_chunk>>>(P, K, ncc);
      clock.end(2.0 * B * t3 * chunk_tiles);
      cudaEventRecord(ev_chunk[K], s_chunk);
      chunk_on[K] = 1;
      last_chunk = K;
    }
  }
  // Join: the caller's stream covers all side work of this call.
  if (last_mid >= 0) cudaStreamWaitEvent(stream, ev_mid[last_mid], 0);
  if (last_chunk >= 0) cudaStreamWaitEvent(stream, ev_chunk[last_chunk], 0);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return clock.finish(stream);
}

}  // namespace bakron
