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
// With L_B = I (row-wise GPTQ) only the row part exists, a tile depends on
// nothing but the earlier tiles of its own tile row, and a step K is a whole
// tile column J = K (QParams::skew = 0) instead of a tile anti-diagonal.
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
// and of its column sum (L_B[p, k-q] G[k-q, q], G = the full row transform,
// published by each entry as it is rounded).
//
// Precision: every accumulation is double-float (df.cuh) or exact (the
// digit products of the chunk products on the tensor cores, see that
// section); the rounding decision is the fp32 quotient fp32(W~) / s_i
// rounded half to even, with the correctly rounded division used whenever
// the quotient is near a tie.  The tile solves also write E and G as bf16
// digit planes, the source operands of the chunk products.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "bakron.h"
#include "df.cuh"
#include "internal.h"
#include "solve_common.cuh"
#include "tc.cuh"

namespace bakron {
namespace {

constexpr int U = 4;   // target tiles per push CTA

constexpr int kPlanes = 6;  // Xm, Xc, Gm, Gc, G, E

struct QParams {
  const float* W;
  const float* LA;
  const float* LB;
  const float* scales;   // m x ngroups row (group) scales, or null
  const float* cscales;  // n column scales, or null
  int group, ngroups;    // columns per scale run; runs per row
  int32_t* V;
  float* Wq;
  float2* Xm;  // column pushes from single tiles (mid)
  long long* Xc;  // column pushes from chunks (64-bit fixed point, see fixed_unit_exp)
  float2* Gm;  // row pushes from single tiles (mid)
  long long* Gc;  // row pushes from chunks (likewise)
  float2* G;   // full row transform of each solved entry
  float2* E;   // errors at rounding time
  Header* hdr;
  int32_t* status;
  const signed char* expA;    // (row, chunk) exponents of L_A and L_B (chunk products)
  const signed char* expB;
  const __nv_bfloat16* FdA;   // factor digits of L_A and L_B, packed for bulk copies (factor_digits_kernel)
  const __nv_bfloat16* FdB;
  __nv_bfloat16* DE;          // digits of E, [digit][row][ldE], ldE = n rounded up to 8
  __nv_bfloat16* DGt;         // digits of G transposed, [digit][col][ldG], ldG = m rounded up to 8
  size_t dstrideE, dstrideG;  // elements per digit plane
  int ldE, ldG;
  int m, n, Mt, Nt, bits, lo, hi, nchA, nchB;
  int ntA, ntB;               // tile rows (32) of the packed factor digits
  // Step of tile (I, J): J + skew I.  skew = 1 (BaKron): tile anti-diagonals;
  // skew = 0 (L_B = I, row-wise GPTQ): tile columns, all rows at once, since
  // a row then depends on nothing but its own earlier entries.
  int skew;
};

// Source tile index s lies in chunk s / B; it pushes itself to the targets
// s + 2 .. mid_end(s) - 1; the chunk product covers targets >= mid_end(s).
__host__ __device__ __forceinline__ int mid_end(int s) { return (s / B + 2) * B; }

// Solves every tile (I, K - skew I), I = I0 + blockIdx.x, of step K (a tile
// anti-diagonal, or with L_B = I a tile column).
// kSolveThreads threads (1024 or 512); lane p owns the kPer = 1024 /
// kSolveThreads entries (p, q_j) of tile row p with p + q_j = kPer w + j
// (mod 32), j < kPer, w the warp: the entries of one anti-diagonal sit in
// one warp and one slot j, so only that warp runs the rounding step while
// the others accumulate.  Measured on one GB300: 1024 threads solve 4096 x
// 4096 in 14.2 ms against 14.7 ms with 512 (256: 19.3 ms); on 14336 x 4096,
// where a 1024-thread solve leaves no room on its SM for a chunk product
// CTA, 512 threads are faster (67.1 against 68.8 ms).
template <int kSolveThreads>
__global__ void __launch_bounds__(kSolveThreads) tile_solve_kernel(QParams P, int K, int I0) {
  constexpr int kPer = T * T / kSolveThreads;  // entries per thread
  constexpr int kRows = kSolveThreads / T;     // rows per pass of the natural mapping
  const int I = I0 + blockIdx.x;
  const int J = K - P.skew * I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2 zero = make_float2(0.f, 0.f);

  // Strides are chosen so that every access pattern below is free of shared
  // memory bank conflicts (at most the two wavefronts of a 64-bit access).
  __shared__ float sLB[T][T + 2];   // L_B[I, I] (unit diagonal, zeros above)
  __shared__ float sLA[T][T + 2];   // L_A[J, J]
  __shared__ float sLBo[T][T + 1];  // L_B[I, I-1]
  __shared__ float sLAo[T][T + 1];  // L_A[J, J-1]
  __shared__ float2 sA[T][T + 2];   // G[I-1, J]; later the tile's own G
  __shared__ float2 sB[T][T + 2];   // E[I, J-1]; later W0 + X; later the tile's errors
  __shared__ float2 sGx[T][T + 1];  // full row-external sum of every entry
  const float sigma = P.hdr->sigma;
  const float from_units = pow2f(fixed_unit_exp(sigma));

  // Each entry's scale in the skewed mapping below (lane p = tile row, slot
  // j = column qj[j]): its row (group) scale times its column scale,
  // rounded once to fp32, and its reciprocal for the rounding decision;
  // loaded first, so that their latency overlaps the loads below.
  float se[kPer], rcpe[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int pr = I * T + lane;
    const int c = J * T + ((kPer * warp + j - lane) & (T - 1));
    float sv = 1.f;
    if (pr < P.m && c < P.n) {
      if (P.scales) sv = P.scales[(size_t)pr * P.ngroups + c / P.group];
      if (P.cscales) sv = __fmul_rn(sv, P.cscales[c]);
    }
    se[j] = sv;
  }
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
    sLB[a][b] = (va && gc < P.m) ? (b < a ? (P.LB ? P.LB[(size_t)ra * P.m + gc] : 0.f) : (b == a ? 1.f : 0.f)) : 0.f;
    sLBo[a][b] = (I > 0 && va && P.LB) ? P.LB[(size_t)ra * P.m + (I - 1) * T + b] : 0.f;
    const int rr = J * T + a, cc = J * T + b;
    sLA[a][b] = (rr < P.n && cc < P.n) ? (b < a ? P.LA[(size_t)rr * P.n + cc] : (b == a ? 1.f : 0.f)) : 0.f;
    sLAo[a][b] = (J > 0 && rr < P.n) ? P.LA[(size_t)rr * P.n + (J - 1) * T + b] : 0.f;
    sA[a][b] = (I > 0 && vb && P.LB) ? P.G[(size_t)((I - 1) * T + a) * P.n + cb] : zero;
    sB[a][b] = (J > 0 && va) ? P.E[(size_t)ra * P.n + (J - 1) * T + b] : zero;
    c0[t] = zero;
    gf[t] = zero;
    if (va && vb) {
      const size_t o = (size_t)ra * P.n + cb;
      c0[t] = df_add(df_add(make_float2(P.W[o], 0.f), P.Xm[o]), df_from_fixed(P.Xc[o], from_units));
      gf[t] = df_add(P.Gm[o], df_from_fixed(P.Gc[o], from_units));
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

  // Skewed mapping.  acc: the tile input, the distance-1 column pull and the
  // in-tile column terms L_B[p, i] G[i, q] (i < p, in the tile); racc: the
  // entry's row transform without its own error, i.e. its row-external sum
  // plus the in-tile row terms, so that racc + e = G[p, q], the value the
  // entry publishes for the column terms of the entries below it.  Both
  // offset accumulators share sigma, so the value to round, acc + racc, is
  // formed from them exactly when the entry's turn comes.
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
    racc[j].mac(1.f, sGx[p][qj[j]]);
  }
  const bool colterms = P.LB != nullptr;  // L_B = I (row-wise GPTQ): no column terms at all
  if (colterms) {
#pragma unroll 4
    for (int i = 0; i < T; ++i) {  // distance-1 neighbour (I-1, J)
      const float l = sLBo[p][i];
#pragma unroll
      for (int j = 0; j < kPer; ++j) acc[j].mac(l, sA[i][qj[j]]);
    }
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) rcpe[j] = __frcp_rn(se[j]);
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
          if (jj >= 0 && jj < q) racc[j].mac(sLA[q][jj], et);                 // row term E[p, jj] L_A[q, jj]
          const int i = ks - q;
          if (colterms && i >= 0 && i < p) acc[j].mac(sLB[p][i], sA[i][q]);     // column term L_B[p, i] G[i, q]
        }
        if (rounds_now && vr && J * T + q < P.n) {
          // (acc.H - sigma) and (racc.H - sigma) are exact and so is their
          // sum (two multiples of the offset's half-ulp, below sigma).
          const float2 x = two_sum((acc[j].H - sigma) + (racc[j].H - sigma), acc[j].L + racc[j].L);
          // fp32 decision: x.x == fp32(x); x.x * rcp is within 2 ulp of the
          // correctly rounded quotient, which is used near a rounding tie
          // (and for an infinite or NaN product: a scale below 2^-128).
          float y = x.x * rcpe[j];
          if (!(fabsf(y) <= 256.f) || fabsf(y - floorf(y) - 0.5f) < 1e-3f) y = __fdiv_rn(x.x, se[j]);
          float v = rintf(y);
          if (P.bits) v = fminf(fmaxf(v, flo), fhi);
          // e = s v - x: exact high-word difference, then the low words
          const float2 sv = two_prod(se[j], v);
          const float2 h = two_sum(sv.x, -x.x);
          const float2 e = fast_two_sum(h.x, (sv.y - x.y) + h.y);
          sB[p][q] = e;
          sA[p][q] = df_add(racc[j].value(sigma), e);  // G[p, q]: the entry's full row transform
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
      P.Wq[o] = se[j] * vkeep[j];
    }
  }
  __syncthreads();
  const float dsc = pow2f(7 - bound_exp(sigma));
  float2 gv[kPer];
#pragma unroll
  for (int t = 0; t < kPer; ++t) {  // natural mapping again: coalesced stores of E and G
    const int a = warp + kRows * t;
    const int ra = I * T + a;
    const float2 e = sB[a][b];
    gv[t] = sA[a][b];  // G, published by the entry's rounding
    if (ra < P.m && vb) {
      const size_t o = (size_t)ra * P.n + cb;
      P.E[o] = e;
      P.G[o] = gv[t];
      put_digits(P.DE, P.dstrideE, (size_t)ra * P.ldE + cb, e, dsc);
    }
  }
  __syncthreads();  // every read of sGx above is done
#pragma unroll
  for (int t = 0; t < kPer; ++t) sGx[warp + kRows * t][b] = gv[t];
  __syncthreads();
#pragma unroll
  for (int t = 0; t < kPer; ++t) {  // G digits transposed (column products only): lane = row, coalesced
    const int col = warp + kRows * t, row = lane;
    const int gr = I * T + row, gc = J * T + col;
    if (P.LB && gr < P.m && gc < P.n) put_digits(P.DGt, P.dstrideG, (size_t)gc * P.ldG + gr, sGx[row][col], dsc);
  }
}

// ---- asynchronous global -> shared copies (cp.async, zero-filled past the end)
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
  if ((d % 4) == 0 && (reinterpret_cast<uintptr_t>(F) & 15) == 0) {  // 16-byte aligned rows
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
  // Read-modify-write of the plane: all loads first, so that they are in
  // flight together (a store between them would order each load after it).
  float2 old[R];
#pragma unroll
  for (int u = 0; u < R; ++u) {
    const int gr = tr0 * T + rbase + u;
    old[u] = (rbase + u < rows && gr < P.m) ? X[(size_t)gr * P.n + gc] : make_float2(0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < R; ++u) {
    const int gr = tr0 * T + rbase + u;
    if (rbase + u < rows && gr < P.m) X[(size_t)gr * P.n + gc] = df_add(old[u], acc[u].value(sigma));
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
  // Read-modify-write of the plane: all loads first (see column_push).
  float2 old[4][U];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < U; ++v) {
      const int gr = I * T + p0 + u, cc = lane + T * v, gc = tc0 * T + cc;
      old[u][v] = (gr < P.m && cc < cols && gc < P.n) ? Gp[(size_t)gr * P.n + gc] : make_float2(0.f, 0.f);
    }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < U; ++v) {
      const int gr = I * T + p0 + u, cc = lane + T * v, gc = tc0 * T + cc;
      if (gr < P.m && cc < cols && gc < P.n) Gp[(size_t)gr * P.n + gc] = df_add(old[u][v], acc[u][v].value(sigma));
    }
}

// Mid pushes of the sources of step K (blockIdx.x: source I = I0 +
// blockIdx.x, J = K - skew I; blockIdx.y: group of U targets, column
// targets first).
__global__ void __launch_bounds__(256) mid_push_kernel(QParams P, int K, int I0) {
  extern __shared__ __align__(16) unsigned char push_smem[];
  PushSmem<1>& sm = *reinterpret_cast<PushSmem<1>*>(push_smem);
  const int I = I0 + blockIdx.x, J = K - P.skew * I;
  const int c_first = I + 2, c_end = P.LB ? min(P.Mt, mid_end(I)) : c_first;  // L_B = I: no column pushes
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

// ---- Chunk products on the tensor cores (tcgen05), by an exact digit split
// (after Ozaki, Ogita, Oishi and Rump, "Error-free transformations of matrix
// multiplication by using fast routines of matrix multiplication and its
// applications", Numer. Algorithms 2012).
//
// A chunk product is Y (128 x T) = F (128 x CK) * D (CK x T): F a block of
// a factor (fp32, 128 target rows), D a source block of G or E^T
// (double-float), CK = B*T.  With e_r bounding row r of F over the chunk
// (|F[r][k]| < 2^e_r) and eD the global exponent of the source digits,
//   F[r][k] ~ 2^(e_r-7) sum_{a<5} f_a[r][k] 256^-a,
//   D[k][q] ~ 2^(eD-7) sum_{b<6} d_b[k][q] 256^-b,
// with integer digits |f_a|, |d_b| <= 128, exact in bf16.  Five digits hold
// every factor element whose magnitude is at least 2^-16 of its row's bound
// exactly (an fp32 significand has 24 bits) and the others to 2^-40 of the
// bound.  (Four factor digits leave an error near 1e-9 of sum |F||D| on
// factor rows whose entries span a few binades; five leave 6e-13.)  Every
// digit product is exact, and per level l = a + b the sum over k and over
// the <= 5 pairs of the level stays below 5 * 128 * 128^2 < 2^24, so the
// fp32 accumulation of each level in tensor memory is exact.  The 20 pairs
// of levels 0..5 are kept (the dropped ones are below 2^-48 of row bound
// times 2^eD); the levels are summed in double-float and scaled by
// 2^(e_r + eD - 14).
constexpr int kTcM = 128;        // target rows per group (UC target tiles)
constexpr int UC = kTcM / T;
constexpr int kMaxItems = 16;  // (candidate, target group) items one chunk product CTA works through
constexpr int kItemsPerCand = 8;  // items per CTA when each CTA serves one candidate (packed digits)

// Chunk product candidates closed by tile anti-diagonal K: for every column
// J whose tile (K - J, J) closes a chunk of B tile rows, and every row I
// whose tile (I, K - I) closes a chunk of B tile columns (candidate t:
// columns first, J = K - (B-1) - B t, then rows likewise).  The product
// covers the target tiles from chunk c + 2 on.
struct ChunkCand {
  bool col;
  int J, I, c, first, ntiles;
};
__host__ __device__ __forceinline__ bool chunk_candidate(const QParams& P, int K, int ncand_col, int t,
                                                         ChunkCand& cc) {
  cc.col = t < ncand_col;
  if (cc.col) {
    cc.J = K - (B - 1) - B * t;
    cc.I = 0;
    const int last = K - cc.J;
    if (cc.J < 0 || cc.J >= P.Nt || last >= P.Mt) return false;
    cc.c = last / B;
    cc.first = (cc.c + 2) * B;
    cc.ntiles = P.Mt - cc.first;
  } else if (P.skew == 0) {
    // tile columns: every row closes a chunk of B tile columns together
    cc.I = t - ncand_col;
    cc.J = 0;
    const int last = K;
    if ((K + 1) % B != 0 || cc.I >= P.Mt || last >= P.Nt) return false;
    cc.c = last / B;
    cc.first = (cc.c + 2) * B;
    cc.ntiles = P.Nt - cc.first;
  } else {
    cc.I = K - (B - 1) - B * (t - ncand_col);
    cc.J = 0;
    const int last = K - cc.I;
    if (cc.I < 0 || cc.I >= P.Mt || last >= P.Nt) return false;
    cc.c = last / B;
    cc.first = (cc.c + 2) * B;
    cc.ntiles = P.Nt - cc.first;
  }
  return cc.ntiles > 0;
}

// Candidates of the chunk products closed by step K (chunk_candidate's t
// ranges over ncc column candidates, then ncr row candidates).
inline void chunk_counts(const QParams& P, int K, bool colpush, int& ncc, int& ncr) {
  ncc = (colpush && std::min(K, P.Mt - 1) >= B - 1) ? (std::min(K, P.Mt - 1) - (B - 1)) / B + 1 : 0;
  ncr = P.skew ? (std::min(K, P.Nt - 1) >= B - 1 ? (std::min(K, P.Nt - 1) - (B - 1)) / B + 1 : 0)
               : ((K + 1) % B == 0 ? P.Mt : 0);  // tile columns: every row closes a chunk
}

// Warp roles of a chunk product CTA.
constexpr int kTcMmaWarp = 0;           // issues the tensor-core products (lane 0)
constexpr int kTcCopyWarp = 1;          // packed digits: lane 0 loads the factor digit slabs (bulk copies)
constexpr int kTcEpiWarp0 = 4;          // warps 4..7: epilogue, tensor-memory lane quarters 0..3
constexpr int kTcStages = 3;            // fp32 factor slabs in flight per producer (digits made in the kernel)
constexpr int kEpiCols = 8;             // output columns per epilogue step (registers: 6 levels each)

// Two ways to feed the factor digits.  Packed (layers of 2^22 weights and
// more): the digits are computed once per solve (factor_digits_kernel) and
// each slab arrives as five bulk copies, 8 warps.  In the kernel (smaller
// layers): 7 producer warps copy fp32 factor slabs with cp.async and split
// them into digits, 12 warps.  Packed reads 10 bytes per factor entry
// instead of 4 but needs no producer warps; measured on one GB300:
// 4096 x 4096 14.7 ms against 15.8 ms, 14336 x 4096 66.8 against 78.6 ms;
// 1024 x 1024 is the same either way.
inline bool use_packed_digits(int64_t m, int64_t n) { return m * n >= ((int64_t)1 << 22); }
// Layers above 2^24 weights, where the chunk products set the pace: one
// candidate per chunk-product CTA, and the tile solves on the caller's
// stream (see quantize_launch).
inline bool large_layer(int64_t m, int64_t n) { return m * n > ((int64_t)1 << 24); }

template <bool kPacked>
struct TcShape {
  static constexpr int kWarps = kPacked ? 8 : 12;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kProducers = kPacked ? 0 : (kWarps - 5) * 32;  // warps 1..3 and 8..11
};

template <bool kPacked>
struct TcStage {
  float stage[kTcStages][kTcM][kSlab];  // fp32 factor slabs as loaded
};
template <>
struct TcStage<true> {};

// Digit slab buffers: three with packed digits (bulk copies in flight while
// two slabs wait for or feed the products), two when the producer warps
// make them (their fp32 staging takes the room of the third).
template <bool kPacked>
constexpr int kDigBufs = kPacked ? 3 : 2;

template <bool kPacked>
struct TcSmem : TcStage<kPacked> {
  __nv_bfloat16 A[kDigBufs<kPacked>][kDigF][kTcM * kSlab];  // factor digit slabs, core-matrix layout (SBO 512 B)
  __nv_bfloat16 Bd[kDigD * T * CK];         // source digits, 192 rows (digit-major) x CK, SBO 2048 B
  signed char er[kMaxItems][kTcM];          // row exponents of each item's factor block
  ChunkCand cand[kMaxItems];                // the candidate of each item
  int grp[kMaxItems];                       // its target group within the candidate
  int seg[kMaxItems];                       // 1 where an item starts a new candidate (after the first)
  int count;                                // items mapped (the CTA's share of the launch)
  uint64_t full[kDigBufs<kPacked>];         // digit slab p ready (producer arrivals / bulk-copy bytes)
  uint64_t empty[kDigBufs<kPacked>];        // products reading digit slab p done (commit)
  uint64_t grp_full[2];                     // products of a group in tensor-memory half h done (commit)
  uint64_t grp_empty[2];                    // epilogue of tensor-memory half h done (epilogue arrivals)
  uint64_t bd_free;                         // products reading the source digits of a candidate done (commit)
  uint64_t bd_full;                         // the next candidate's source digits loaded (copier arrivals)
  uint32_t tmem_base;
};

// Chunk products closed by tile anti-diagonal K.  The work of a launch is
// the list of items (candidate t, target group g of 128 target rows),
// ordered by candidate and then group, G items in all; CTA b takes the
// items G b / gridDim.x .. G (b + 1) / gridDim.x - 1 (at most kMaxItems),
// so that one wave of CTAs shares the launch evenly.  Column products:
//   Xc[targets, J] += L_B[targets, chunk rows] G[chunk rows, J];
// row products, as their transpose:
//   Gc[I, targets]^T += L_A[targets, chunk cols] E[I, chunk cols]^T.
// Warp-specialized pipeline over the k-slabs of all items of the CTA:
//  * the next slab's five factor digit blocks go into one of the digit
//    buffers (three with packed digits, else two) once the products that
//    read that buffer are done: bulk copies of the packed digits by one
//    thread, or fp32 slabs copied two ahead (cp.async) by the producer
//    warps and split into digits there;
//  * one thread issues, per 16-deep k-step, five MMAs: factor digit a times
//    the source digits 0 .. 5-a stacked along N (N = 32 (6 - a)), written at
//    tensor-memory column 32 a, so the block of source digit b lands on
//    level a + b: the 20 digit pairs in five products;
//  * epilogue warps turn each finished group's six levels into fixed-point
//    updates of the plane, while the next group is multiplied in the other
//    tensor-memory half.
// The source digits of one candidate stay in shared memory for all of its
// items; where a CTA's items pass into the next candidate, the products of
// the last item commit bd_free, the copiers load the next candidate's
// digits and arrive on bd_full, and the products wait for it.
// Handshakes are mbarriers; every wait is bounded.
// (At most 80 registers: 30 K registers, so that a tile solve fits beside
// it; its shared memory admits one per SM.)
template <bool kPacked>
__device__ __forceinline__ void load_source_digits(const QParams& P, TcSmem<kPacked>& sm, const ChunkCand& cc,
                                                   int copier, int ncopiers) {
  const __nv_bfloat16* dp = cc.col ? P.DGt : P.DE;
  const size_t pst = cc.col ? P.dstrideG : P.dstrideE;
  const int ld = cc.col ? P.ldG : P.ldE;
  const int qlim = cc.col ? P.n : P.m, klim = cc.col ? P.m : P.n;
  const int q0 = cc.col ? cc.J * T : cc.I * T;
  for (int e = copier; e < kDigD * T * (CK / 8); e += ncopiers) {
    const int b = e / (T * (CK / 8));
    const int q = (e / (CK / 8)) % T;
    const int k8 = 8 * (e % (CK / 8));
    const int gq = q0 + q, gk = cc.c * CK + k8;
    const bool ok = gq < qlim && gk < klim;
    const __nv_bfloat16* p = dp + (ok ? b * pst + (size_t)gq * ld + gk : 0);
    const int row = b * T + q;  // stacked digit-major
    unsigned char* dst = reinterpret_cast<unsigned char*>(sm.Bd) + (row / 8) * 2048 + (k8 / 8) * 128 + (row % 8) * 16;
    cp_async(dst, p, ok ? 16 : 0, 16);
  }
  cp_async_commit();
}

template <bool kPacked>
__global__ void __maxnreg__(80) chunk_tc_kernel(QParams P, int K, int ncand_col, int ncand, int nitems,
                                                int per_cand) {
  using Shape = TcShape<kPacked>;
  constexpr int NBUF = kDigBufs<kPacked>;
  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  TcSmem<kPacked>& sm = *reinterpret_cast<TcSmem<kPacked>*>(tc_smem_raw);
  const int i0 = (int)(((long long)blockIdx.x * nitems) / gridDim.x);
  const int i1 = (int)(((long long)(blockIdx.x + 1) * nitems) / gridDim.x);
  // the host sizes the grid so that a CTA's share is at most kMaxItems
  const int mygroups = per_cand ? per_cand : min(i1 - i0, kMaxItems);
  if (mygroups <= 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  static_assert(Shape::kWarps >= kTcEpiWarp0 + 4 && kTcCopyWarp < kTcEpiWarp0,
                "warp roles: MMA, copies or producers, 4 epilogue warps");
  // Item map: candidate and group of each of this CTA's items.
  if (tid == 0 && per_cand) {
    // Per candidate: CTA (t, y) takes groups y, y + gridDim.y, ... of
    // candidate t = blockIdx.x (at most per_cand of them).
    ChunkCand c;
    int k = 0;
    if (chunk_candidate(P, K, ncand_col, blockIdx.x, c)) {
      const int ng = (c.ntiles + UC - 1) / UC;
      for (int g = blockIdx.y; g < ng && k < mygroups; g += gridDim.y, ++k) {
        sm.cand[k] = c;
        sm.grp[k] = g;
        sm.seg[k] = 0;
      }
    }
    sm.count = k;
  } else if (tid == 0) {
    int first = 0, k = 0;  // first item index of candidate t
    for (int t = 0; t < ncand && k < mygroups; ++t) {
      ChunkCand c;
      if (!chunk_candidate(P, K, ncand_col, t, c)) continue;
      const int ng = (c.ntiles + UC - 1) / UC;
      for (int g = max(i0 + k - first, 0); g < ng && k < mygroups; ++g, ++k) {
        sm.cand[k] = c;
        sm.grp[k] = g;
        sm.seg[k] = k > 0 ? 1 : 0;
        if (k > 0 && g > 0) sm.seg[k] = 0;
      }
      first += ng;
    }
    sm.count = k;  // equal to mygroups when the host's item count matches the candidates
  }
  __syncthreads();
  const int nitems_cta = sm.count;
  if (nitems_cta <= 0) return;
  const bool is_epi = warp >= kTcEpiWarp0 && warp < kTcEpiWarp0 + 4;
  const bool is_prod = !kPacked && warp != kTcMmaWarp && !is_epi;
  const int ptid = is_prod ? (warp < kTcEpiWarp0 ? tid - 32 : tid - 160) : -1;  // 0 .. kProducers-1
  constexpr int nslab = CK / kSlab;
  const int nz = nitems_cta * nslab;  // slabs of all items, in order
  auto group_row0 = [&](int gi) { return (sm.cand[gi].first + sm.grp[gi] * UC) * T; };
  auto group_rows = [&](int gi) {
    return min(kTcM, (sm.cand[gi].first + sm.cand[gi].ntiles) * T - group_row0(gi));
  };

  // Producer item it (of kTcM * kSlab / 8): row it / 4, columns 8 (it mod 4) .. +7.
  auto copy_slab = [&](int z) {
    if constexpr (!kPacked) {
      if (z < nz) {
        const int gi = z / nslab, s = z % nslab;
        const ChunkCand& cc = sm.cand[gi];
        const float* F = cc.col ? P.LB : P.LA;
        const int d = cc.col ? P.m : P.n;
        const bool vec4 = (d % 4) == 0 && (reinterpret_cast<uintptr_t>(F) & 15) == 0;
        const int row0 = group_row0(gi), rows = group_rows(gi);
        for (int it = ptid; it < kTcM * kSlab / 8; it += Shape::kProducers) {
          const int r = it / 4, k8 = 8 * (it % 4);
          const int gr = row0 + r, gk = cc.c * CK + s * kSlab + k8;
          const bool rok = r < rows && gr < d;
          float* dst = &sm.stage[z % kTcStages][r][k8];
          const float* src = F + (size_t)(rok ? gr : 0) * d;
          if (vec4) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const bool ok = rok && gk + 4 * h < d;
              cp_async(dst + 4 * h, ok ? (const void*)(src + gk + 4 * h) : (const void*)F, ok ? 16 : 0, 16);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const bool ok = rok && gk + e < d;
              cp_async(dst + e, ok ? (const void*)(src + gk + e) : (const void*)F, ok ? 4 : 0, 4);
            }
          }
        }
      }
      cp_async_commit();  // one group per slab, empty past the end, so that the counts stay uniform
    }
  };

  // Prologue: source digits of the first item's candidate (written by the
  // tile solves; by all threads, or by the producers), row exponents,
  // mbarriers, tensor memory; without packed digits also the first two fp32
  // slabs.
  const int copier = kPacked ? tid : ptid;
  const int ncopiers = kPacked ? Shape::kThreads : Shape::kProducers;
  if (copier >= 0) {
    load_source_digits(P, sm, sm.cand[0], copier, ncopiers);
    copy_slab(0);
    copy_slab(1);
  }
  for (int e = tid; e < nitems_cta * kTcM; e += blockDim.x) {
    const int gi = e / kTcM, r = e % kTcM;
    const ChunkCand& cc = sm.cand[gi];
    const int gr = group_row0(gi) + r;
    const int d = cc.col ? P.m : P.n;
    const signed char* fexp = cc.col ? P.expB : P.expA;
    const int nch = cc.col ? P.nchB : P.nchA;
    sm.er[gi][r] = gr < d ? fexp[(size_t)gr * nch + cc.c] : (signed char)-100;
  }
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < NBUF; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(&sm.full[i])),
                   "r"(kPacked ? 1 : Shape::kProducers));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.empty[i])));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.grp_full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;\n" ::"r"(smem_u32(&sm.grp_empty[i])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.bd_free)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(&sm.bd_full)),
                 "r"(kPacked ? 32 : Shape::kProducers));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kTcMmaWarp) {  // two tensor-memory halves of 256 columns (6 levels x 32 used in each)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(&sm.tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  if (copier >= 0) {
    // the source digits (without packed digits slabs 0, 1 may be in flight)
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kPacked ? 0 : 2) : "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int eD = bound_exp(P.hdr->sigma);
  bool broken = false;
  // Source digits of the candidate starting at item gi (gi > 0, sm.seg[gi]):
  // once the products of the previous candidate are done (bd_free, phase
  // nseg - 1), the copiers load them and arrive on bd_full.
  auto next_sources = [&](int gi, uint32_t nseg, int cp, int ncp) {
    mbar_wait(&sm.bd_free, (nseg - 1) & 1u, broken);
    load_source_digits(P, sm, sm.cand[gi], cp, ncp);
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.bd_full)) : "memory");
  };

  if (kPacked ? warp == kTcCopyWarp : is_prod) {
    if constexpr (kPacked) {
      // Slab z of item gi: for each digit a, the group's tiles (at most UC)
      // are contiguous 2 KB blocks of the packed digits: one bulk copy by
      // lane 0.  The whole warp loads the next candidate's source digits.
      uint32_t nseg = 0;
      for (int z = 0; z < nz; ++z) {
        const int p = z % NBUF, gi = z / nslab, s = z % nslab;
        if (s == 0 && sm.seg[gi]) next_sources(gi, ++nseg, lane, 32);
        if (lane == 0) {
          const ChunkCand& cc = sm.cand[gi];
          const __nv_bfloat16* Fd = cc.col ? P.FdB : P.FdA;
          const int nt = cc.col ? P.ntB : P.ntA;
          const int t0 = group_row0(gi) / T;
          const int ntg = min(UC, nt - t0);
          const uint32_t bytes = (uint32_t)ntg * 2048u;
          if (z >= NBUF) mbar_wait(&sm.empty[p], (uint32_t)(z / NBUF - 1) & 1u, broken);
          if (!broken) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(&sm.full[p])),
                         "r"(bytes * kDigF)
                         : "memory");
            const size_t cs = (size_t)cc.c * nslab + s;
#pragma unroll
            for (int a = 0; a < kDigF; ++a) {
              const unsigned char* src =
                  reinterpret_cast<const unsigned char*>(Fd) + ((cs * kDigF + a) * nt + t0) * 2048;
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                      smem_u32(sm.A[p][a])),
                  "l"(src), "r"(bytes), "r"(smem_u32(&sm.full[p]))
                  : "memory");
            }
          }
        }
        __syncwarp();
        if (__shfl_sync(0xffffffffu, broken ? 1 : 0, 0)) break;
      }
    } else {
      uint32_t nseg = 0;
      for (int z = 0; z < nz; ++z) {
        const int p = z % NBUF, gi = z / nslab, s = z % nslab;
        copy_slab(z + 2);
        asm volatile("cp.async.wait_group 2;\n" ::: "memory");  // this thread's items of slab z
        if (z >= NBUF) mbar_wait(&sm.empty[p], (uint32_t)(z / NBUF - 1) & 1u, broken);
        if (s == 0 && sm.seg[gi]) next_sources(gi, ++nseg, ptid, Shape::kProducers);
        for (int it = ptid; it < kTcM * kSlab / 8; it += Shape::kProducers) {
          const int r = it / 4, k8 = 8 * (it % 4);
          const float sc = pow2f(7 - sm.er[gi][r]);
          const float4 x0 = *reinterpret_cast<const float4*>(&sm.stage[z % kTcStages][r][k8]);
          const float4 x1 = *reinterpret_cast<const float4*>(&sm.stage[z % kTcStages][r][k8 + 4]);
          float u[8] = {x0.x * sc, x0.y * sc, x0.z * sc, x0.w * sc, x1.x * sc, x1.y * sc, x1.z * sc, x1.w * sc};
          const int off = (r / 8) * 512 + (k8 / 8) * 128 + (r % 8) * 16;
#pragma unroll
          for (int a = 0; a < kDigF; ++a) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              // The same digit split as factor_digits_kernel (round to the
              // nearest integer by adding and subtracting 1.5 * 2^23, bf16
              // pattern = the fp32 pattern's upper half, two per word).
              const float d0 = (u[2 * e] + 0x1.8p23f) - 0x1.8p23f;
              const float d1 = (u[2 * e + 1] + 0x1.8p23f) - 0x1.8p23f;
              w[e] = __byte_perm(__float_as_uint(d0), __float_as_uint(d1), 0x7632);
              u[2 * e] = (u[2 * e] - d0) * 256.f;
              u[2 * e + 1] = (u[2 * e + 1] - d1) * 256.f;
            }
            *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(sm.A[p][a]) + off) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.full[p])) : "memory");
      }
    }
  } else if (warp == kTcMmaWarp) {
    if (lane == 0) {
      uint32_t nseg = 0;
      for (int z = 0; z < nz; ++z) {
        const int p = z % NBUF, gi = z / nslab, s = z % nslab, h = gi & 1;
        if (s == 0 && gi >= 2) mbar_wait(&sm.grp_empty[h], (uint32_t)((gi >> 1) - 1) & 1u, broken);
        if (s == 0 && sm.seg[gi]) mbar_wait(&sm.bd_full, nseg++ & 1u, broken);
        mbar_wait(&sm.full[p], (uint32_t)(z / NBUF) & 1u, broken);
        if (broken) break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < kSlab / 16; ++j) {
          const uint64_t db = umma_sdesc(smem_u32(sm.Bd) + (uint32_t)((s * kSlab + 16 * j) / 8) * 128u, 128u, 2048u);
#pragma unroll
          for (int a = 0; a < kDigF; ++a) {
            const uint64_t da = umma_sdesc(smem_u32(sm.A[p][a]) + (uint32_t)(2 * j) * 128u, 128u, 512u);
            const uint32_t acc = (s > 0 || j > 0 || a > 0) ? 1u : 0u;
            umma_bf16(tmem + (uint32_t)(256 * h + 32 * a), da, db, umma_idesc_bf16(kTcM, T * (kDigD - a)), acc);
          }
        }
        umma_commit(&sm.empty[p]);
        if (s == nslab - 1) {
          umma_commit(&sm.grp_full[h]);
          if (gi + 1 < nitems_cta && sm.seg[gi + 1]) umma_commit(&sm.bd_free);
        }
      }
    }
    __syncwarp();
  } else if (warp >= kTcEpiWarp0 && warp < kTcEpiWarp0 + 4) {  // epilogue warps
    const int qd = warp - kTcEpiWarp0;  // tensor-memory lane quarter
    const int r = 32 * qd + lane;       // output row of this thread within the group
    for (int gi = 0; gi < nitems_cta; ++gi) {
      const int h = gi & 1;
      mbar_wait(&sm.grp_full[h], (uint32_t)(gi >> 1) & 1u, broken);
      tc_fence_after();
      const ChunkCand& cc = sm.cand[gi];
      const int row0 = group_row0(gi), rows = group_rows(gi);
      // levels -> value: 2^(e_r + eD - 14); value -> fixed-point units: 2^-unit_exp
      const int ex = sm.er[gi][r] + eD - 14 - fixed_unit_exp(P.hdr->sigma);
      const float sc = ex >= -126 ? pow2f(min(ex, 127)) : 0.f;
      // Output (row r, column q) of the group: column products update
      // Xc[row0 + r][J*T + q], row products Gc[I*T + q][row0 + r], each as
      // one 64-bit integer reduction in L2 (red.global.add.u64: no load, no
      // wait) of the fixed-point value (see fixed_unit_exp).
      unsigned long long* plane = reinterpret_cast<unsigned long long*>(cc.col ? P.Xc : P.Gc);
      const int gr0 = cc.col ? row0 + r : cc.I * T, gc0 = cc.col ? cc.J * T : row0 + r;
      const bool rok = r < rows && (cc.col ? gr0 < P.m : gc0 < P.n);
      const size_t obase = rok ? (size_t)gr0 * P.n + gc0 : 0;
      const size_t ostep = cc.col ? 1 : (size_t)P.n;  // next q
      const int qlim = cc.col ? P.n - gc0 : P.m - gr0;
#pragma unroll 1
      for (int qb = 0; qb < T; qb += kEpiCols) {
        float lv[kLevels][kEpiCols];
#pragma unroll
        for (int l = 0; l < kLevels; ++l)
          tmem_ld(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(256 * h + 32 * l + qb), lv[l]);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) {
          // levels 0..2 exactly (each an integer sum below 2^24 on its own
          // grid), the rest (below 2^-24 of the total) in one fp32 sum
          float2 y = two_sum(lv[0][j], lv[1][j] * 0x1p-8f);
          const float2 y2 = two_sum(y.y, lv[2][j] * 0x1p-16f);
          const float tail = lv[3][j] * 0x1p-24f + lv[4][j] * 0x1p-32f + lv[5][j] * 0x1p-40f;
          y = two_sum(y.x, y2.x);  // any level may be zero: no ordering of magnitudes holds
          y = two_sum(y.x, y.y + (y2.y + tail));
          if (rok && qb + j < qlim)
            atomicAdd(plane + obase + (size_t)(qb + j) * ostep, (unsigned long long)df_to_fixed(y, sc));
        }
      }
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.grp_empty[h])) : "memory");
    }
  }
  if (broken) atomicOr(P.status, BAKRON_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem));
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

// The side streams (mid pushes; chunk products) and the ordering events,
// one set per device, reused by every call.  Streams and events are driver objects, not device memory.
// Calls that share a set serialize their side work on its streams, which
// is correct: each call's main stream waits only on its own events' records.
// Dynamic shared memory: a mid push CTA holds one stage; a chunk product
// CTA the source digits, three factor digit slabs with packed digits, or
// two and three fp32 factor slabs when it makes the digits itself (about
// 175 KB either way: one per SM, with room beside it for a tile solve).
constexpr int kMidSmem = (int)sizeof(PushSmem<1>);
template <bool kPacked>
constexpr int kChunkSmem = (int)sizeof(TcSmem<kPacked>);
// A tile solve (43008 bytes of static shared memory) must fit beside one
// chunk product CTA on an SM (228 KB, 1 KB reserved per CTA): the solve
// chain would otherwise wait for whole chunk CTAs to finish before each of
// its launches.
static_assert(sizeof(TcSmem<false>) + 43008 + 2048 <= 228 * 1024 &&
                  sizeof(TcSmem<true>) + 43008 + 2048 <= 228 * 1024,
              "a tile solve must fit beside a chunk product CTA");

// Chunk launches of consecutive tile anti-diagonals go round-robin over
// kChunkStreams streams.  With more than one they overlap and may update
// the same plane elements, which the 64-bit integer reductions keep exact in
// any order; one stream is the default (more were not faster when measured,
// with the earlier floating-point reductions: 19.0 against 19.3 ms on a
// 4096 x 4096 layer, 95.4 against 91.4 ms on 14336 x 4096).
constexpr int kChunkStreams = 1;

struct StreamSet {
  bool ready = false;
  unsigned long long ctx_id = 0;  // context the streams and events belong to
  cudaStream_t solve = nullptr, mid = nullptr, mid_low = nullptr, chunk[kChunkStreams] = {};
  int sms = 0;  // multiprocessors of the device
  std::vector<cudaEvent_t> ev;
};
constexpr int kMaxDevices = 128;
StreamSet g_sets[kMaxDevices];
std::mutex g_set_mutex;

cudaError_t prepare_set(StreamSet& S, size_t nev) {
  unsigned long long ctx = 0;
  cudaError_t e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  if (S.ready && S.ctx_id != ctx) S = StreamSet();  // the old context (and its handles) is gone
  if (!S.ready) {
    S.ctx_id = ctx;
    int lo = 0, hi = 0;
    e = cudaDeviceGetStreamPriorityRange(&lo, &hi);  // hi is the most urgent (numerically lowest)
    if (e != cudaSuccess) return e;
    // The chunk stream gets the highest priority: the chunk products are
    // the largest block of work and their stream sets the pace (measured on
    // 4096 x 4096: 23.3 ms with the chunk stream at the lowest priority, 22.6 ms
    // here).  The mid pushes run on a stream of either priority (see
    // quantize_launch).
    e = cudaStreamCreateWithPriority(&S.solve, cudaStreamNonBlocking, hi);
    if (e != cudaSuccess) return e;
    e = cudaStreamCreateWithPriority(&S.mid, cudaStreamNonBlocking, hi);
    if (e != cudaSuccess) return e;
    e = cudaStreamCreateWithPriority(&S.mid_low, cudaStreamNonBlocking, lo);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < kChunkStreams; ++i) {
      e = cudaStreamCreateWithPriority(&S.chunk[i], cudaStreamNonBlocking, hi);
      if (e != cudaSuccess) return e;
    }
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&S.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chunk_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kChunkSmem<false>);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chunk_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kChunkSmem<true>);
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

// Workspace: header, the six planes, the factor exponents, the source
// digits of E and G.
struct WsLayout {
  size_t plane, expA, expB, DE, DG, dplaneE, dplaneG, FdA, FdB, total;
  int ldE, ldG;
};
WsLayout ws_layout(int64_t m, int64_t n) {
  WsLayout L;
  const size_t nchA = (size_t)((n + CK - 1) / CK), nchB = (size_t)((m + CK - 1) / CK);
  L.plane = align_up((size_t)m * (size_t)n * sizeof(float2));
  size_t off = sizeof(Header) + kPlanes * L.plane;
  L.expA = off;
  off += align_up((size_t)n * nchA);
  L.expB = off;
  off += align_up((size_t)m * nchB);
  L.ldE = (int)((n + 7) / 8 * 8);
  L.ldG = (int)((m + 7) / 8 * 8);
  L.dplaneE = align_up((size_t)m * L.ldE * sizeof(__nv_bfloat16));
  L.dplaneG = align_up((size_t)n * L.ldG * sizeof(__nv_bfloat16));
  L.DE = off;
  off += kDigD * L.dplaneE;
  L.DG = off;
  off += kDigD * L.dplaneG;
  // packed factor digits (layers above 2^24 weights): nch chunks x
  // (CK / kSlab) slabs x kDigF digits x nt tiles x 2 KB per factor
  const bool packed = use_packed_digits(m, n);
  const size_t ntA = (size_t)((n + T - 1) / T), ntB = (size_t)((m + T - 1) / T);
  L.FdA = off;
  if (packed) off += align_up(nchA * (CK / kSlab) * kDigF * ntA * 2048);
  L.FdB = off;
  if (packed) off += align_up(nchB * (CK / kSlab) * kDigF * ntB * 2048);
  L.total = off;
  return L;
}

size_t quantize_workspace_bytes(int64_t m, int64_t n) {
  return std::max(ws_layout(m, n).total, sweep_workspace_bytes(m, n));
}

cudaError_t quantize_launch(const float* W, const float* LA, const float* LB, Scales sc,
                            Alphabet al, int m, int n, int32_t* V, float* Wq, void* ws,
                            int32_t* status_dev, cudaStream_t stream, KernelTimer* timer) {
  const WsLayout lay = ws_layout(m, n);
  const bool packed = use_packed_digits(m, n);
  const size_t plane = lay.plane;
  char* base = static_cast<char*>(ws);
  float2* planes = reinterpret_cast<float2*>(base + sizeof(Header));
  const size_t pstride = plane / sizeof(float2);
  QParams P;
  P.W = W;
  P.LA = LA;
  P.LB = LB;
  P.scales = sc.R;
  P.cscales = sc.t;
  P.group = (sc.group <= 0 || sc.group > n) ? n : sc.group;
  P.ngroups = (n + P.group - 1) / P.group;
  P.V = V;
  P.Wq = Wq;
  P.hdr = reinterpret_cast<Header*>(base);
  P.Xm = planes;
  P.Xc = reinterpret_cast<long long*>(planes + pstride);
  P.Gm = planes + 2 * pstride;
  P.Gc = reinterpret_cast<long long*>(planes + 3 * pstride);
  P.G = planes + 4 * pstride;
  P.E = planes + 5 * pstride;
  P.status = status_dev;
  P.expA = reinterpret_cast<const signed char*>(base + lay.expA);
  P.expB = reinterpret_cast<const signed char*>(base + lay.expB);
  P.DE = reinterpret_cast<__nv_bfloat16*>(base + lay.DE);
  P.DGt = reinterpret_cast<__nv_bfloat16*>(base + lay.DG);
  P.dstrideE = lay.dplaneE / sizeof(__nv_bfloat16);
  P.dstrideG = lay.dplaneG / sizeof(__nv_bfloat16);
  P.ldE = lay.ldE;
  P.ldG = lay.ldG;
  P.nchA = (n + CK - 1) / CK;
  P.nchB = (m + CK - 1) / CK;
  P.ntA = (n + T - 1) / T;
  P.ntB = (m + T - 1) / T;
  P.skew = LB ? 1 : 0;
  P.FdA = reinterpret_cast<const __nv_bfloat16*>(base + lay.FdA);
  P.FdB = reinterpret_cast<const __nv_bfloat16*>(base + lay.FdB);
  P.m = m;
  P.n = n;
  P.Mt = (m + T - 1) / T;
  P.Nt = (n + T - 1) / T;
  P.bits = al.bounded ? 1 : 0;  // 1: the codes are clamped to {lo .. hi}
  P.lo = al.lo;
  P.hi = al.hi;
  const int Kmax = P.skew ? P.Mt + P.Nt - 2 : P.Nt - 1;

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
  // Mid pushes at the lowest priority from 2^22 weights on, so that the
  // block scheduler places a pending tile solve's CTAs before theirs
  // (measured on one GB300, 4096 x 4096: 13.6 against 14.0 ms, row-wise
  // GPTQ 7.11 against 7.24 ms; 14336 x 4096 and 4096 x 14336 the same
  // either way); at the highest on smaller layers, where they are on the
  // chain's critical path (1024 x 1024: 2.35 against 2.41 ms).
  cudaStream_t s_mid = timer ? stream : (use_packed_digits(m, n) ? S.mid_low : S.mid);
  // Layers up to 2^24 weights: the tile solves run on a stream of the
  // highest priority, beside the products (measured on 4096 x 4096: 15.9
  // against 16.6 ms); on larger layers the products set the pace, and the
  // solves stay on the caller's stream (measured on 14336 x 4096: 66.7
  // against 80.9 ms).
  cudaStream_t s_solve = (timer || large_layer(m, n)) ? stream : S.solve;
  auto s_chunk = [&](int K) { return timer ? stream : S.chunk[K % kChunkStreams]; };

  LaunchClock clock(timer);
  err = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(P.hdr, 0, sizeof(Header), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(planes, 0, 4 * plane, stream);  // Xm, Xc, Gm, Gc
  // Digit rows are padded to a multiple of 8 entries; the chunk products
  // read the padding, which must then be zero.
  if (err == cudaSuccess && (lay.ldE != n || lay.ldG != m))
    err = cudaMemsetAsync(base + lay.DE, 0, kDigD * (lay.dplaneE + lay.dplaneG), stream);
  if (err != cudaSuccess) return err;
  const size_t total = (size_t)m * n;
  const int pre_blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 8);
  const InputDesc in{W, P.scales, P.cscales, P.ngroups, m, n, P.bits, P.lo, P.hi, P.hdr, status_dev};
  clock.begin(0, stream);
  prepass_kernel<<<pre_blocks, 256, 0, stream>>>(in);
  sigma_kernel<<<1, 1, 0, stream>>>(in);
  {
    signed char* eA = reinterpret_cast<signed char*>(base + lay.expA);
    signed char* eB = reinterpret_cast<signed char*>(base + lay.expB);
    const size_t wA = (size_t)n * P.nchA, wB = (size_t)m * P.nchB;  // one warp per (row, chunk)
    factor_exp_kernel<<<(unsigned)((wA + 7) / 8), 256, 0, stream>>>(LA, n, P.nchA, eA);
    if (LB) factor_exp_kernel<<<(unsigned)((wB + 7) / 8), 256, 0, stream>>>(LB, m, P.nchB, eB);
    if (packed) {  // the factors' digits, once per solve, for the chunk products' bulk copies
      const int digit_blocks = 152 * 8;
      factor_digits_kernel<<<digit_blocks, 256, 0, stream>>>(LA, n, P.nchA, P.ntA, eA,
                                                             const_cast<__nv_bfloat16*>(P.FdA));
      if (LB)
        factor_digits_kernel<<<digit_blocks, 256, 0, stream>>>(LB, m, P.nchB, P.ntB, eB,
                                                               const_cast<__nv_bfloat16*>(P.FdB));
    }
  }
  clock.end(0.0);
  cudaEventRecord(ev_start, stream);
  cudaStreamWaitEvent(s_mid, ev_start, 0);
  for (int i = 0; i < kChunkStreams; ++i) cudaStreamWaitEvent(s_chunk(i), ev_start, 0);
  if (s_solve != stream) cudaStreamWaitEvent(s_solve, ev_start, 0);

  const double t3 = (double)T * T * T;
  std::vector<char> mid_on(Kmax + 1, 0), chunk_on(Kmax + 1, 0);
  int last_mid = -1;
  int last_chunk[kChunkStreams];
  for (int i = 0; i < kChunkStreams; ++i) last_chunk[i] = -1;
  for (int K = 0; K <= Kmax; ++K) {
    const int I0 = P.skew ? std::max(0, K - (P.Nt - 1)) : 0;
    const int I1 = P.skew ? std::min(K, P.Mt - 1) : P.Mt - 1;
    const int nsrc = I1 - I0 + 1;
    if (K >= 2 && mid_on[K - 2]) cudaStreamWaitEvent(s_solve, ev_mid[K - 2], 0);
    // One wait each is enough: mid(K-2) follows every earlier mid launch on
    // its stream, every chunk launch before chunk(K-B-1) was waited for by an
    // earlier solve (the solves are in order on one stream), and a missing
    // launch was covered by the wait of an earlier solve.
    if (K >= B + 1 && chunk_on[K - B - 1]) cudaStreamWaitEvent(s_solve, ev_chunk[K - B - 1], 0);
    clock.begin(1, s_solve);
    if (large_layer(m, n))
      tile_solve_kernel<512><<<nsrc, 512, 0, s_solve>>>(P, K, I0);
    else
      tile_solve_kernel<1024><<<nsrc, 1024, 0, s_solve>>>(P, K, I0);
    clock.end(2.0 * 3.5 * t3 * nsrc);  // in-tile sums, L_B[I,I] row part, two distance-1 pulls
    cudaEventRecord(ev_solve[K], s_solve);

    // mid pushes from the sources of K
    double mid_tiles = 0;
    for (int I = I0; I <= I1; ++I) {
      const int J = K - P.skew * I;
      if (LB) mid_tiles += std::max(0, std::min(P.Mt, mid_end(I)) - (I + 2));
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

    // chunk products closed by K, and their items (target groups)
    int ncc = 0, ncr = 0;
    chunk_counts(P, K, LB != nullptr, ncc, ncr);
    double chunk_tiles = 0;
    int nitems = 0, most = 0;  // items (target groups) in all; most of one candidate
    for (int t = 0; t < ncc + ncr; ++t) {
      ChunkCand cc;
      if (!chunk_candidate(P, K, ncc, t, cc)) continue;
      chunk_tiles += cc.ntiles;
      nitems += (cc.ntiles + UC - 1) / UC;
      most = std::max(most, (cc.ntiles + UC - 1) / UC);
    }
    if (chunk_tiles > 0) {
      cudaStreamWaitEvent(s_chunk(K), ev_solve[K], 0);
      clock.begin(3, s_chunk(K));
      if (large_layer(m, n)) {
        // Each CTA serves one candidate, at most kItemsPerCand of its groups.
        const int ctas = (most + kItemsPerCand - 1) / kItemsPerCand;
        if (packed)
          chunk_tc_kernel<true><<<dim3(ncc + ncr, ctas), TcShape<true>::kThreads, kChunkSmem<true>, s_chunk(K)>>>(
              P, K, ncc, ncc + ncr, nitems, kItemsPerCand);
        else
          chunk_tc_kernel<false><<<dim3(ncc + ncr, ctas), TcShape<false>::kThreads, kChunkSmem<false>, s_chunk(K)>>>(
              P, K, ncc, ncc + ncr, nitems, kItemsPerCand);
      } else {
        // The launch's items shared evenly: small launches over at most
        // five eighths of the SMs (one CTA each), so that the next tile
        // solves find SMs without a chunk product CTA; large ones in whole
        // waves of one CTA per SM; at most kMaxItems items per CTA.
        // Measured on 4096 x 4096 (mid pushes at the lowest priority):
        // 13.51 ms at 5/8, 13.60 at 3/4, 13.77 at 7/8; 9/16 and 11/16 (with
        // mid pushes at the highest priority) were between 5/8 and 3/4.
        const int cap = std::max(1, S.sms * 5 / 8);
        int ctas = std::min(nitems, cap);
        if (nitems > cap * kMaxItems) {
          const int waves = (nitems + S.sms * kMaxItems - 1) / (S.sms * kMaxItems);
          ctas = std::min(nitems, S.sms * waves);
        }
        if (packed)
          chunk_tc_kernel<true><<<ctas, TcShape<true>::kThreads, kChunkSmem<true>, s_chunk(K)>>>(
              P, K, ncc, ncc + ncr, nitems, 0);
        else
          chunk_tc_kernel<false><<<ctas, TcShape<false>::kThreads, kChunkSmem<false>, s_chunk(K)>>>(
              P, K, ncc, ncc + ncr, nitems, 0);
      }
      clock.end(2.0 * B * t3 * chunk_tiles);
      cudaEventRecord(ev_chunk[K], s_chunk(K));
      chunk_on[K] = 1;
      last_chunk[K % kChunkStreams] = K;
    }
  }
  // Join: the caller's stream covers all side work of this call.
  if (s_solve != stream) cudaStreamWaitEvent(stream, ev_solve[Kmax], 0);
  if (last_mid >= 0) cudaStreamWaitEvent(stream, ev_mid[last_mid], 0);
  for (int i = 0; i < kChunkStreams; ++i)
    if (last_chunk[i] >= 0) cudaStreamWaitEvent(stream, ev_chunk[last_chunk[i]], 0);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return clock.finish(stream);
}

// Host-only check of the launch schedule above, from the same pieces
// (step numbering, mid_end and mid_push_kernel's target ranges,
// chunk_counts and chunk_candidate).  Along every tile column (column
// terms, when L_B is given) and every tile row (row terms), each pair of a
// source tile s and a later target tile t must be carried exactly once: by
// the target's own solve (t = s + 1, the distance-1 pulls), by a mid push
// or by a chunk product.  A mid push launched after step K reaches its
// targets when the solve of step K + 2 waits for it; a chunk product when
// the solve of step K + lag does (quantize_launch: lag = B + 1); the mid
// and chunk streams each run their launches in order.  Every source must be
// solved by the step after which its push is launched, every tile solved
// exactly once, and mid_push_kernel's grid must reach every target group.
// stats: [0] pushes and pulls recorded, [1] the smallest number of steps
// between a chunk product's launch and its first target's solve (-1 if
// there is none), [2] errors.  Returns 0 when there are none.
int wavefront_plan_check(int64_t m, int64_t n, bool colpush, int lag, int64_t* stats) {
  QParams P{};
  P.Mt = (int)((m + T - 1) / T);
  P.Nt = (int)((n + T - 1) / T);
  P.skew = colpush ? 1 : 0;
  const int Kmax = P.skew ? P.Mt + P.Nt - 2 : P.Nt - 1;
  auto step_of = [&](int I, int J) { return J + P.skew * I; };
  struct Rec {
    bool col;  // column terms (line = tile column J, indices = tile rows), else row terms
    int line, s0, s1, t0, t1, K, kind;  // kind 0: pull, 1: mid push, 2: chunk product
  };
  std::vector<Rec> recs;
  int64_t errors = 0;
  std::vector<int> solved((size_t)P.Mt * P.Nt, -1);
  const int units = 2 * ((2 * B - 2 + U - 1) / U);  // mid_push_kernel's grid.y
  for (int K = 0; K <= Kmax; ++K) {
    const int I0 = P.skew ? std::max(0, K - (P.Nt - 1)) : 0;
    const int I1 = P.skew ? std::min(K, P.Mt - 1) : P.Mt - 1;
    for (int I = I0; I <= I1; ++I) {
      const int J = K - P.skew * I;
      if (J < 0 || J >= P.Nt) {
        ++errors;
        continue;
      }
      if (solved[(size_t)I * P.Nt + J] >= 0) ++errors;
      solved[(size_t)I * P.Nt + J] = K;
      if (colpush && I > 0) recs.push_back({true, J, I - 1, I, I, I + 1, K, 0});
      if (J > 0) recs.push_back({false, I, J - 1, J, J, J + 1, K, 0});
      const int c_first = I + 2, c_end = colpush ? std::min(P.Mt, mid_end(I)) : c_first;
      const int r_first = J + 2, r_end = std::min(P.Nt, mid_end(J));
      const int ncu = c_end > c_first ? (c_end - c_first + U - 1) / U : 0;
      const int nru = r_end > r_first ? (r_end - r_first + U - 1) / U : 0;
      if (ncu + nru > units) ++errors;
      if (c_end > c_first) recs.push_back({true, J, I, I + 1, c_first, c_end, K, 1});
      if (r_end > r_first) recs.push_back({false, I, J, J + 1, r_first, r_end, K, 1});
    }
    int ncc = 0, ncr = 0;
    chunk_counts(P, K, colpush, ncc, ncr);
    for (int t = 0; t < ncc + ncr; ++t) {
      ChunkCand cc;
      if (!chunk_candidate(P, K, ncc, t, cc)) continue;
      const int len = cc.col ? P.Mt : P.Nt;
      recs.push_back({cc.col, cc.col ? cc.J : cc.I, cc.c * B, std::min((cc.c + 1) * B, len), cc.first,
                      cc.first + cc.ntiles, K, 2});
    }
  }
  for (int v : solved)
    if (v < 0) ++errors;
  int64_t min_slack = -1;
  for (int dir = 0; dir < 2; ++dir) {
    const bool col = dir == 0;
    if (col && !colpush) {
      for (const Rec& r : recs)
        if (r.col) ++errors;
      continue;
    }
    const int nlines = col ? P.Nt : P.Mt, len = col ? P.Mt : P.Nt;
    std::vector<std::vector<const Rec*>> by_line(nlines);
    for (const Rec& r : recs)
      if (r.col == col) {
        if (r.line < 0 || r.line >= nlines) {
          ++errors;
          continue;
        }
        by_line[r.line].push_back(&r);
      }
    std::vector<int> cnt((size_t)len * len);
    for (int line = 0; line < nlines; ++line) {
      std::fill(cnt.begin(), cnt.end(), 0);
      for (const Rec* r : by_line[line]) {
        if (r->s0 < 0 || r->s1 > len || r->t0 < 0 || r->t1 > len) {
          ++errors;
          continue;
        }
        for (int s = r->s0; s < r->s1; ++s) {
          const int src_step = col ? step_of(s, line) : step_of(line, s);
          if (r->kind == 0 ? src_step >= r->K : src_step > r->K) ++errors;  // source not solved in time
          for (int t = r->t0; t < r->t1; ++t) {
            if (t <= s) {
              ++errors;
              continue;
            }
            ++cnt[(size_t)s * len + t];
            const int tgt_step = col ? step_of(t, line) : step_of(line, t);
            const int need = r->kind == 0 ? 0 : (r->kind == 1 ? 2 : lag);
            if (r->kind == 0 ? tgt_step != r->K : tgt_step < r->K + need) ++errors;
            if (r->kind == 2 && (min_slack < 0 || tgt_step - r->K < min_slack)) min_slack = tgt_step - r->K;
          }
        }
      }
      for (int s = 0; s < len; ++s)
        for (int t = s + 1; t < len; ++t)
          if (cnt[(size_t)s * len + t] != 1) ++errors;
    }
  }
  stats[0] = (int64_t)recs.size();
  stats[1] = min_slack;
  stats[2] = errors;
  return errors == 0 ? 0 : 1;
}

}  // namespace bakron
