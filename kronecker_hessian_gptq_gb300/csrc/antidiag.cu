// antidiag.cu -- BaKron-antidiagonal on the GPU ("BaKron: Efficient
// Quantization with Kronecker-Factored Hessians", Sec. 3.2, Algorithm 3; the
// BaKron-antidiag. column of Table 3).  The anti-diagonals of W are rounded
// one after another; after each, the errors Delta of the whole anti-diagonal
// update every later entry at once,
//     W~ += L_B Delta L_A^T      (Delta nonzero on one anti-diagonal),
// i.e. entry (p, q) gains sum_i L_B[p, i] Delta_i L_A[q, k - i] over the
// entries (i, k - i) of anti-diagonal k with i <= p and k - i <= q.  That is
// (p + 1)(q + 1) - 1 multiply-adds per entry over the whole run, about
// m^2 n^2 / 4 in all (the quartic cost of Sec. 3.2), against m + n - 1
// sequential steps.  By Theorem 3.2 the codes equal BaKron's.
//
// Layout: W~ is double-float (the precision of the BaKron solve, so that
// both reproduce the oracle's codes).  Launch k updates every later entry
// tile by tile and, in the same pass, rounds the entries of anti-diagonal
// k + 1 (whose update is then complete) and publishes their errors for
// launch k + 1.  An output tile of 32 x 32 stages M[p, i] = L_B[p, i] Delta_i
// (double-float) and L_A[q, k - i] for 32 diagonal entries at a time in
// shared memory, the next chunk's operands loaded into registers while the
// current one is multiplied; each thread accumulates a 2 x 4 block (2 x 2
// on layers of up to 2^21 weights) with offset accumulators (5 fp32
// instructions per multiply-add).  Small tiles keep the longest tile short:
// within one launch the tile nearest the end has the most terms, up to the
// anti-diagonal's length.
#include <algorithm>

#include "bakron.h"
#include "df.cuh"
#include "internal.h"

namespace bakron {
namespace {

constexpr int kAdT = 32;         // output tile edge
constexpr int kAdKC = 32;        // diagonal entries per shared-memory stage
constexpr int kAdRM = 2;         // rows per thread
// Columns per thread RN: 4 (128 threads, two 16-byte shared loads per 8
// multiply-adds) for large layers, where throughput counts; 2 (256 threads,
// half the work per thread) for small ones, where the tile with the most
// terms sets the time of each launch.
template <int RN>
struct AdShape {
  static constexpr int kThreads = (kAdT / kAdRM) * (kAdT / RN);
  static constexpr int kSlots = kAdKC * kAdT / kThreads;  // staging slots per thread
};
constexpr int kAdPadM = kAdT + 2;  // row strides: 16-byte rows for vector loads
constexpr int kAdPadL = kAdT + 4;

struct AdParams {
  const float* W;
  const float* LA;
  const float* LB;
  const float* scales;
  int32_t* V;
  float* Wq;
  float2* Wt;  // W~, m x n double-float
  float2* D;   // errors of two consecutive anti-diagonals, 2 x m, indexed by row
  int32_t* status;
  int m, n, bounded, lo, hi;
};

// Checks the inputs and sets W~ = W.
__global__ void ad_prepass_kernel(AdParams P) {
  const size_t total = (size_t)P.m * P.n;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  int bad = 0;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const float w = P.W[idx];
    if (!isfinite(w)) bad |= BAKRON_DEV_NONFINITE_W;
    P.Wt[idx] = make_float2(w, 0.f);
  }
  if (P.scales) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)P.m; i += stride) {
      const float s = P.scales[i];
      if (!(s > 0.f) || !isfinite(s)) bad |= BAKRON_DEV_BAD_SCALE;
    }
  }
  if (bad) atomicOr(P.status, bad);
}

// Rounds entry (p, q) holding x = W~[p, q]: the fp32 decision of the BaKron
// solve (x.x * (1/s) within 2 ulp of the correctly rounded quotient, which is
// taken near a tie or for a large or non-finite product), the error
// Delta = s v - x in double-float.
__device__ __forceinline__ void ad_round(const AdParams& P, int p, int q, float2 x, float2* Dn) {
  const float s = P.scales ? P.scales[p] : 1.f;
  float y = x.x * __frcp_rn(s);
  if (!(fabsf(y) <= 256.f) || fabsf(y - floorf(y) - 0.5f) < 1e-3f) y = __fdiv_rn(x.x, s);
  float v = rintf(y);
  if (P.bounded) v = fminf(fmaxf(v, (float)P.lo), (float)P.hi);
  const float2 sv = two_prod(s, v);
  const float2 h = two_sum(sv.x, -x.x);
  Dn[p] = fast_two_sum(h.x, (sv.y - x.y) + h.y);
  const size_t o = (size_t)p * P.n + q;
  P.V[o] = (int32_t)v;
  P.Wq[o] = s * v;
}

// Raw operands of a thread's staging slots (diagonal entry kk, tile rows and
// columns r): L_B[p, i] (1 on the diagonal, 0 where p < i or outside),
// L_A[q, k - i] (likewise), and Delta_i -- one kk per thread, so one Delta.
// Loaded a chunk ahead into registers.
template <int RN>
struct AdSlot {
  static_assert(AdShape<RN>::kThreads % kAdKC == 0, "a thread's slots share one diagonal entry");
  float l[AdShape<RN>::kSlots];
  float a[AdShape<RN>::kSlots];
  float2 d;
};

template <int RN>
__device__ __forceinline__ void ad_load(const AdParams& P, const float2* D, int k, int ib, int i1, int P0, int Q0,
                                        AdSlot<RN>& st) {
  constexpr int kAdThreads = AdShape<RN>::kThreads, kAdSlots = AdShape<RN>::kSlots;
  const int kk = threadIdx.x % kAdKC;
  const int i = ib + kk, j = k - i;
  const bool vi = i <= i1;
  st.d = vi ? D[i] : make_float2(0.f, 0.f);
#pragma unroll
  for (int s = 0; s < kAdSlots; ++s) {
    const int r = (threadIdx.x + s * kAdThreads) / kAdKC;
    const int p = P0 + r, q = Q0 + r;
    st.l[s] = (vi && p < P.m && i <= p) ? (i == p ? 1.f : P.LB[(size_t)p * P.m + i]) : 0.f;
    st.a[s] = (vi && q < P.n && j <= q) ? (j == q ? 1.f : P.LA[(size_t)q * P.n + j]) : 0.f;
  }
}

// Launch k (k = -1 .. m + n - 3): the update from anti-diagonal k (none for
// k = -1), then the rounding of anti-diagonal k + 1.
template <int RN>
__global__ void __launch_bounds__(AdShape<RN>::kThreads, 512 / AdShape<RN>::kThreads) ad_step_kernel(AdParams P,
                                                                                                      int k) {
  constexpr int kAdRN = RN, kAdThreads = AdShape<RN>::kThreads, kAdSlots = AdShape<RN>::kSlots;
  const int P0 = blockIdx.y * kAdT, Q0 = blockIdx.x * kAdT;
  const int pmax = min(P0 + kAdT, P.m) - 1, qmax = min(Q0 + kAdT, P.n) - 1;
  if (pmax + qmax <= k) return;  // every entry of the tile is rounded
  const int ilo = max(0, k - P.n + 1), ihi = min(k, P.m - 1);  // rows of anti-diagonal k
  const int i0 = max(ilo, k - qmax), i1 = min(ihi, pmax);     // those with a term in this tile
  const bool has_next = P0 + Q0 <= k + 1;                      // an entry of anti-diagonal k + 1
  if (i0 > i1 && !has_next) return;
  const float2* D = P.D + (size_t)((k + 2) & 1) * P.m;
  float2* Dn = P.D + (size_t)((k + 3) & 1) * P.m;

  __shared__ __align__(16) float2 sM[kAdKC][kAdPadM];  // L_B[p, i] Delta_i
  __shared__ __align__(16) float sL[kAdKC][kAdPadL];   // L_A[q, k - i]
  __shared__ float sMax[2][kAdThreads / 32];           // per-warp max |M|, max |L_A| of the chunk
  const int tr = threadIdx.x / (kAdT / kAdRN), tc = threadIdx.x % (kAdT / kAdRN);  // rows 2 tr.., columns RN tc..
  // Each chunk of at most kAdKC terms is summed by offset accumulators on an
  // offset of its own, from the chunk's largest operands, and folded into a
  // double-float total: the rounding error then scales with the terms
  // actually added, not with the weights (over m + n steps of updates an
  // error of 2^-48 of the weights' offset per term would flip codes).
  OffsetAcc acc[kAdRM][kAdRN];
  float2 tot[kAdRM][kAdRN];
#pragma unroll
  for (int a = 0; a < kAdRM; ++a)
#pragma unroll
    for (int b = 0; b < kAdRN; ++b) tot[a][b] = make_float2(0.f, 0.f);

  AdSlot<RN> st;
  if (i0 <= i1) ad_load(P, D, k, i0, i1, P0, Q0, st);
  for (int ib = i0; ib <= i1; ib += kAdKC) {
    float mmax = 0.f, lmax = 0.f;
#pragma unroll
    for (int s = 0; s < kAdSlots; ++s) {
      const int e = threadIdx.x + s * kAdThreads;
      const int kk = e % kAdKC, r = e / kAdKC;
      const float2 t = two_prod(st.l[s], st.d.x);
      const float2 mv = fast_two_sum(t.x, fmaf(st.l[s], st.d.y, t.y));
      sM[kk][r] = mv;
      sL[kk][r] = st.a[s];
      mmax = fmaxf(mmax, fabsf(mv.x));
      lmax = fmaxf(lmax, fabsf(st.a[s]));
    }
    for (int o = 16; o; o >>= 1) {
      mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
      lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    }
    if ((threadIdx.x & 31) == 0) {
      sMax[0][threadIdx.x >> 5] = mmax;
      sMax[1][threadIdx.x >> 5] = lmax;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kAdThreads / 32; ++w) {
      mmax = fmaxf(mmax, sMax[0][w]);
      lmax = fmaxf(lmax, sMax[1][w]);
    }
    // |sum of the chunk| <= kAdKC * (1 + 2^-23) * mmax * lmax (the low words
    // of M are below 2^-23 of the high ones); the offset is 4 to 8 times that.
    const float sig = offset_for_bound(1.001f * kAdKC * mmax * lmax);
#pragma unroll
    for (int a = 0; a < kAdRM; ++a)
#pragma unroll
      for (int b = 0; b < kAdRN; ++b) acc[a][b].init(sig);
    if (ib + kAdKC <= i1) ad_load(P, D, k, ib + kAdKC, i1, P0, Q0, st);  // next chunk, behind the products
    const int kn = min(kAdKC, i1 - ib + 1);
#pragma unroll 4
    for (int kk = 0; kk < kn; ++kk) {
      const float4 mm = *reinterpret_cast<const float4*>(&sM[kk][kAdRM * tr]);  // rows 2 tr, 2 tr + 1
      const float2 m0 = make_float2(mm.x, mm.y), m1 = make_float2(mm.z, mm.w);
      float lv[kAdRN];
      if constexpr (kAdRN == 4) {
        const float4 ll = *reinterpret_cast<const float4*>(&sL[kk][4 * tc]);  // columns 4 tc .. 4 tc + 3
        lv[0] = ll.x, lv[1] = ll.y, lv[2] = ll.z, lv[3] = ll.w;
      } else {
        const float2 ll = *reinterpret_cast<const float2*>(&sL[kk][2 * tc]);  // columns 2 tc, 2 tc + 1
        lv[0] = ll.x, lv[1] = ll.y;
      }
#pragma unroll
      for (int b = 0; b < kAdRN; ++b) {
        acc[0][b].mac(lv[b], m0);
        acc[1][b].mac(lv[b], m1);
      }
    }
#pragma unroll
    for (int a = 0; a < kAdRM; ++a)
#pragma unroll
      for (int b = 0; b < kAdRN; ++b) tot[a][b] = df_add(tot[a][b], acc[a][b].value(sig));
    __syncthreads();
  }

  const bool terms = i0 <= i1;
#pragma unroll
  for (int a = 0; a < kAdRM; ++a) {
    const int p = P0 + kAdRM * tr + a;
    if (p >= P.m) continue;
#pragma unroll
    for (int b = 0; b < kAdRN; ++b) {
      const int q = Q0 + kAdRN * tc + b;
      if (q >= P.n || p + q <= k) continue;
      const size_t o = (size_t)p * P.n + q;
      float2 x = P.Wt[o];
      if (terms) x = df_add(x, tot[a][b]);
      if (p + q == k + 1) ad_round(P, p, q, x, Dn);
      else if (terms) P.Wt[o] = x;
    }
  }
}

struct AdLayout {
  size_t wt, d, total;
};
AdLayout ad_layout(int64_t m, int64_t n) {
  AdLayout L;
  L.wt = 0;
  L.d = L.wt + align_up((size_t)m * (size_t)n * sizeof(float2));
  L.total = L.d + align_up(2 * (size_t)m * sizeof(float2));
  return L;
}

}  // namespace

size_t antidiag_workspace_bytes(int64_t m, int64_t n) { return ad_layout(m, n).total; }

cudaError_t antidiag_launch(const float* W, const float* LA, const float* LB, const float* scales, Alphabet al,
                            int m, int n, int32_t* V, float* Wq, void* ws, int32_t* status_dev,
                            cudaStream_t stream) {
  const AdLayout lay = ad_layout(m, n);
  char* base = static_cast<char*>(ws);
  AdParams P;
  P.W = W;
  P.LA = LA;
  P.LB = LB;
  P.scales = scales;
  P.V = V;
  P.Wq = Wq;
  P.Wt = reinterpret_cast<float2*>(base + lay.wt);
  P.D = reinterpret_cast<float2*>(base + lay.d);
  P.status = status_dev;
  P.m = m;
  P.n = n;
  P.bounded = al.bounded ? 1 : 0;
  P.lo = al.lo;
  P.hi = al.hi;
  const cudaError_t err = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  const size_t total = (size_t)m * n;
  const int pre_blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 8);
  ad_prepass_kernel<<<pre_blocks, 256, 0, stream>>>(P);
  const dim3 grid((unsigned)((n + kAdT - 1) / kAdT), (unsigned)((m + kAdT - 1) / kAdT));
  if ((int64_t)m * n <= (int64_t)1 << 21) {
    for (int k = -1; k <= m + n - 3; ++k) ad_step_kernel<2><<<grid, AdShape<2>::kThreads, 0, stream>>>(P, k);
  } else {
    for (int k = -1; k <= m + n - 3; ++k) ad_step_kernel<4><<<grid, AdShape<4>::kThreads, 0, stream>>>(P, k);
  }
  return cudaGetLastError();
}

}  // namespace bakron
