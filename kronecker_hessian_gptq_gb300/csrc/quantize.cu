// quantize.cu -- the BaKron core on sm_103a (tile wavefront, double-float state).
//
// "BaKron: Efficient Quantization with Kronecker-Factored Hessians":
//   App. B eq. (2): W~ = W0 + L_B (sum of earlier errors) L_A^T on every
//     anti-diagonal, v = round(W~), E = v - W~.
//   Sec. 3.3: entries on one anti-diagonal never affect one another, so they
//     are rounded in parallel; more generally entry (i, j) only affects
//     entries (p, q) with i <= p and j <= q.
//   Sec. 3.4 / 3.5 and App. B eq. (1): the updates from a finished set of
//     entries to a later set are one dense product L_B E L_A^T restricted to
//     the later set, so they can be delayed and batched.
//
// Decomposition used here.  With G = E L_A^T (row transform; G[i, q] only
// depends on row i's errors in columns <= q) and L_B unit lower triangular,
//     W~[p, q] = W0[p, q] + sum_{i < p} L_B[p, i] G[i, q] + (G[p, q] - E[p, q]).
// The matrix is cut into T x T tiles.  Tile (I, J) depends on tiles (I', J')
// with I' <= I, J' <= J, so all tiles on one tile anti-diagonal I + J = K are
// independent (the tile-level version of Sec. 3.3).  Per tile:
//   X  = W0 + sum_{I' < I} L_B[I, I'] G[I', J]         column-external part
//   Gx = sum_{J' < J} E[I, J'] L_A[J, J']^T             row-external part
//   C  = X + L_B[I, I] Gx                               tile input
// and the tile itself is a T x T BaKron problem on C with the diagonal
// blocks L_B[I, I], L_A[J, J].  After tile (I, J) is solved, its errors are
// pushed forward (Sec. 3.4's delayed update, one T x T x T product each):
//   Gx[I, J''] += E[I, J] L_A[J'', J]^T    for every J'' > J   (same tile row)
//   X[I'', J]  += L_B[I'', I] G[I, J]      for every I'' > I   (same tile column)
// with G[I, J] = Gx[I, J] + (in-tile row transform).  Every later tile
// receives exactly one such product per tile anti-diagonal and array, so
// the pushes of one anti-diagonal are race-free without atomics.
//
// Inside a tile one thread owns one entry; at in-tile step k the entries with
// p + q = k are rounded, then every later entry folds in the one new term of
// its row sum (E[p, k-p] L_A[q, k-p]) and the one new term of its column sum
// (L_B[p, k-q] G[k-q, q]).  2T-1 steps, one barrier each.
//
// Precision: all of X, Gx/G, E and every accumulation are double-float
// (df.cuh); the rounding decision itself is the fp32 division
// fp32(W~) / s_i rounded half to even, and E = s_i v - W~ is formed exactly.
#include <algorithm>
#include <vector>

#include "bakron.h"
#include "df.cuh"
#include "internal.h"

namespace bakron {
namespace {

constexpr int T = 32;  // tile edge

struct Header {
  unsigned maxw_bits;  // max |W| as ordered uint bits
  unsigned maxs_bits;  // max scale
  float sigma;         // offset of the offset accumulators
  int pad[61];
};
static_assert(sizeof(Header) == 256, "header is one alignment unit");

struct QParams {
  const float* W;
  const float* LA;
  const float* LB;
  const float* scales;
  int32_t* V;
  float* Wq;
  float2* X;   // m x n
  float2* GG;  // m x n: row-external sum, then the full row transform G
  float2* E;   // m x n
  Header* hdr;
  int32_t* status;
  int m, n, Mt, Nt, bits, lo, hi;
};

__device__ __forceinline__ unsigned warp_max(unsigned v) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Checks the inputs, finds max |W| and max scale, and initializes the state.
__global__ void prepass_kernel(QParams P) {
  const size_t total = (size_t)P.m * P.n;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  unsigned wmax = 0, smax = 0;
  int bad = 0;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    float w = P.W[idx];
    if (!isfinite(w)) {
      bad |= BAKRON_DEV_NONFINITE_W;
    } else {
      wmax = max(wmax, __float_as_uint(fabsf(w)));
    }
    P.X[idx] = make_float2(w, 0.f);
    P.GG[idx] = make_float2(0.f, 0.f);
    P.E[idx] = make_float2(0.f, 0.f);
  }
  if (P.scales) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)P.m; i += stride) {
      float s = P.scales[i];
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
  float maxw = __uint_as_float(P.hdr->maxw_bits);
  float maxs = P.scales ? __uint_as_float(P.hdr->maxs_bits) : 1.f;
  float levels = P.bits ? (float)(1 << (P.bits - 1)) : 1.f;
  // Every value rounded or accumulated stays within a few alphabet steps of
  // the weights; the offset leaves a wide margin above that.
  float bound = 16.f * (maxw + maxs * (levels + 2.f));
  P.hdr->sigma = offset_for_bound(bound);
}

// Solves every tile (I, K - I), I = I0 + blockIdx.x, of tile anti-diagonal K.
__global__ void __launch_bounds__(T* T, 1) tile_solve_kernel(QParams P, int K, int I0) {
  const int I = I0 + blockIdx.x;
  const int J = K - I;
  const int p = threadIdx.y, q = threadIdx.x;
  const int r = I * T + p, c = J * T + q;
  const bool valid = (r < P.m) && (c < P.n);
  const size_t idx = (size_t)r * P.n + c;

  __shared__ float sLB[T][T + 1];
  __shared__ float sLA[T][T + 1];
  __shared__ float2 sG[T][T + 1];
  __shared__ float2 sE[T][T + 1];

  const float sigma = P.hdr->sigma;
  {
    const int gr = I * T + p, gc = I * T + q;
    float v = 0.f;
    if (gr < P.m && gc < P.m) v = (q < p) ? P.LB[(size_t)gr * P.m + gc] : (q == p ? 1.f : 0.f);
    sLB[p][q] = v;
  }
  {
    const int gr = J * T + p, gc = J * T + q;
    float v = 0.f;
    if (gr < P.n && gc < P.n) v = (q < p) ? P.LA[(size_t)gr * P.n + gc] : (q == p ? 1.f : 0.f);
    sLA[p][q] = v;
  }
  const float2 gext = valid ? P.GG[idx] : make_float2(0.f, 0.f);
  sG[p][q] = gext;
  __syncthreads();

  // C = X + L_B[I, I] Gx (unit diagonal included).
  OffsetAcc a;
  a.init(sigma);
  for (int i = 0; i <= p; ++i) a.mac(sLB[p][i], sG[i][q]);
  const float2 cin = valid ? df_add(P.X[idx], a.value(sigma)) : make_float2(0.f, 0.f);
  __syncthreads();
  sG[p][q] = make_float2(0.f, 0.f);
  sE[p][q] = make_float2(0.f, 0.f);
  const float s = (P.scales != nullptr && r < P.m) ? P.scales[r] : 1.f;
  OffsetAcc racc, cacc;
  racc.init(sigma);
  cacc.init(sigma);
  __syncthreads();

  for (int k = 0; k < 2 * T - 1; ++k) {
    if (p + q == k && valid) {
      const float2 rv = racc.value(sigma);
      const float2 x = df_add(df_add(cin, rv), cacc.value(sigma));
      // Rounding decision in fp32: x.x == fp32(x) since x is normalized.
      float v = rintf(__fdiv_rn(x.x, s));
      if (P.bits) v = fminf(fmaxf(v, (float)P.lo), (float)P.hi);
      const float2 sv = two_prod(s, v);
      const float2 e = df_sub(sv, x);
      const float2 gin = df_add(rv, e);
      sE[p][q] = e;
      sG[p][q] = gin;
      P.V[idx] = (int32_t)v;
      P.Wq[idx] = sv.x;
      P.E[idx] = e;
      P.GG[idx] = df_add(gext, gin);
    }
    __syncthreads();
    if (p + q > k) {
      const int j = k - p;
      if (j >= 0 && j < q) racc.mac(sLA[q][j], sE[p][j]);
      const int i = k - q;
      if (i >= 0 && i < p) cacc.mac(sLB[p][i], sG[i][q]);
    }
  }
}

// Pushes the errors of every tile of anti-diagonal K to the later tiles of
// its tile row (into Gx) and tile column (into X).  blockIdx.x: source tile;
// blockIdx.y: target, first the Nt-1-J row targets, then the column targets.
__global__ void __launch_bounds__(256) propagate_kernel(QParams P, int K, int I0) {
  const int I = I0 + blockIdx.x;
  const int J = K - I;
  const int nrow = P.Nt - 1 - J;
  const int t = blockIdx.y;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;

  __shared__ float sL[T][T + 1];
  __shared__ float2 sS[T][T + 1];
  const float sigma = P.hdr->sigma;
  OffsetAcc acc[4];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) acc[rr].init(sigma);

  if (t < nrow) {
    const int J2 = J + 1 + t;
    for (int e = threadIdx.x; e < T * T; e += blockDim.x) {
      const int a = e / T, b = e % T;
      const int gr = I * T + a, gc = J * T + b;
      sS[a][b] = (gr < P.m && gc < P.n) ? P.E[(size_t)gr * P.n + gc] : make_float2(0.f, 0.f);
      const int lr = J2 * T + a;
      sL[a][b] = (lr < P.n && gc < P.n) ? P.LA[(size_t)lr * P.n + gc] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < T; ++j) {
      const float l = sL[tx][j];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) acc[rr].mac(l, sS[ty + 8 * rr][j]);
    }
    const int gc = J2 * T + tx;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int gr = I * T + ty + 8 * rr;
      if (gr < P.m && gc < P.n) {
        const size_t o = (size_t)gr * P.n + gc;
        P.GG[o] = df_add(P.GG[o], acc[rr].value(sigma));
      }
    }
  } else {
    const int I2 = I + 1 + (t - nrow);
    for (int e = threadIdx.x; e < T * T; e += blockDim.x) {
      const int a = e / T, b = e % T;
      const int gr = I * T + a, gc = J * T + b;
      sS[a][b] = (gr < P.m && gc < P.n) ? P.GG[(size_t)gr * P.n + gc] : make_float2(0.f, 0.f);
      const int lr = I2 * T + a, lc = I * T + b;
      sL[a][b] = (lr < P.m && lc < P.m) ? P.LB[(size_t)lr * P.m + lc] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < T; ++i) {
      const float2 g = sS[i][tx];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) acc[rr].mac(sL[ty + 8 * rr][i], g);
    }
    const int gc = J * T + tx;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int gr = I2 * T + ty + 8 * rr;
      if (gr < P.m && gc < P.n) {
        const size_t o = (size_t)gr * P.n + gc;
        P.X[o] = df_add(P.X[o], acc[rr].value(sigma));
      }
    }
  }
}

}  // namespace

size_t quantize_workspace_bytes(int64_t m, int64_t n) {
  const size_t plane = align_up((size_t)m * (size_t)n * sizeof(float2));
  return sizeof(Header) + 3 * plane;
}

// Event pairs around launches when a KernelTimer is given.
class LaunchClock {
 public:
  LaunchClock(KernelTimer* t, cudaStream_t s) : t_(t), s_(s) {
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
  void begin(int cls) {
    if (!t_) return;
    Rec r;
    r.cls = cls;
    cudaEventCreate(&r.a);
    cudaEventCreate(&r.b);
    cudaEventRecord(r.a, s_);
    recs_.push_back(r);
  }
  void end(double flops) {
    if (!t_) return;
    Rec& r = recs_.back();
    cudaEventRecord(r.b, s_);
    t_->launches[r.cls] += 1;
    t_->flops[r.cls] += flops;
  }
  cudaError_t finish() {
    if (!t_) return cudaSuccess;
    cudaError_t e = cudaStreamSynchronize(s_);
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
    cudaEvent_t a, b;
  };
  KernelTimer* t_;
  cudaStream_t s_;
  std::vector<Rec> recs_;
};

cudaError_t quantize_launch(const float* W, const float* LA, const float* LB, const float* scales,
                            int bits, int m, int n, int32_t* V, float* Wq, void* ws,
                            int32_t* status_dev, cudaStream_t stream, KernelTimer* timer) {
  const size_t plane = align_up((size_t)m * (size_t)n * sizeof(float2));
  char* base = static_cast<char*>(ws);
  QParams P;
  P.W = W;
  P.LA = LA;
  P.LB = LB;
  P.scales = scales;
  P.V = V;
  P.Wq = Wq;
  P.hdr = reinterpret_cast<Header*>(base);
  P.X = reinterpret_cast<float2*>(base + sizeof(Header));
  P.GG = reinterpret_cast<float2*>(base + sizeof(Header) + plane);
  P.E = reinterpret_cast<float2*>(base + sizeof(Header) + 2 * plane);
  P.status = status_dev;
  P.m = m;
  P.n = n;
  P.Mt = (m + T - 1) / T;
  P.Nt = (n + T - 1) / T;
  P.bits = bits;
  P.lo = bits ? -(1 << (bits - 1)) : 0;
  P.hi = bits ? (1 << (bits - 1)) - 1 : 0;

  LaunchClock clock(timer, stream);
  cudaError_t err = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(P.hdr, 0, sizeof(Header), stream);
  if (err != cudaSuccess) return err;
  const size_t total = (size_t)m * n;
  const int pre_blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 8);
  clock.begin(0);
  prepass_kernel<<<pre_blocks, 256, 0, stream>>>(P);
  sigma_kernel<<<1, 1, 0, stream>>>(P);
  clock.end(0.0);
  const double t3 = (double)T * T * T;
  for (int K = 0; K <= P.Mt + P.Nt - 2; ++K) {
    const int I0 = K - (P.Nt - 1) > 0 ? K - (P.Nt - 1) : 0;
    const int I1 = K < P.Mt - 1 ? K : P.Mt - 1;
    const int nsrc = I1 - I0 + 1;
    clock.begin(1);
    tile_solve_kernel<<<nsrc, dim3(T, T), 0, stream>>>(P, K, I0);
    clock.end(2.0 * 1.5 * t3 * nsrc);  // in-tile row and column sums + L_B[I,I] Gx
    const int ntgt = P.Mt + P.Nt - 2 - K;
    if (ntgt > 0) {
      clock.begin(2);
      propagate_kernel<<<dim3(nsrc, ntgt), 256, 0, stream>>>(P, K, I0);
      clock.end(2.0 * t3 * (double)nsrc * ntgt);
    }
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return clock.finish();
}

}  // namespace bakron
