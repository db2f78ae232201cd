// sweep.cu -- the BaKron core as one persistent cooperative kernel on
// sm_103a: a band-by-band sweep of the anti-diagonals on the fp32 pipes
// (double-float), fed by delayed products on the tensor cores that the same
// kernel runs from a ready-ordered task queue.
//
// "BaKron: Efficient Quantization with Kronecker-Factored Hessians":
//   App. B eq. (2): W~_k = W0 + L_B (sum of earlier errors) L_A^T on every
//     anti-diagonal k, v = round(W~_k), E_k = v - W~_k;
//   Sec. 3.3: the entries of one anti-diagonal are independent, so all of
//     them are rounded in one step (m + n - 1 dependent steps in all);
//   Sec. 3.4, 3.5, App. B eq. (1): the updates from finished entries to
//     later ones are one product L_B E L_A^T restricted to the later
//     entries; delayed and batched, they become the dense products that
//     carry the O(mn(m+n)) work.
//
// Decomposition (sweep_plan.h has the full map).  With G = E L_A^T,
//     W~[r, q] = W0[r, q] + sum_{i<r} L_B[r, i] G[i, q] + sum_{j<q} E[r, j] L_A[q, j].
// Band I (rows 32I .. 32I+31) is swept by one CTA's band warps, one band
// anti-diagonal per step (row p rounds column s - p at band step s):
//   ring warps (8): warp w owns the band anti-diagonals k = w (mod 8); lane
//     p holds, for its next 12 anti-diagonals, the column and row offset
//     accumulators of entry (p, k - p).  Each step every warp folds in the
//     previous step's errors E (row terms from source tiles 0..2 back) and
//     row transforms G (column terms from the band's own rows); the owner of
//     the step's anti-diagonal rounds it and publishes E and G.
//   write-out warp: coalesced stores of V, Wq, the bf16 digits of E (row
//     products) and of G (column products), and the band's G columns for
//     the band below; publishes the band's progress.
//   band-above warps (2): fold the previous band's published G columns into
//     this band (column terms at band distance 1).
// Everything farther is carried by tensor-core products that the product
// warps of every CTA take from a queue ordered by the time their sources
// complete: slices (8 source lines, K = 32) for the middle distances,
// chunks (K = 128) for the far ones.  They add into two 64-bit fixed-point
// planes (exact, order-independent integer reductions) and count their
// completion per target; a band loads a target's delayed sums 16 steps
// before rounding it, after its counts are complete.
// Every wait is bounded (about a second); one that runs out sets
// BAKRON_DEV_TIMEOUT and an abort flag, after which every wait returns at
// once and the kernel runs to its end without further waiting.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "bakron.h"
#include "df.cuh"
#include "internal.h"
#include "solve_common.cuh"
#include "sweep_plan.h"
#include "tc.cuh"

namespace bakron {
namespace {

using sweep::Geom;
using sweep::Task;

constexpr int kRingWarps = 8;
constexpr int kSlots = 12;        // anti-diagonals held per ring lane: k0, k0 + 8, ..., k0 + 88
constexpr int kCSlots = 4;        // of which the first 4 can still receive in-band column terms
constexpr int kRing = 48;         // columns kept in the shared rings (E, v, Wq, G, band-above sums)
constexpr int kWoWarp = 8;        // write-out warp
constexpr int kBaWarp0 = 9;       // band-above warps 9, 10
constexpr int kBandWarps = 11;
constexpr int kEpiWarp0 = 12;     // epilogue warps 12..15 (tensor-memory lane quarters 0..3)
constexpr int kMmaWarp = 16;
constexpr int kSchedWarp = 17;
constexpr int kWarps = 18;
constexpr int kThreads = kWarps * 32;
constexpr int kProdThreads = (kWarps - kEpiWarp0) * 32;  // 192
constexpr int kTcM = 128;         // target lines per product group
constexpr int kGroups = sweep::kGroupsPerTask;
constexpr int kPubBufs = 3;       // step publications kept (see the ring loop)
constexpr long long kWaitNs = 1000000000ll;  // one second

// Named barriers (0 is __syncthreads).
constexpr int kBarRing = 1, kBarProd = 2, kBarEpi = 3, kBarBand = 4;

struct SweepParams {
  const float* W;
  const float* LA;
  const float* LB;
  const float* scales;   // m x ngroups, or null
  const float* cscales;  // n, or null
  int group, ngroups;
  int32_t* V;
  float* Wq;
  long long* Xc;         // column-direction delayed sums (fixed point), m x n
  long long* Gc;         // row-direction delayed sums, m x n
  float2* Gt;            // published G: [band][column][32 rows]
  __nv_bfloat16* DE;     // E digits [digit][row][ldE]
  __nv_bfloat16* DGt;    // G digits [digit][column][ldG]
  size_t dstrideE, dstrideG;
  int ldE, ldG;
  const signed char* expA;
  const signed char* expB;
  const __nv_bfloat16* FdA;
  const __nv_bfloat16* FdB;
  int ntA, ntB, nchA, nchB;
  int* progress;         // [Mt]: last band step written out (-1: none)
  unsigned* cnt_col;     // [Mt][ncs] completed column-direction products per (band, 8 columns)
  const unsigned* exp_col;
  unsigned* cnt_row;     // [Mt][Nt][4] completed row-direction products per (band, tile, 8 rows)
  const unsigned* exp_row;
  const int* tasks;      // canonical task indices in ready order
  const unsigned* ntasks;
  Header* hdr;
  int32_t* status;
  int m, n, Mt, Nt, ncs, bounded, lo, hi;
  Geom geom;
};

// ------------------------------------------------------------- shared memory
struct ProdSmem {
  __nv_bfloat16 A[2][kDigF][kTcM * kSlab];  // factor digit slabs (core-matrix layout, SBO 512 B)
  __nv_bfloat16 Bd[kDigD * T * CK];         // source digits, digit-major rows x K (SBO = K / 8 * 128 B)
  int er[kGroups][kTcM];                    // factor row exponents of each group
  uint64_t afull[2], aempty[2], gfull[2], gempty[2], bfull;
  uint32_t tmem_base;
  int task_idx;                             // canonical index of the posted task, -1: stop
};

struct BandSmem {
  float LA[3][3 * T][T];        // L_A panels [source tile mod 3]: rows 32j .. 32j+95, columns 32j .. 32j+31
  float LB0[T][T];              // L_B[band, band]
  float LB1[T][T + 1];          // L_B[band, band - 1]
  float2 sE[kPubBufs][T];       // the last rounded anti-diagonals' errors, by row
  float2 sG[kPubBufs][T];       // and row transforms
  float4 EV[kRing][T];          // (E hi, E lo, v, Wq) by (column mod kRing, row)
  float2 Gr[kRing][T];          // G by (column mod kRing, row)
  float2 BA[kRing][T];          // band-above sums by (column mod kRing, row)
  float2 Ga[2][T];              // band-above staging of one G column per warp
  int rounded;                  // last band step rounded
  int written;                  // last band step written out
  int ba_done[2];               // last column of each band-above warp's sums
  int panel;                    // last L_A panel loaded
};

constexpr size_t kSmemBytes = sizeof(ProdSmem) + sizeof(BandSmem) + 1024;

// ------------------------------------------------------------------ waits
__device__ __forceinline__ long long gtimer() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_u(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ long long ldcg_ll(const long long* p) { return __ldcg(p); }

__device__ __forceinline__ bool aborted(const Header* h) { return *(volatile const int*)&h->abort != 0; }

__device__ __noinline__ void raise_timeout(const SweepParams& P) {
  atomicOr(P.status, BAKRON_DEV_TIMEOUT);
  atomicExch(&P.hdr->abort, 1);
}

// Spins until *p >= v (global, acquire).  False once the wait ran out or the
// kernel is aborting: the caller then proceeds as if it had been satisfied.
__device__ bool wait_global_ge(const SweepParams& P, const int* p, int v) {
  if (ld_acquire(p) >= v) return true;
  const long long t0 = gtimer();
  while (ld_acquire(p) < v) {
    if (aborted(P.hdr)) return false;
    if (gtimer() - t0 > kWaitNs) {
      raise_timeout(P);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}
__device__ bool wait_count(const SweepParams& P, const unsigned* p, unsigned v) {
  if (ld_acquire_u(p) >= v) return true;
  const long long t0 = gtimer();
  while (ld_acquire_u(p) < v) {
    if (aborted(P.hdr)) return false;
    if (gtimer() - t0 > kWaitNs) {
      raise_timeout(P);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}
// The same on a shared-memory counter written by other warps of the CTA.
__device__ bool wait_shared_ge(const SweepParams& P, const int* p, int v) {
  if (*(volatile const int*)p >= v) return true;
  const long long t0 = gtimer();
  while (*(volatile const int*)p < v) {
    if (aborted(P.hdr)) return false;
    if (gtimer() - t0 > kWaitNs) {
      raise_timeout(P);
      return false;
    }
    __nanosleep(20);
  }
  return true;
}

__device__ __forceinline__ void bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Entry scale fp32(R[r, q / group] t[q]) (1 without scales).
__device__ __forceinline__ float entry_scale(const SweepParams& P, int r, int q) {
  float sv = 1.f;
  if (P.scales) sv = P.scales[(size_t)r * P.ngroups + q / P.group];
  if (P.cscales) sv = __fmul_rn(sv, P.cscales[q]);
  return sv;
}

// ---------------------------------------------------------------- band role
// Loads the L_A panel of source tile j (rows 32j .. 32j+95, columns 32j ..
// 32j+31; zero outside the matrix) into slot j mod 3: one warp, cp.async.
__device__ void load_panel(const SweepParams& P, BandSmem& sb, int j) {
  const int lane = threadIdx.x & 31;
  float(*dst)[T] = sb.LA[j % 3];
  const bool vec = (P.n % 4) == 0 && (reinterpret_cast<uintptr_t>(P.LA) & 15) == 0;
  for (int e = lane; e < 3 * T * (T / 4); e += 32) {
    const int u = e / (T / 4), c4 = 4 * (e % (T / 4));
    const int gr = T * j + u, gc = T * j + c4;
    if (vec) {
      const bool ok = gr < P.n && gc < P.n;
      cp_async(&dst[u][c4], ok ? (const void*)(P.LA + (size_t)gr * P.n + gc) : (const void*)P.LA, ok ? 16 : 0, 16);
    } else {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const bool ok = gr < P.n && gc + x < P.n;
        cp_async(&dst[u][c4 + x], ok ? (const void*)(P.LA + (size_t)gr * P.n + gc + x) : (const void*)P.LA,
                 ok ? 4 : 0, 4);
      }
    }
  }
  cp_async_commit();
}

// The ring warps of band I.
__device__ void band_ring(const SweepParams& P, BandSmem& sb, int I, float sigma) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int p = lane, r = I * T + p;
  const bool vr = r < P.m;
  const int n = P.n;
  const int steps = n + T - 1;
  const float flo = (float)P.lo, fhi = (float)P.hi;
  const float from_units = pow2f(fixed_unit_exp(sigma));

  // Row accumulators for all slots; column accumulators only for slots
  // 0..kCSlots-1: a slot's in-band column terms come from rows at most 31
  // anti-diagonals back, and slot i is at least 8i + 1 ahead of the source.
  float rH[kSlots], rL[kSlots], cH[kCSlots], cL[kCSlots];
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    rH[i] = sigma;
    rL[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < kCSlots; ++i) {
    cH[i] = sigma;
    cL[i] = 0.f;
  }
  int k0 = w;  // next anti-diagonal this warp rounds (slot 0)
  // Delayed sums, input and scale of the entry of slot 1, loaded ahead.
  float pW = 0.f, pS = 1.f;
  long long pX = 0, pG = 0;
  float se0 = 1.f, rcp0 = 1.f;  // scale of slot 0's entry

  auto prefetch = [&](int k) {
    const int q = k - p;
    pW = 0.f;
    pX = pG = 0;
    pS = 1.f;
    if (vr && q >= 0 && q < n) {
      wait_count(P, P.cnt_col + (size_t)I * P.ncs + (q >> 3), P.exp_col[(size_t)I * P.ncs + (q >> 3)]);
      const size_t ri = ((size_t)I * P.Nt + (q >> 5)) * 4 + (p >> 3);
      wait_count(P, P.cnt_row + ri, P.exp_row[ri]);
      const size_t o = (size_t)r * n + q;
      pW = __ldg(P.W + o);
      pX = ldcg_ll(P.Xc + o);
      pG = ldcg_ll(P.Gc + o);
      pS = entry_scale(P, r, q);
    }
  };
  // Slot 0 now holds anti-diagonal k: add its input, delayed sums and band-above sum.
  auto refresh0 = [&](int k) {
    const int q = k - p;
    if (I > 0) {
      const int need = min(k, n - 1);
      wait_shared_ge(P, &sb.ba_done[0], need);
      wait_shared_ge(P, &sb.ba_done[1], need);
    }
    se0 = pS;
    rcp0 = __frcp_rn(pS);
    if (vr && q >= 0 && q < n) {
      OffsetAcc c{cH[0], cL[0]}, rr{rH[0], rL[0]};
      c.mac(1.f, pW);
      c.mac(1.f, df_from_fixed(pX, from_units));
      if (I > 0) c.mac(1.f, sb.BA[q % kRing][p]);
      rr.mac(1.f, df_from_fixed(pG, from_units));
      cH[0] = c.H;
      cL[0] = c.L;
      rH[0] = rr.H;
      rL[0] = rr.L;
    }
  };
  // Folds the errors and row transforms published by step ps (anti-diagonal
  // ps) into slots [i0, i1).
  auto fold = [&](int ps, int i0, int i1) {
    const int buf = ps % kPubBufs;
    const int qsrc = ps - p;  // this row's source column
    const bool rowok = vr && qsrc >= 0 && qsrc < n;
    const float2 eP = sb.sE[buf][p];
    const int c = qsrc & (T - 1);
    const float* panel = &sb.LA[(rowok ? (qsrc >> 5) : 0) % 3][0][0];
    const int d0 = k0 - ps;  // distance of slot 0's anti-diagonal (>= 1)
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      if (i < i0 || i >= i1) continue;
      const int delta = d0 + 8 * i;
      const int q = k0 + 8 * i - p;  // the slot's column
      const bool tok = vr && q >= 0 && q < n;
      // row term E[p, qsrc] L_A[q, qsrc], source within 2 tiles of the target
      const int u = c + delta;
      if (rowok && tok && u < 3 * T) {
        OffsetAcc a{rH[i], rL[i]};
        a.mac(panel[u * T + c], eP);
        rH[i] = a.H;
        rL[i] = a.L;
      }
      // column term L_B[p, p'] G[p', q], p' = p - delta (same band)
      if (i < kCSlots && delta < T) {  // warp-uniform
        if (tok && delta <= p) {
          const int pp = p - delta;
          OffsetAcc a{cH[i], cL[i]};
          a.mac(sb.LB0[p][pp], sb.sG[buf][pp]);
          cH[i] = a.H;
          cL[i] = a.L;
        }
      }
    }
  };

  // Set-up: slot 0 = anti-diagonal w, prefetched and refreshed; slot 1 prefetched.
  prefetch(k0);
  refresh0(k0);
  prefetch(k0 + 8);
  bool arrived = false;  // this warp already arrived at the current step's barrier

  for (int s = 0; s < steps; ++s) {
    if (!arrived) bar_sync(kBarRing, kRingWarps * 32);
    arrived = false;
    // The source L_A panel of the newest source column s - 1 (row 0's).
    if (s >= 1 && ((s - 1) & (T - 1)) == 0) wait_shared_ge(P, &sb.panel, (s - 1) >> 5);
    if (k0 == s) {
      if (s >= 1) fold(s - 1, 0, 1);
      // Round anti-diagonal s: entry (p, s - p).
      const int q = s - p;
      float2 e = make_float2(0.f, 0.f), g = e;
      float v = 0.f, wq = 0.f;
      if (vr && q >= 0 && q < n) {
        // (cH - sigma) and (rH - sigma) are exact, and so is their sum.
        const float2 x = two_sum((cH[0] - sigma) + (rH[0] - sigma), cL[0] + rL[0]);
        float y = x.x * rcp0;
        if (!(fabsf(y) <= 256.f) || fabsf(y - floorf(y) - 0.5f) < 1e-3f) y = __fdiv_rn(x.x, se0);
        v = rintf(y);
        if (P.bounded) v = fminf(fmaxf(v, flo), fhi);
        const float2 sv = two_prod(se0, v);
        const float2 h = two_sum(sv.x, -x.x);
        e = fast_two_sum(h.x, (sv.y - x.y) + h.y);
        g = df_add(two_sum(rH[0] - sigma, rL[0]), e);
        wq = se0 * v;
      }
      // The rings' slots of column q were written out at least 16 steps ago.
      wait_shared_ge(P, &sb.written, s - (kRing - T));
      const int buf = s % kPubBufs;
      sb.sE[buf][p] = e;
      sb.sG[buf][p] = g;
      if (q >= 0 && q < n) {
        sb.EV[q % kRing][p] = make_float4(e.x, e.y, v, wq);
        sb.Gr[q % kRing][p] = g;
      }
      __syncwarp();
      __threadfence_block();
      if (p == 0) *(volatile int*)&sb.rounded = s;
      bar_arrive(kBarRing, kRingWarps * 32);
      arrived = true;
      if (s >= 1) fold(s - 1, 1, kSlots);
      // Shift the ring: slot i takes slot i + 1, a new anti-diagonal enters.
#pragma unroll
      for (int i = 0; i + 1 < kSlots; ++i) {
        rH[i] = rH[i + 1];
        rL[i] = rL[i + 1];
      }
#pragma unroll
      for (int i = 0; i + 1 < kCSlots; ++i) {
        cH[i] = cH[i + 1];
        cL[i] = cL[i + 1];
      }
      rH[kSlots - 1] = sigma;
      rL[kSlots - 1] = 0.f;
      cH[kCSlots - 1] = sigma;
      cL[kCSlots - 1] = 0.f;
      k0 += 8;
      if (k0 < steps) {
        refresh0(k0);
        prefetch(k0 + 8);
      }
    } else if (s >= 1) {
      fold(s - 1, 0, kSlots);
    }
  }
  if (!arrived) bar_sync(kBarRing, kRingWarps * 32);
}

// The write-out warp of band I: V, Wq and the digits of E for every row
// tile a row completes, G (published and as digits) for every column the
// band completes, the L_A panels ahead of the sweep, and the band's progress.
__device__ void band_writeout(const SweepParams& P, BandSmem& sb, int I, float sigma) {
  const int lane = threadIdx.x & 31;
  const int n = P.n, steps = n + T - 1;
  const float dsc = pow2f(7 - bound_exp(sigma));
  const int r0 = I * T;
  int next_panel = 1;  // panel 0 is loaded before the sweep starts
  for (int s = 0; s < steps; ++s) {
    // Panel j is first read at step 32j + 1.  Its slot's previous panel
    // (j - 3) is read for source anti-diagonals up to 32j - 34, the last of
    // them by a warp's deferred folds before its barrier of step 32j - 31;
    // this iteration starts once step s - 1 is rounded, so s >= 32j - 24 is
    // safe, and leaves 25 steps to load.
    if (next_panel < P.Nt && s >= T * next_panel - 24) {
      load_panel(P, sb, next_panel);
      cp_async_wait_all();
      __syncwarp();
      __threadfence_block();
      if (lane == 0) *(volatile int*)&sb.panel = next_panel;
      ++next_panel;
    }
    wait_shared_ge(P, &sb.rounded, s);
    // Row tiles completed at step s: row p completes tile j when it rounds
    // column min(32j + 31, n - 1).
    for (int ev = 0; ev < 2; ++ev) {
      int p = -1, j = -1;
      if (ev == 0 && s >= T - 1) {
        p = (s - (T - 1)) & (T - 1);
        j = (s - (T - 1) - p) / T;
        if (T * j + T - 1 > n - 1) p = -1;  // the ragged last tile completes at column n - 1
      } else if (ev == 1 && (n % T) != 0) {
        p = s - (n - 1);
        j = P.Nt - 1;
        if (p < 0 || p >= T) p = -1;
      }
      if (p < 0 || r0 + p >= P.m) continue;
      const int q = T * j + lane;
      if (q < n) {
        const float4 ev4 = sb.EV[q % kRing][p];
        const size_t o = (size_t)(r0 + p) * n + q;
        P.V[o] = (int32_t)ev4.z;
        P.Wq[o] = ev4.w;
        put_digits(P.DE, P.dstrideE, (size_t)(r0 + p) * P.ldE + q, make_float2(ev4.x, ev4.y), dsc);
      }
    }
    // The column completed at step s (row 31 rounded it).
    const int c = s - (T - 1);
    if (c >= 0 && c < n) {
      const float2 g = sb.Gr[c % kRing][lane];
      P.Gt[((size_t)I * n + c) * T + lane] = g;
      if (r0 + lane < P.m) put_digits(P.DGt, P.dstrideG, (size_t)c * P.ldG + r0 + lane, g, dsc);
    }
    __syncwarp();
    if (lane == 0) *(volatile int*)&sb.written = s;
    if ((s & 3) == 3 || s == steps - 1) {
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release(P.progress + I, s);
    }
  }
}

// Band-above warp h (0, 1) of band I: for columns c = h (mod 2), the sums
// sum_i L_B[32I + p, 32(I-1) + i] G[32(I-1) + i, c] of band I - 1's
// published G, into the ring BA.
__device__ void band_above(const SweepParams& P, BandSmem& sb, int I, int h, float sigma) {
  const int lane = threadIdx.x & 31;
  const int n = P.n;
  if (I == 0) {
    if (lane == 0) *(volatile int*)&sb.ba_done[h] = n;
    return;
  }
  int seen = -1;  // band I - 1's progress, last read
  for (int c = h; c < n; c += 2) {
    if (seen < c + T - 1) {
      wait_global_ge(P, P.progress + (I - 1), c + T - 1);
      seen = ld_acquire(P.progress + (I - 1));
    }
    // The ring slot of column c - kRing is free once every row consumed it:
    // row p consumes column c' at the refresh of anti-diagonal c' + p, done
    // by the warp that rounds c' + p - 8 before its barrier of step
    // c' + p - 6; so step c' + 31 - 6 rounded means all rows did.
    wait_shared_ge(P, &sb.rounded, c - kRing + T - 6);
    sb.Ga[h][lane] = __ldcg(P.Gt + ((size_t)(I - 1) * n + c) * T + lane);
    __syncwarp();
    OffsetAcc a;
    a.init(sigma);
#pragma unroll 8
    for (int i = 0; i < T; ++i) a.mac(sb.LB1[lane][i], sb.Ga[h][i]);
    sb.BA[c % kRing][lane] = a.value(sigma);
    __syncwarp();
    __threadfence_block();
    if (lane == 0) *(volatile int*)&sb.ba_done[h] = c;
  }
  if (lane == 0) *(volatile int*)&sb.ba_done[h] = n;
}

// --------------------------------------------------------------- product role
// One task at a time: the scheduler lane fetches the next task of the queue
// and waits until its sources are complete; the epilogue warps copy the
// source digits; the scheduler lane streams the factor digit slabs (bulk
// copies); the MMA lane multiplies (tcgen05, five products per 16-deep
// step: factor digit a against all source digits stacked along N); the
// epilogue warps fold the levels into the fixed-point planes and count the
// task's completion for each of its targets.
struct TaskView {
  Task t;
  bool row;      // row-direction task (factor L_A, plane Gc) or column-direction (L_B, Xc)
  bool chunk;    // K up to 128 and 32 source lines, else a slice: K = 32, 8 lines
  int nl;        // source lines per digit block in Bd (32; a slice uses its first 8)
  int kmax;      // K extent of Bd (32 or 128)
  int nslab;     // factor slabs per group
  int ngroups;
  int c;         // factor chunk of the source K range
  int s0;        // first slab within the chunk
  int tgt0;      // first target line (factor row)
  int tgt_end;   // one past the last target line
};

__device__ __forceinline__ TaskView view_of(const SweepParams& P, long long idx) {
  TaskView v;
  v.t = sweep::decode(P.geom, idx);
  v.row = v.t.type == sweep::kRowSlice || v.t.type == sweep::kRowChunk;
  v.chunk = v.t.type == sweep::kRowChunk || v.t.type == sweep::kColChunk;
  // Every product uses the chunk products' tensor-memory layout: source
  // digit blocks of 32 lines (a slice's 8 lines zero-padded), level l of
  // the digit products at tensor-memory columns 32 l .. 32 l + 31.
  v.nl = T;
  v.kmax = v.chunk ? CK : T;
  v.nslab = (v.t.kLen + kSlab - 1) / kSlab;
  const int dlim = v.row ? P.n : P.m;
  v.tgt0 = T * v.t.t0;
  v.tgt_end = min(T * v.t.t1, dlim);
  v.ngroups = (v.tgt_end - v.tgt0 + kTcM - 1) / kTcM;
  v.c = v.t.k0 / CK;
  v.s0 = (v.t.k0 % CK) / kSlab;
  return v;
}

__device__ void product_role(const SweepParams& P, ProdSmem& sm, float sigma) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool is_epi = warp >= kEpiWarp0 && warp < kEpiWarp0 + 4;
  const int eD = bound_exp(sigma);
  const int fexp_unit = fixed_unit_exp(sigma);
  const uint32_t tmem = sm.tmem_base;
  bool broken = false;
  // Running counts for the mbarrier phases (all roles count the same way).
  uint32_t zc = 0;   // factor slabs issued
  uint32_t gc = 0;   // groups multiplied
  uint32_t tc = 0;   // tasks whose source digits were loaded

  for (;;) {
    // Fetch and wait (scheduler lane), post to the product warps.
    if (warp == kSchedWarp && lane == 0) {
      int post = -1;
      if (!aborted(P.hdr)) {
        const unsigned i = atomicAdd(&P.hdr->queue_head, 1u);
        if (i < *P.ntasks) {
          post = P.tasks[i];
          const Task t = sweep::decode(P.geom, post);
          for (int b = t.srcBand0; b < t.srcBand1; ++b) wait_global_ge(P, P.progress + b, t.readyStep);
        }
      }
      sm.task_idx = post;
    }
    bar_sync(kBarProd, kProdThreads);
    const int idx = sm.task_idx;
    if (idx < 0) break;
    const TaskView v = view_of(P, idx);
    const __nv_bfloat16* Fd = v.row ? P.FdA : P.FdB;
    const signed char* fexp = v.row ? P.expA : P.expB;
    const int nch = v.row ? P.nchA : P.nchB;
    const int nt = v.row ? P.ntA : P.ntB;
    const int dlim = v.row ? P.n : P.m;
    const int nz = v.ngroups * v.nslab;

    if (is_epi) {
      // Source digits: row tasks read E digits of rows line0.. at columns
      // k0.., column tasks G digits of columns line0.. at rows k0...
      const int et = tid - kEpiWarp0 * 32;
      const __nv_bfloat16* dp = v.row ? P.DE : P.DGt;
      const size_t pst = v.row ? P.dstrideE : P.dstrideG;
      const int ld = v.row ? P.ldE : P.ldG;
      const int sbo = v.kmax / 8 * 128;
      const int pieces = kDigD * v.nl * (v.kmax / 8);
      for (int e = et; e < pieces; e += 128) {
        const int k8 = 8 * (e % (v.kmax / 8));
        const int line = (e / (v.kmax / 8)) % v.nl;
        const int b = e / (v.kmax / 8 * v.nl);
        const bool ok = line < v.t.nLines && k8 < v.t.kLen;
        const __nv_bfloat16* src = dp + (ok ? b * pst + (size_t)(v.t.line0 + line) * ld + v.t.k0 + k8 : 0);
        const int row = b * v.nl + line;
        unsigned char* dst = reinterpret_cast<unsigned char*>(sm.Bd) + (row / 8) * sbo + (k8 / 8) * 128 + (row % 8) * 16;
        cp_async(dst, src, ok ? 16 : 0, 16);
      }
      cp_async_commit();
      for (int e = et; e < v.ngroups * kTcM; e += 128) {
        const int gi = e / kTcM, rr = e % kTcM;
        const int gr = v.tgt0 + gi * kTcM + rr;
        sm.er[gi][rr] = gr < dlim ? (int)fexp[(size_t)gr * nch + v.c] : -100;
      }
      cp_async_wait_all();
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.bfull)) : "memory");
    }
    bar_sync(kBarProd, kProdThreads);  // er[] written, Bd in flight to the tensor cores' view

    if (warp == kSchedWarp) {
      if (lane == 0) {
        for (int z = 0; z < nz; ++z) {
          const uint32_t zz = zc + z;
          const int pb = zz & 1, gi = z / v.nslab, s = v.s0 + z % v.nslab;
          const int t0 = (v.tgt0 + gi * kTcM) / T;
          const int ntg = min(kTcM / T, nt - t0);
          const uint32_t bytes = (uint32_t)ntg * 2048u;
          if (zz >= 2) mbar_wait(&sm.aempty[pb], ((zz >> 1) - 1) & 1u, broken);
          if (broken) break;
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(&sm.afull[pb])),
                       "r"(bytes * kDigF)
                       : "memory");
          const size_t cs = (size_t)v.c * (CK / kSlab) + s;
#pragma unroll
          for (int a = 0; a < kDigF; ++a) {
            const unsigned char* src = reinterpret_cast<const unsigned char*>(Fd) + ((cs * kDigF + a) * nt + t0) * 2048;
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                    smem_u32(sm.A[pb][a])),
                "l"(src), "r"(bytes), "r"(smem_u32(&sm.afull[pb]))
                : "memory");
          }
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        mbar_wait(&sm.bfull, tc & 1u, broken);
        tc_fence_after();
        const uint32_t sbo = (uint32_t)(v.kmax / 8 * 128);
        for (int z = 0; z < nz && !broken; ++z) {
          const uint32_t zz = zc + z;
          const int pb = zz & 1, gi = z / v.nslab, sl = z % v.nslab;
          const uint32_t gg = gc + gi, h = gg & 1;
          if (sl == 0 && gg >= 2) mbar_wait(&sm.gempty[h], ((gg >> 1) - 1) & 1u, broken);
          mbar_wait(&sm.afull[pb], (zz >> 1) & 1u, broken);
          if (broken) break;
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < kSlab / 16; ++j) {
            const uint32_t kb = (uint32_t)((sl * kSlab + 16 * j) / 8) * 128u;
            const uint64_t db = umma_sdesc(smem_u32(sm.Bd) + kb, 128u, sbo);
#pragma unroll
            for (int a = 0; a < kDigF; ++a) {
              const uint64_t da = umma_sdesc(smem_u32(sm.A[pb][a]) + (uint32_t)(2 * j) * 128u, 128u, 512u);
              const uint32_t acc = (sl > 0 || j > 0 || a > 0) ? 1u : 0u;
              umma_bf16(tmem + (uint32_t)(256 * h + 32 * a), da, db, umma_idesc_bf16(kTcM, T * (kDigD - a)), acc);
            }
          }
          umma_commit(&sm.aempty[pb]);
          if (sl == v.nslab - 1) umma_commit(&sm.gfull[h]);
        }
      }
      __syncwarp();
    } else if (is_epi) {
      const int qd = warp - kEpiWarp0;  // tensor-memory lane quarter
      const int rr = 32 * qd + lane;    // target line within the group
      const int lvl_stride = T;
      for (int gi = 0; gi < v.ngroups; ++gi) {
        const uint32_t gg = gc + gi, h = gg & 1;
        mbar_wait(&sm.gfull[h], (gg >> 1) & 1u, broken);
        tc_fence_after();
        const int tgt = v.tgt0 + gi * kTcM + rr;  // factor row = target line
        const bool rok = tgt < v.tgt_end;
        const int ex = sm.er[gi][rr] + eD - 14 - fexp_unit;
        const float sc = ex >= -126 ? pow2f(min(ex, 127)) : 0.f;
        unsigned long long* plane = reinterpret_cast<unsigned long long*>(v.row ? P.Gc : P.Xc);
        // Row tasks: Gc[source row line0 + q][target column tgt];
        // column tasks: Xc[target row tgt][source column line0 + q].
        const size_t obase = v.row ? (size_t)v.t.line0 * P.n + tgt : (size_t)tgt * P.n + v.t.line0;
        const size_t ostep = v.row ? (size_t)P.n : 1;
#pragma unroll 1
        for (int qb = 0; qb < v.t.nLines; qb += 8) {
          float lv[kLevels][8];
#pragma unroll
          for (int l = 0; l < kLevels; ++l)
            tmem_ld(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(256 * h + lvl_stride * l + qb), lv[l]);
          asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            // levels 0..2 exactly, the rest (below 2^-24 of the total) in one fp32 sum
            float2 y = two_sum(lv[0][j], lv[1][j] * 0x1p-8f);
            const float2 y2 = two_sum(y.y, lv[2][j] * 0x1p-16f);
            const float tail = lv[3][j] * 0x1p-24f + lv[4][j] * 0x1p-32f + lv[5][j] * 0x1p-40f;
            y = two_sum(y.x, y2.x);
            y = two_sum(y.x, y.y + (y2.y + tail));
            if (rok && qb + j < v.t.nLines)
              atomicAdd(plane + obase + (size_t)(qb + j) * ostep, (unsigned long long)df_to_fixed(y, sc));
          }
        }
        tc_fence_before();
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.gempty[h])) : "memory");
      }
      // Completion: every update of the task is in L2; count it per target.
      __threadfence();
      bar_sync(kBarEpi, 128);
      if (warp == kEpiWarp0) {
        if (v.row) {
          const int nps = (v.t.t1 - v.t.t0) * (v.t.ps1 - v.t.ps0);
          for (int e = lane; e < nps; e += 32) {
            const int t = v.t.t0 + e / (v.t.ps1 - v.t.ps0), ps = v.t.ps0 + e % (v.t.ps1 - v.t.ps0);
            red_release_add(P.cnt_row + ((size_t)v.t.a * P.Nt + t) * 4 + ps, 1u);
          }
        } else {
          const int ncs = v.t.cs1 - v.t.cs0;
          const int tot = (v.t.t1 - v.t.t0) * ncs;
          for (int e = lane; e < tot; e += 32) {
            const int band = v.t.t0 + e / ncs, cs = v.t.cs0 + e % ncs;
            red_release_add(P.cnt_col + (size_t)band * P.ncs + cs, 1u);
          }
        }
      }
    }
    zc += nz;
    gc += v.ngroups;
    tc += 1;
    if (broken) raise_timeout(P);
    bar_sync(kBarProd, kProdThreads);  // task done: Bd, er and the tensor memory may be reused
  }
  // Leave no bulk copy in flight: wait (bounded) for the last phase of both
  // factor slab buffers the scheduler lane filled.
  if (warp == kSchedWarp && lane == 0) {
    bool gone = false;
    for (int pb = 0; pb < 2; ++pb) {
      const uint32_t uses = (zc + 1 - pb) / 2;  // fills of buffer pb: slabs zz < zc with zz % 2 == pb
      if (uses > 0) mbar_wait(&sm.afull[pb], (uses - 1) & 1u, gone);
    }
  }
}

// -------------------------------------------------------------------- kernel
__global__ void __maxnreg__(112) sweep_kernel(SweepParams P) {
  extern __shared__ __align__(1024) unsigned char sweep_smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sweep_smem_raw) + 1023) & ~uintptr_t(1023));
  ProdSmem& sm = *reinterpret_cast<ProdSmem*>(base);
  BandSmem& sb = *reinterpret_cast<BandSmem*>(base + sizeof(ProdSmem));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float sigma = P.hdr->sigma;

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.afull[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.aempty[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.gfull[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;\n" ::"r"(smem_u32(&sm.gempty[i])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;\n" ::"r"(smem_u32(&sm.bfull)));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kMmaWarp) {  // two tensor-memory halves of 256 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(&sm.tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp >= kEpiWarp0) {
    product_role(P, sm, sigma);
  } else {
    for (int I = blockIdx.x; I < P.Mt; I += gridDim.x) {
      // Band set-up by all band warps: factor blocks, counters, first panel.
      const int bt = tid;  // 0 .. kBandWarps * 32 - 1
      for (int e = bt; e < T * T; e += kBandWarps * 32) {
        const int a = e / T, b = e % T;
        const int ra = I * T + a, cb = I * T + b;
        sb.LB0[a][b] = (ra < P.m && cb < P.m && b < a) ? P.LB[(size_t)ra * P.m + cb] : 0.f;
        const int cb1 = (I - 1) * T + b;
        sb.LB1[a][b] = (I > 0 && ra < P.m) ? P.LB[(size_t)ra * P.m + cb1] : 0.f;
      }
      if (bt == 0) {
        sb.rounded = -1;
        sb.written = -1;
        sb.ba_done[0] = -1;
        sb.ba_done[1] = -1;
        sb.panel = 0;
      }
      if (warp == kWoWarp) {
        load_panel(P, sb, 0);
        cp_async_wait_all();
      }
      __threadfence_block();
      bar_sync(kBarBand, kBandWarps * 32);
      if (warp < kRingWarps) {
        band_ring(P, sb, I, sigma);
      } else if (warp == kWoWarp) {
        band_writeout(P, sb, I, sigma);
      } else {
        band_above(P, sb, I, warp - kBaWarp0, sigma);
      }
      bar_sync(kBarBand, kBandWarps * 32);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(sm.tmem_base));
  (void)lane;
}

// ------------------------------------------------------------ task queue
// The canonical tasks (sweep_plan.h) are sorted by the ideal time at which
// their sources complete (buckets of 8 steps; order inside a bucket is free,
// since a task needs no other task that becomes ready within 26 steps of
// it), and the number of tasks serving each target is counted.
constexpr int kBucketShift = 3;

__global__ void plan_count_kernel(Geom g, unsigned* bucket_cnt, unsigned* exp_col, unsigned* exp_row, int ncs) {
  const long long total = sweep::total_tasks(g);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const Task t = sweep::decode(g, idx);
    if (t.type == sweep::kEmpty) continue;
    atomicAdd(bucket_cnt + (sweep::ready_time(t) >> kBucketShift), 1u);
    if (t.type == sweep::kRowSlice || t.type == sweep::kRowChunk) {
      for (int tt = t.t0; tt < t.t1; ++tt)
        for (int ps = t.ps0; ps < t.ps1; ++ps) atomicAdd(exp_row + ((size_t)t.a * g.Nt + tt) * 4 + ps, 1u);
    } else {
      for (int b = t.t0; b < t.t1; ++b)
        for (int cs = t.cs0; cs < t.cs1; ++cs) atomicAdd(exp_col + (size_t)b * ncs + cs, 1u);
    }
  }
}

// Exclusive scan of the bucket counts (one CTA); the total goes to *ntasks.
__global__ void __launch_bounds__(1024) plan_scan_kernel(unsigned* bucket, int nb, unsigned* ntasks) {
  __shared__ unsigned part[1024];
  const int tid = threadIdx.x;
  const int per = (nb + 1023) / 1024;
  const int b0 = tid * per, b1 = min(b0 + per, nb);
  unsigned s = 0;
  for (int b = b0; b < b1; ++b) s += bucket[b];
  part[tid] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const unsigned x = tid >= o ? part[tid - o] : 0u;
    __syncthreads();
    part[tid] += x;
    __syncthreads();
  }
  unsigned run = tid ? part[tid - 1] : 0u;
  for (int b = b0; b < b1; ++b) {
    const unsigned c = bucket[b];
    bucket[b] = run;
    run += c;
  }
  if (tid == 1023) *ntasks = part[1023];
}

__global__ void plan_scatter_kernel(Geom g, unsigned* bucket_off, int* list) {
  const long long total = sweep::total_tasks(g);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const Task t = sweep::decode(g, idx);
    if (t.type == sweep::kEmpty) continue;
    const unsigned pos = atomicAdd(bucket_off + (sweep::ready_time(t) >> kBucketShift), 1u);
    list[pos] = (int)idx;
  }
}

int num_buckets(const Geom& g) {
  // The latest ready time: the last band's last step.
  const long long last = sweep::ideal_time(g.Mt - 1, g.n + T - 2);
  return (int)(last >> kBucketShift) + 2;
}

struct DeviceInfo {
  bool ready = false;
  unsigned long long ctx_id = 0;
  int sms = 0;
  bool coop = false;
};
constexpr int kMaxDevs = 128;
DeviceInfo g_dev[kMaxDevs];
std::mutex g_dev_mutex;

cudaError_t device_info(DeviceInfo& out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevs) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready || d.ctx_id != ctx) {
    d = DeviceInfo();
    int coop = 0;
    e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sweep_kernel, kThreads, kSmemBytes);
    if (e != cudaSuccess) return e;
    d.coop = coop != 0 && per_sm >= 1;
    d.ctx_id = ctx;
    d.ready = true;
  }
  out = d;
  return cudaSuccess;
}

}  // namespace

// ------------------------------------------------------------- workspace
struct SweepLayout {
  size_t plane, Gt, DE, DG, dplaneE, dplaneG, expA, expB, FdA, FdB, progress, cnt_col, exp_col, cnt_row, exp_row,
      buckets, list, ntasks, total;
  int ldE, ldG, nbuckets;
};

SweepLayout sweep_layout(int64_t m, int64_t n) {
  SweepLayout L;
  const Geom g = sweep::make_geom((int)m, (int)n);
  const size_t nchA = (size_t)((n + CK - 1) / CK), nchB = (size_t)((m + CK - 1) / CK);
  const size_t ntA = (size_t)g.Nt, ntB = (size_t)g.Mt;
  size_t off = sizeof(Header);
  L.plane = align_up((size_t)m * n * sizeof(long long));
  off += 2 * L.plane;  // Xc, Gc
  L.Gt = off;
  off += align_up((size_t)g.Mt * n * T * sizeof(float2));
  L.ldE = (int)((n + 7) / 8 * 8);
  L.ldG = (int)((m + 7) / 8 * 8);
  L.dplaneE = align_up((size_t)m * L.ldE * sizeof(__nv_bfloat16));
  L.dplaneG = align_up((size_t)n * L.ldG * sizeof(__nv_bfloat16));
  L.DE = off;
  off += kDigD * L.dplaneE;
  L.DG = off;
  off += kDigD * L.dplaneG;
  L.expA = off;
  off += align_up((size_t)n * nchA);
  L.expB = off;
  off += align_up((size_t)m * nchB);
  L.FdA = off;
  off += align_up(nchA * (CK / kSlab) * kDigF * ntA * 2048);
  L.FdB = off;
  off += align_up(nchB * (CK / kSlab) * kDigF * ntB * 2048);
  L.progress = off;
  off += align_up((size_t)g.Mt * sizeof(int));
  const size_t ncs = (size_t)((n + 7) / 8);
  L.cnt_col = off;
  off += align_up((size_t)g.Mt * ncs * sizeof(unsigned));
  L.exp_col = off;
  off += align_up((size_t)g.Mt * ncs * sizeof(unsigned));
  L.cnt_row = off;
  off += align_up((size_t)g.Mt * g.Nt * 4 * sizeof(unsigned));
  L.exp_row = off;
  off += align_up((size_t)g.Mt * g.Nt * 4 * sizeof(unsigned));
  L.nbuckets = num_buckets(g);
  L.buckets = off;
  off += align_up((size_t)L.nbuckets * sizeof(unsigned));
  L.ntasks = off;
  off += align_up(sizeof(unsigned));
  L.list = off;
  off += align_up((size_t)sweep::total_tasks(g) * sizeof(int));
  L.total = off;
  return L;
}

size_t sweep_workspace_bytes(int64_t m, int64_t n) { return sweep_layout(m, n).total; }

bool sweep_supported(int64_t m, int64_t n) {
  // int indexing of the canonical task list, and the L_A panels need n >= 1
  return m >= 1 && n >= 1 && sweep::total_tasks(sweep::make_geom((int)m, (int)n)) < ((long long)1 << 31);
}

cudaError_t sweep_launch(const float* W, const float* LA, const float* LB, Scales sc, Alphabet al, int m, int n,
                         int32_t* V, float* Wq, void* ws, int32_t* status_dev, cudaStream_t stream,
                         float* kernel_ms) {
  DeviceInfo di;
  cudaError_t err = device_info(di);
  if (err != cudaSuccess) return err;
  if (!di.coop) return cudaErrorCooperativeLaunchTooLarge;
  const SweepLayout lay = sweep_layout(m, n);
  char* base = static_cast<char*>(ws);
  SweepParams P;
  P.geom = sweep::make_geom(m, n);
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
  P.Xc = reinterpret_cast<long long*>(base + sizeof(Header));
  P.Gc = reinterpret_cast<long long*>(base + sizeof(Header) + lay.plane);
  P.Gt = reinterpret_cast<float2*>(base + lay.Gt);
  P.DE = reinterpret_cast<__nv_bfloat16*>(base + lay.DE);
  P.DGt = reinterpret_cast<__nv_bfloat16*>(base + lay.DG);
  P.dstrideE = lay.dplaneE / sizeof(__nv_bfloat16);
  P.dstrideG = lay.dplaneG / sizeof(__nv_bfloat16);
  P.ldE = lay.ldE;
  P.ldG = lay.ldG;
  P.nchA = (n + CK - 1) / CK;
  P.nchB = (m + CK - 1) / CK;
  P.ntA = P.geom.Nt;
  P.ntB = P.geom.Mt;
  P.expA = reinterpret_cast<const signed char*>(base + lay.expA);
  P.expB = reinterpret_cast<const signed char*>(base + lay.expB);
  P.FdA = reinterpret_cast<const __nv_bfloat16*>(base + lay.FdA);
  P.FdB = reinterpret_cast<const __nv_bfloat16*>(base + lay.FdB);
  P.progress = reinterpret_cast<int*>(base + lay.progress);
  P.cnt_col = reinterpret_cast<unsigned*>(base + lay.cnt_col);
  P.exp_col = reinterpret_cast<const unsigned*>(base + lay.exp_col);
  P.cnt_row = reinterpret_cast<unsigned*>(base + lay.cnt_row);
  P.exp_row = reinterpret_cast<const unsigned*>(base + lay.exp_row);
  P.tasks = reinterpret_cast<const int*>(base + lay.list);
  P.ntasks = reinterpret_cast<const unsigned*>(base + lay.ntasks);
  P.status = status_dev;
  P.m = m;
  P.n = n;
  P.Mt = P.geom.Mt;
  P.Nt = P.geom.Nt;
  P.ncs = (n + 7) / 8;
  P.bounded = al.bounded ? 1 : 0;
  P.lo = al.lo;
  P.hi = al.hi;

  // Zeroed state: status, header, the two planes, the counters and buckets;
  // progress = -1.  Digit rows are padded to 8 entries and the products read
  // the padding, which must then be zero.
  err = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(P.hdr, 0, sizeof(Header), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(P.Xc, 0, 2 * lay.plane, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(base + lay.progress, 0xFF, lay.cnt_col - lay.progress, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(base + lay.cnt_col, 0, lay.list - lay.cnt_col, stream);
  if (err == cudaSuccess && (lay.ldE != n || lay.ldG != m))
    err = cudaMemsetAsync(base + lay.DE, 0, kDigD * (lay.dplaneE + lay.dplaneG), stream);
  if (err != cudaSuccess) return err;

  const InputDesc in{W, P.scales, P.cscales, P.ngroups, m, n, P.bounded, P.lo, P.hi, P.hdr, status_dev};
  const size_t total = (size_t)m * n;
  prepass_kernel<<<(int)std::min<size_t>((total + 255) / 256, 152 * 8), 256, 0, stream>>>(in);
  sigma_kernel<<<1, 1, 0, stream>>>(in);
  {
    signed char* eA = reinterpret_cast<signed char*>(base + lay.expA);
    signed char* eB = reinterpret_cast<signed char*>(base + lay.expB);
    const size_t wA = (size_t)n * P.nchA, wB = (size_t)m * P.nchB;  // one warp per (row, chunk)
    factor_exp_kernel<<<(unsigned)((wA + 7) / 8), 256, 0, stream>>>(LA, n, P.nchA, eA);
    factor_exp_kernel<<<(unsigned)((wB + 7) / 8), 256, 0, stream>>>(LB, m, P.nchB, eB);
    factor_digits_kernel<<<152 * 8, 256, 0, stream>>>(LA, n, P.nchA, P.ntA, eA, const_cast<__nv_bfloat16*>(P.FdA));
    factor_digits_kernel<<<152 * 8, 256, 0, stream>>>(LB, m, P.nchB, P.ntB, eB, const_cast<__nv_bfloat16*>(P.FdB));
  }
  {
    unsigned* bk = reinterpret_cast<unsigned*>(base + lay.buckets);
    const long long ntot = sweep::total_tasks(P.geom);
    const unsigned blocks = (unsigned)std::min<long long>((ntot + 255) / 256, 152 * 16);
    plan_count_kernel<<<blocks, 256, 0, stream>>>(P.geom, bk, reinterpret_cast<unsigned*>(base + lay.exp_col),
                                                  reinterpret_cast<unsigned*>(base + lay.exp_row), P.ncs);
    plan_scan_kernel<<<1, 1024, 0, stream>>>(bk, lay.nbuckets, reinterpret_cast<unsigned*>(base + lay.ntasks));
    plan_scatter_kernel<<<blocks, 256, 0, stream>>>(P.geom, bk, reinterpret_cast<int*>(base + lay.list));
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (kernel_ms) {
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0, stream);
  }
  void* args[] = {&P};
  err = cudaLaunchCooperativeKernel((const void*)sweep_kernel, dim3(di.sms), dim3(kThreads), args, kSmemBytes,
                                    stream);
  if (kernel_ms) {
    cudaEventRecord(e1, stream);
    if (err == cudaSuccess) err = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
    *kernel_ms = ms;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
  }
  return err;
}

// Host-side check of the task plan (no GPU): every delayed update is carried
// by exactly one task (row terms from source tiles >= 3 back, column terms
// from bands >= 2 above), none carries an update the bands apply themselves,
// and in the ideal schedule every task's sources complete before its
// targets are needed.  stats: [0] tasks, [1] smallest slack in steps,
// [2] coverage errors.
int sweep_plan_check(int64_t m, int64_t n, int64_t* stats) {
  const Geom g = sweep::make_geom((int)m, (int)n);
  const int nps = T / sweep::kSliceLines;
  std::vector<int> rowcov((size_t)g.Mt * nps * g.Nt * g.Nt, 0);  // [band][ps][source tile][target tile]
  const int ncs = (int)((n + 7) / 8);
  std::vector<int> colcov((size_t)g.Mt * g.Mt * ncs, 0);  // [source band][target band][column slice]
  long long ntask = 0, minslack = (long long)1 << 40, errors = 0;
  const long long total = sweep::total_tasks(g);
  for (long long idx = 0; idx < total; ++idx) {
    const Task t = sweep::decode(g, idx);
    if (t.type == sweep::kEmpty) continue;
    ++ntask;
    minslack = std::min(minslack, sweep::need_time(t) - sweep::ready_time(t));
    if (t.type == sweep::kRowSlice || t.type == sweep::kRowChunk) {
      const int j0 = t.k0 / T, j1 = (t.k0 + t.kLen + T - 1) / T;
      for (int ps = t.ps0; ps < t.ps1; ++ps)
        for (int j = j0; j < j1; ++j)
          for (int tt = t.t0; tt < t.t1; ++tt) ++rowcov[(((size_t)t.a * nps + ps) * g.Nt + j) * g.Nt + tt];
    } else {
      const int b0 = t.k0 / T, b1 = (t.k0 + t.kLen + T - 1) / T;
      for (int sb = b0; sb < b1; ++sb)
        for (int tb = t.t0; tb < t.t1; ++tb)
          for (int cs = t.cs0; cs < t.cs1; ++cs) ++colcov[((size_t)sb * g.Mt + tb) * ncs + cs];
    }
  }
  for (int I = 0; I < g.Mt; ++I)
    for (int ps = 0; ps < nps; ++ps) {
      if (I * T + ps * sweep::kSliceLines >= m) continue;
      for (int j = 0; j < g.Nt; ++j)
        for (int tt = 0; tt < g.Nt; ++tt) {
          const int want = (tt - j >= sweep::kRowAluTiles) ? 1 : 0;
          if (rowcov[(((size_t)I * nps + ps) * g.Nt + j) * g.Nt + tt] != want) ++errors;
        }
    }
  for (int sb = 0; sb < g.Mt; ++sb)
    for (int tb = 0; tb < g.Mt; ++tb)
      for (int cs = 0; cs < ncs; ++cs) {
        const int want = (tb - sb >= 2) ? 1 : 0;
        if (colcov[((size_t)sb * g.Mt + tb) * ncs + cs] != want) ++errors;
      }
  stats[0] = ntask;
  stats[1] = ntask ? minslack : 0;
  stats[2] = errors;
  return errors == 0 ? 0 : 1;
}

}  // namespace bakron
