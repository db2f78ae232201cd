// sweep.cu -- the BaKron core as one persistent cooperative kernel on
// sm_103a: a band-by-band sweep of the anti-diagonals on the fp32 pipes
// (double-float), fed by delayed products on the tensor cores that the same
// kernel runs from a queue of ready tasks.
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
//     the band below; publishes the band's progress and puts the products
//     whose sources it completed into the ready queue.
//   loader warp: stages, ahead of the ring, each anti-diagonal's inputs and
//     delayed sums, and the previous band's published G columns (column
//     terms at band distance 1, which the ring folds in).
// Everything farther is carried by tensor-core products that the product
// warps of every CTA take from the ready queue in the order their sources
// completed: slices (8 source lines, K = 32) for the middle distances,
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
constexpr int kRing = 44;         // columns kept in the shared rings of rounded values (E, v, Wq, G)
constexpr int kBag = 48;          // band-above G columns kept in shared memory
constexpr int kFar = 32;          // anti-diagonals of staged inputs and delayed sums
constexpr int kWoWarp = 8;        // write-out warp
constexpr int kLoadWarp = 9;      // loader warp: inputs, delayed sums and the band above's G, staged ahead
constexpr int kBandWarps = 10;
constexpr int kEpiWarp0 = 10;     // epilogue warps 10..13; warp w reads tensor-memory lane quarter w % 4
constexpr int kMmaWarp = 14;
constexpr int kSchedWarp = 15;
constexpr int kWarps = 16;        // 4 warps per SM sub-partition: 128 registers each
constexpr int kThreads = kWarps * 32;
constexpr int kTcM = 128;         // target lines per product group
constexpr int kPubBufs = 8;       // step publications kept (see the ring barrier)
constexpr long long kWaitNs = 1000000000ll;  // one second

// Named barriers (0 is __syncthreads).  The ring warps' step barrier
// rotates through kRingBars ids, step s using kBarRing + (s mod kRingBars).
// The warp that rounds step s arrives early at the barriers of steps
// s + 1 .. s + kRingBars - 1 (bar.arrive) and next waits at step
// s + kRingBars's: its deferred work (the rest of its fold, the ring shift,
// the refresh of its next anti-diagonal) then has kRingBars steps instead
// of one.  A barrier id is reused only kRingBars steps later, and passing a
// step's barrier requires every warp to have arrived at the step before,
// so no arrival can land in the wrong phase.  During the steps it skips,
// the warp reads a step's publication only after the step's rounding is
// flagged (rounded), and the kPubBufs publication buffers are reused only
// after every warp has synchronized past the step that read them.
constexpr int kBarRing = 1, kRingBars = 4, kBarBand = kBarRing + kRingBars;
__device__ __forceinline__ int ring_bar(int s) { return kBarRing + (s & (kRingBars - 1)); }

struct SweepParams {
  const float* W;
  const float* LA;
  const float* LB;
  const float* scales;   // m x ngroups, or null
  const float* cscales;  // n, or null
  int group, ngroups;
  int32_t* V;
  float* Wq;
  long long* Xc;         // column-direction delayed sums (fixed point): entry (r, q) at q * m + r
  long long* Gc;         // row-direction delayed sums, m x n
  float2* Gt;            // published G: [band][column][32 rows]
  __nv_bfloat16* EB;     // E digits in source blocks [band][tile][digit][32 rows x 32 columns, core-matrix order]
  __nv_bfloat16* GB;     // G digits in source blocks [column tile][band][digit][32 columns x 32 rows]
  const signed char* expA;
  const signed char* expB;
  const __nv_bfloat16* FdA;
  const __nv_bfloat16* FdB;
  int ntA, ntB, nchA, nchB;
  int* progress;         // [Mt]: last band step written out (-1: none)
  // Completion counters, each started at minus the number of products that
  // serve its targets (so a target's delayed sums are complete once its
  // counter, read as a signed int, is >= 0):
  unsigned* cnt_col;     // [Mt][ncs] column-direction products per (band, 8 columns)
  unsigned* cnt_row;     // [Mt][Nt][4] row-direction products per (band, tile, 8 rows)
  const unsigned* rdy_end;  // [Mt * steps]: end of band I's ready list up to step s, at I * steps + s
  const int* rdy_list;   // canonical task indices per (source band, ready step), in that order
  unsigned* arrive;      // [column chunks]: source bands that have completed each one's sources
  int* qslot;            // the ready queue: canonical task indices (-1: not yet filled)
  unsigned qcap;         // its length (the canonical task count)
  const unsigned* ntasks;  // tasks in the plan (each enters the ready queue once)
  long long cc_base;     // canonical index of the first column chunk
  Header* hdr;
  int32_t* status;
  int m, n, Mt, Nt, ncs, bounded, lo, hi;
  Geom geom;
};

// A task as the product warps use it: its plan entry and derived sizes.
struct TaskView {
  Task t;
  bool row;      // row-direction task (factor L_A, sources E, plane Gc) or column-direction (L_B, G, Xc)
  int lb;        // first of the task's source lines within the 32-line source block
  int nslab;     // slabs per group (source tiles or bands along K)
  int ngroups;
  int c;         // factor chunk of the source K range
  int s0;        // first slab within the chunk
  int tgt0;      // first target line (factor row)
  int tgt_end;   // one past the last target line
};

__device__ __noinline__ TaskView view_of(const SweepParams& P, long long idx) {
  TaskView v;
  v.t = sweep::decode(P.geom, idx);
  v.row = v.t.type == sweep::kRowSlice || v.t.type == sweep::kRowChunk;
  v.lb = v.t.line0 % T;
  v.nslab = (v.t.kLen + kSlab - 1) / kSlab;
  const int dlim = v.row ? P.n : P.m;
  v.tgt0 = T * v.t.t0;
  v.tgt_end = min(T * v.t.t1, dlim);
  v.ngroups = (v.tgt_end - v.tgt0 + kTcM - 1) / kTcM;
  v.c = v.t.k0 / CK;
  v.s0 = (v.t.k0 % CK) / kSlab;
  return v;
}

// ------------------------------------------------------------- shared memory
struct ProdSmem {
  struct Buf {
    __nv_bfloat16 A[kDigF][kTcM * kSlab];  // factor digit slab (core-matrix layout, SBO 512 B)
    __nv_bfloat16 B[kDigD * T * kSlab];     // source block: 6 digits x 32 lines x 32 (SBO 512 B)
  } buf[2];
  int4 gdesc[2];        // group in tensor-memory half h: (task, group, last of task, -)
  TaskView gview[2];    // and its task, decoded once by the scheduler lane
  int unit[2];          // unit in buffer p: 1 first slab of its group, 2 last slab, 4 stop
  uint64_t full[2], empty[2], gfull[2], gempty[2];
  uint64_t gready[2];   // gdesc[h] written (scheduler lane's arrival, a release the epilogue acquires)
  uint64_t edone;       // the epilogue threads' updates of a task are fenced (128 arrivals per task)
  uint32_t tmem_base;
};

struct BandSmem {
  float LA[3][3 * T][T];        // L_A panels [source tile mod 3]: rows 32j .. 32j+95, columns 32j .. 32j+31
  float LB0[T][T];              // L_B[band, band]
  float LB1[T][T + 1];          // L_B[band, band - 1]
  float2 sE[kPubBufs][T];       // the last rounded anti-diagonals' errors, by row
  float2 sG[kPubBufs][T];       // and row transforms
  float4 EV[kRing][T];          // (E hi, E lo, v, Wq) by (column mod kRing, row)
  float2 Gr[kRing][T];          // G by (column mod kRing, row)
  float BAh[kBag][T + 1];       // G of band I - 1 by (column mod kBag, row): high words
  float BAl[kBag][T + 1];       // and low words
  float2 FC[kFar][T];           // W0 + column-direction delayed sum, by (anti-diagonal mod kFar, row)
  float2 FR[kFar][T];           // row-direction delayed sum
  float FS[kFar][T];            // entry scale
  int rounded;                  // last band step rounded
  int written;                  // last band step written out
  int bag_done;                 // last band-above column staged
  int far_done;                 // last anti-diagonal staged
  int panel;                    // last L_A panel loaded
};

constexpr size_t kProdSmemBytes = (sizeof(ProdSmem) + 15) / 16 * 16;  // the band state after it stays 16-byte aligned
constexpr size_t kSmemBytes = kProdSmemBytes + sizeof(BandSmem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM: at most 227 KB of shared memory");

// ------------------------------------------------------------------ waits
__device__ __forceinline__ long long gtimer() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_relaxed_u(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Acquire fence: every load after it sees the writes released before the
// relaxed observations made before it.
__device__ __forceinline__ void fence_acquire() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ bool aborted(const Header* h) { return *(volatile const int*)&h->abort != 0; }

__device__ __noinline__ void raise_timeout(const SweepParams& P) {
  atomicOr(P.status, BAKRON_DEV_TIMEOUT);
  atomicExch(&P.hdr->abort, 1);
}

// Polls between two looks at the abort flag and the clock in the waits
// below: the abort flag lives in global memory, and reading it on every poll
// would put an L2 round trip between the flag turning and the waiter seeing
// it.
constexpr unsigned kPollsPerCheck = 256;

// Spins until *p >= v with relaxed loads; the caller fences before reading
// what the value guards.  False once the wait ran out or the kernel aborts.
__device__ bool wait_relaxed_ge(const SweepParams& P, const int* p, int v) {
  if (ld_relaxed(p) >= v) return true;
  const long long t0 = gtimer();
  for (unsigned it = 1; ld_relaxed(p) < v; ++it) {
    if (it % kPollsPerCheck == 0) {
      if (aborted(P.hdr)) return false;
      if (gtimer() - t0 > kWaitNs) {
        raise_timeout(P);
        return false;
      }
    }
    __nanosleep(64);
  }
  return true;
}
// The same on a shared-memory counter written by other warps of the CTA.
__device__ bool wait_shared_ge(const SweepParams& P, const int* p, int v) {
  if (*(volatile const int*)p >= v) return true;
  const long long t0 = gtimer();
  for (unsigned it = 1; *(volatile const int*)p < v; ++it) {
    if (it % kPollsPerCheck == 0) {
      if (aborted(P.hdr)) return false;
      if (gtimer() - t0 > kWaitNs) {
        raise_timeout(P);
        return false;
      }
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


// The six bf16 digits of a solver value (put_digits) into a source block:
// line l, depth k of a 32 x 32 block, digit b at element b * 1024 +
// (l / 8) * 256 + (k / 8) * 64 + (l % 8) * 8 + k % 8 -- the K-major
// core-matrix order of the products' B operand (8 x 16-byte core matrices,
// leading offset 128 B, stride offset 512 B), so that a block is one bulk
// copy and six stacked digits are one operand.
__device__ __forceinline__ void put_block_digits(__nv_bfloat16* blk, int l, int k, float2 x, float sc) {
  put_digits(blk, 1024, (size_t)((l >> 3) * 256 + (k >> 3) * 64 + (l & 7) * 8 + (k & 7)), x, sc);
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
  float se0 = 1.f, rcp0 = 1.f;  // scale of slot 0's entry

  // Slot 0 now holds anti-diagonal k: add its input and delayed sums (staged
  // by the loader warp) and its band-above sum.
  auto refresh0 = [&](int k) {
    const int q = k - p;
    wait_shared_ge(P, &sb.far_done, k);
    if (I > 0) wait_shared_ge(P, &sb.bag_done, min(k, n - 1));
    const int f = k % kFar;
    se0 = sb.FS[f][p];
    rcp0 = __frcp_rn(se0);
    if (vr && q >= 0 && q < n) {
      OffsetAcc c{cH[0], cL[0]}, rr{rH[0], rL[0]};
      c.mac(1.f, sb.FC[f][p]);
      if (I > 0) {  // band I - 1: sum_i L_B[r, 32(I-1) + i] G[32(I-1) + i, q]
        const int slot = q % kBag;
#pragma unroll 8
        for (int i = 0; i < T; ++i) c.mac(sb.LB1[p][i], make_float2(sb.BAh[slot][i], sb.BAl[slot][i]));
      }
      rr.mac(1.f, sb.FR[f][p]);
      cH[0] = c.H;
      cL[0] = c.L;
      rH[0] = rr.H;
      rL[0] = rr.L;
    }
  };
  // Folds the errors and row transforms published by step ps (anti-diagonal
  // ps) into slots [i0, i1).
  auto fold = [&](int ps, int i0, int i1) {
    const int buf = ps & (kPubBufs - 1);
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

  refresh0(k0);  // slot 0 = anti-diagonal w
  int skip_until = -1;  // this warp arrived early at the barriers of the steps up to here

  for (int s = 0; s < steps; ++s) {
    if (s > skip_until) {
      bar_sync(ring_bar(s), kRingWarps * 32);
    } else if (s >= 1) {
      wait_shared_ge(P, &sb.rounded, s - 1);  // step s - 1's publication is written
    }
    // The source L_A panel of the newest source column s - 1 (row 0's).
    if (s >= 1 && ((s - 1) & (T - 1)) == 0 && ((s - 1) >> 5) < P.Nt) wait_shared_ge(P, &sb.panel, (s - 1) >> 5);
    // Step s - 1's errors go into slot 0 first (the owner rounds it next),
    // then into the other slots; one copy of the fold serves both cases.
    const bool own = k0 == s;
    if (s >= 1) fold(s - 1, 0, 1);
    if (own) {
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
      // The rings' slots of column q were written out at least kRing - 32 steps ago.
      wait_shared_ge(P, &sb.written, s - (kRing - T));
      const int buf = s & (kPubBufs - 1);
      sb.sE[buf][p] = e;
      sb.sG[buf][p] = g;
      if (q >= 0 && q < n) {
        sb.EV[q % kRing][p] = make_float4(e.x, e.y, v, wq);
        sb.Gr[q % kRing][p] = g;
      }
      __syncwarp();
      __threadfence_block();
      if (p == 0) *(volatile int*)&sb.rounded = s;
      skip_until = min(s + kRingBars - 1, steps - 1);
      for (int t = s + 1; t <= skip_until; ++t) bar_arrive(ring_bar(t), kRingWarps * 32);
    }
    if (s >= 1) fold(s - 1, 1, kSlots);
    if (own) {
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
      if (k0 < steps) refresh0(k0);
    }
  }
}

// Puts the tasks whose sources band I completed up to step s (its list
// entries [next, end(I, s))) into the ready queue.  A column chunk has
// several source bands and goes in with the last of them to arrive.  Each
// lane takes one entry at a time; one atomic reserves the warp's queue
// positions.  Called by the write-out warp right after it published step s.
// Each entry is a release store (and each arrival an acquire-release
// atomic): the source writes of this band, and through the arrivals those
// of the other source bands, are visible before the entry is.
__device__ void enqueue_ready(const SweepParams& P, int I, int s, unsigned& next) {
  const int lane = threadIdx.x & 31;
  const int steps = P.n + T - 1;
  const unsigned end = __ldg(P.rdy_end + (size_t)I * steps + s);
  if (next >= end) return;
  __syncwarp();
  for (unsigned b = next; b < end; b += 32) {
    const unsigned e = b + lane;
    int id = -1;
    bool go = false;
    if (e < end) {
      id = __ldg(P.rdy_list + e);
      if (id >= P.cc_base) {
        const long long local = id - P.cc_base;
        const int h = (int)(local / ((long long)P.geom.colParts * P.Nt));
        const int nsrc = min(sweep::kChunk * h + sweep::kChunk, P.Mt) - sweep::kChunk * h;
        unsigned old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(P.arrive + local) : "memory");
        go = old + 1 == (unsigned)nsrc;
      } else {
        go = true;
      }
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, go);
    unsigned pos = 0;
    if (lane == 0 && ballot) pos = atomicAdd(&P.hdr->queue_tail, (unsigned)__popc(ballot));
    pos = __shfl_sync(0xffffffffu, pos, 0);
    const unsigned at = pos + __popc(ballot & ((1u << lane) - 1u));
    if (go && at < P.qcap) st_release(P.qslot + at, id);
  }
  next = end;
}

// The write-out warp of band I: V, Wq and the digits of E for every row
// tile a row completes, G (published and as digits) for every column the
// band completes, the L_A panels ahead of the sweep, and the band's progress.
// Every decision of this warp is taken by lane 0 and broadcast.
__device__ void band_writeout(const SweepParams& P, BandSmem& sb, int I, float sigma) {
  const int lane = threadIdx.x & 31;
  const int n = P.n, steps = n + T - 1;
  // Ready-list position of the band's next task to enqueue.
  unsigned rdy_next = I > 0 ? __ldg(P.rdy_end + (size_t)I * steps - 1) : 0u;
  const float dsc = pow2f(7 - bound_exp(sigma));
  const int r0 = I * T;
  int issued_panel = 0, ready_panel = 0;  // panel 0 is loaded before the sweep starts
  for (int s = 0; s < steps; ++s) {
    // Panel j is first read at step 32j + 1.  Its slot's previous panel
    // (j - 3) serves source anti-diagonals up to 32j - 34, read at the
    // latest by a warp's deferred folds before its barrier of step
    // 32j - 33 + kRingBars; this iteration starts once step s - 1 is
    // rounded, so the copy may be issued at s = 32j - 32 + kRingBars and is
    // waited for at s = 32j - 8.
    if (issued_panel + 1 < P.Nt && s >= T * (issued_panel + 1) - T + kRingBars) {
      ++issued_panel;
      load_panel(P, sb, issued_panel);
    }
    if (ready_panel < issued_panel && s >= T * (ready_panel + 1) - 8) {
      cp_async_wait_all();
      __syncwarp();
      __threadfence_block();
      ready_panel = issued_panel;
      if (lane == 0) *(volatile int*)&sb.panel = ready_panel;
    }
    {  // wait for step s to be rounded
      const long long t0 = gtimer();
      for (unsigned it = 1;; ++it) {
        int go = 0;  // 1: step s is rounded (or the kernel is aborting), 2: the wait ran out
        if (lane == 0) {
          if (*(volatile int*)&sb.rounded >= s)
            go = 1;
          else if (it % kPollsPerCheck == 0)
            go = aborted(P.hdr) ? 1 : (gtimer() - t0 > kWaitNs ? 2 : 0);
        }
        go = __shfl_sync(0xffffffffu, go, 0);
        if (go == 2 && lane == 0) raise_timeout(P);
        if (go) break;
        __nanosleep(64);
      }
    }
    // Row tiles completed at step s: row p completes tile j when it rounds
    // column min(32j + 31, n - 1).
#pragma unroll 1
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
      float2 e = make_float2(0.f, 0.f);  // past the last column: zero digits (the products' K padding)
      if (q < n) {
        const float4 ev4 = sb.EV[q % kRing][p];
        const size_t o = (size_t)(r0 + p) * n + q;
        P.V[o] = (int32_t)ev4.z;
        P.Wq[o] = ev4.w;
        e = make_float2(ev4.x, ev4.y);
      }
      put_block_digits(P.EB + ((size_t)I * P.Nt + j) * (kDigD * 1024), p, lane, e, dsc);
    }
    // The column completed at step s (row 31 rounded it).
    const int c = s - (T - 1);
    if (c >= 0 && c < n) {
      const float2 g = sb.Gr[c % kRing][lane];  // zero for rows past the last (the products' K padding)
      P.Gt[((size_t)I * n + c) * T + lane] = g;
      put_block_digits(P.GB + ((size_t)(c / T) * P.Mt + I) * (kDigD * 1024), c % T, lane, g, dsc);
    }
    __syncwarp();
    if (lane == 0) *(volatile int*)&sb.written = s;
    // Publish: the warp's stores happen before lane 0's release (warp
    // barrier), and the release makes them visible with the new progress.
    if ((s & 3) == 3 || s == steps - 1) {
      if (lane == 0) st_release(P.progress + I, s);
      enqueue_ready(P, I, s, rdy_next);
    }
  }
}

// The loader warp of band I, running ahead of the ring warps:
//  * band-above G: column c of band I - 1 goes to slot c mod kBag once band
//    I - 1 has written it out (its step c + 31) and the slot's previous
//    column (c - kBag) is consumed -- row p folds column c' at the refresh
//    of anti-diagonal c' + p, done by the warp that rounds c' + p - 8 before
//    its barrier of step c' + p - 8 + kRingBars, so all rows did once step
//    c' + 23 + kRingBars is rounded (kBagFree);
//  * for anti-diagonal k (entries (p, k - p)), once every product serving
//    those entries has counted its completion: W0 plus the column-direction
//    delayed sum, the row-direction delayed sum and the entry scale, to slot
//    k mod kFar.  The ring refreshes anti-diagonal k after rounding k - 8,
//    before its barrier of step k - 8 + kRingBars; so the slot's previous
//    anti-diagonal (k - kFar) is consumed once step k - kFar - 8 + kRingBars
//    is rounded.  The loader stays at most kFar anti-diagonals ahead of the
//    ring, which is enough while kRingBars <= 8.
// Counters and progress are polled with relaxed loads, a batch at a time,
// followed by one acquire fence before the data they guard is read.
// Every decision of this warp is taken by lane 0 or by a warp vote.
static_assert(kRingBars <= 8, "the loader's staging window assumes refreshes within 8 steps");
constexpr int kLoadBatch = 4;
constexpr int kBagFree = T - 1 - 8 + kRingBars;  // steps after column c' until its band-above slot is free

__device__ void band_loader(const SweepParams& P, BandSmem& sb, int I, float sigma) {
  const int lane = threadIdx.x & 31, p = lane;
  const int n = P.n, steps = n + T - 1;
  const int r = I * T + p;
  const bool vr = r < P.m;
  const float from_units = pow2f(fixed_unit_exp(sigma));
  const unsigned* cnt_col_band = P.cnt_col + (size_t)I * P.ncs;
  const unsigned* cnt_row_band = P.cnt_row + (size_t)I * P.Nt * 4 + (p >> 3);
  const float* srow = P.scales ? P.scales + (size_t)r * P.ngroups : nullptr;
  int next_bag = I > 0 ? 0 : n, seen = -1;
  int next_k = 0;
  long long idle_since = 0;
  unsigned idle_polls = 0;  // loader passes in a row that staged nothing
  while (next_k < steps || next_bag < n) {
    int rd = 0;
    if (lane == 0) rd = *(volatile int*)&sb.rounded;
    const int rounded = __shfl_sync(0xffffffffu, rd, 0);
    bool did = false;
    // Band-above columns: up to kLoadBatch at a time, loads issued together.
    if (next_bag < n && next_bag - kBag + kBagFree <= rounded) {
      if (seen < next_bag + T - 1) {
        int pr = 0;
        if (lane == 0) pr = ld_relaxed(P.progress + (I - 1));
        const int now = __shfl_sync(0xffffffffu, pr, 0);
        if (now > seen) {
          fence_acquire();
          seen = now;
        }
      }
      int c1 = next_bag;
      while (c1 < n && c1 < next_bag + kLoadBatch && c1 - kBag + kBagFree <= rounded && c1 + T - 1 <= seen) ++c1;
      if (c1 > next_bag) {
        float2 g[kLoadBatch];
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i)
          if (next_bag + i < c1) g[i] = __ldcg(P.Gt + ((size_t)(I - 1) * n + next_bag + i) * T + lane);
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i)
          if (next_bag + i < c1) {
            sb.BAh[(next_bag + i) % kBag][lane] = g[i].x;
            sb.BAl[(next_bag + i) % kBag][lane] = g[i].y;
          }
        __syncwarp();
        __threadfence_block();
        if (lane == 0) *(volatile int*)&sb.bag_done = c1 - 1;
        next_bag = c1;
        did = true;
      }
    }
    // Inputs and delayed sums of the next batch of anti-diagonals: every
    // counter of the batch read at once (relaxed); the leading anti-diagonals
    // whose serving products have all counted are staged after one acquire
    // fence, their data loads issued together.
    const int kend = min(min(steps, next_k + kLoadBatch), rounded + kFar + 1);
    if (next_k < kend) {
      int nready = 0;  // leading anti-diagonals of the batch that are ready
      {
        int cc[kLoadBatch], cr[kLoadBatch];
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i) {
          const int q = next_k + i - p;
          cc[i] = cr[i] = 0;
          if (next_k + i < kend && vr && q >= 0 && q < n) {
            cc[i] = ld_relaxed(reinterpret_cast<const int*>(cnt_col_band + (q >> 3)));
            cr[i] = ld_relaxed(reinterpret_cast<const int*>(cnt_row_band + (q >> 5) * 4));
          }
        }
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i)
          if (__all_sync(0xffffffffu, (cc[i] | cr[i]) >= 0) && nready == i) nready = i + 1;
      }
      const int k1 = min(kend, next_k + nready);
      if (k1 > next_k) {
        fence_acquire();
        float wv[kLoadBatch], rv[kLoadBatch], tv[kLoadBatch];
        long long xv[kLoadBatch], gv[kLoadBatch];
        // Scale group of the batch's first column of this row, then one
        // column further per anti-diagonal (no division per entry).
        const int q0 = max(next_k - p, 0);
        int grp = q0 / P.group, rem = q0 - grp * P.group;
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i) {
          const int q = next_k + i - p;
          wv[i] = 0.f;
          rv[i] = tv[i] = 1.f;
          xv[i] = gv[i] = 0;
          if (next_k + i < k1 && vr && q >= 0 && q < n) {
            wv[i] = __ldg(P.W + (size_t)r * n + q);
            xv[i] = __ldcg(P.Xc + (size_t)q * P.m + r);
            gv[i] = __ldcg(P.Gc + (size_t)r * n + q);
            if (srow) rv[i] = __ldg(srow + grp);
            if (P.cscales) tv[i] = __ldg(P.cscales + q);
          }
          if (q >= 0 && ++rem == P.group) {
            rem = 0;
            ++grp;
          }
        }
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i) {
          if (next_k + i < k1) {
            const int f = (next_k + i) % kFar;
            sb.FC[f][p] = df_add(make_float2(wv[i], 0.f), df_from_fixed(xv[i], from_units));
            sb.FR[f][p] = df_from_fixed(gv[i], from_units);
            sb.FS[f][p] = __fmul_rn(rv[i], tv[i]);  // fp32(R[r, q / group] t[q]); 1 where absent
          }
        }
        __syncwarp();
        __threadfence_block();
        if (lane == 0) *(volatile int*)&sb.far_done = k1 - 1;
        next_k = k1;
        did = true;
      }
    }
    if (did) {
      idle_polls = 0;
    } else {
      int out = 0;
      if (++idle_polls == 1) idle_since = gtimer();
      if (lane == 0 && idle_polls % 64 == 0) out = (aborted(P.hdr) || gtimer() - idle_since > kWaitNs) ? 1 : 0;
      out = __shfl_sync(0xffffffffu, out, 0);
      if (out) {  // nothing could be staged for a second: give up (or the kernel is aborting)
        if (lane == 0 && !aborted(P.hdr)) raise_timeout(P);
        if (lane == 0) {
          *(volatile int*)&sb.bag_done = n;
          *(volatile int*)&sb.far_done = steps;
        }
        break;
      }
      __nanosleep(200);
    }
  }
}

// --------------------------------------------------------------- product role
// A stream of slab units through two shared-memory buffers, three roles:
//  * the scheduler lane fetches tasks in queue order, waits until each
//    one's sources are complete, and for every (group, slab) of the task
//    bulk-copies the factor digit slab (A: 128 target lines x 32, five
//    digits) and the source block (B: 32 lines x 32, six digits, already in
//    the core-matrix layout) into a free buffer;
//  * the MMA lane multiplies each unit into the group's tensor-memory half
//    (five products per 16-deep step: factor digit a against source digits
//    0 .. 5-a stacked along N, landing on levels a + b);
//  * the epilogue warps turn each finished group's six levels into
//    fixed-point updates of the planes, and after a task's last group count
//    its completion for each of its targets.
// Units of consecutive tasks follow each other without a pause; mbarriers
// carry every hand-off, and every wait is bounded.
// Source block of slab sl of a task: row tasks the E digits of (band, source
// tile), column tasks the G digits of (column tile, source band); 6 digits x
// 2 KB, contiguous.
__device__ __forceinline__ const __nv_bfloat16* source_block(const SweepParams& P, const TaskView& v, int sl) {
  const int k_tile = v.t.k0 / T + sl;
  const size_t blk = v.row ? ((size_t)v.t.a * P.Nt + k_tile) : ((size_t)(v.t.line0 / T) * P.Mt + k_tile);
  return (v.row ? P.EB : P.GB) + blk * (kDigD * 1024);
}

__device__ void product_role(const SweepParams& P, ProdSmem& sm, float sigma) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  bool broken = false;

  if (warp == kSchedWarp) {
    if (lane == 0) {
      uint32_t zz = 0, gg = 0;  // slab units and groups issued
      const unsigned ntasks = *P.ntasks;
      // Ready-queue position of the next task, taken one task ahead so that
      // its atomic is in flight while the current task is served.  Every
      // task in the queue is ready, and every task of the plan enters it
      // once, so each position is filled in time (the wait is bounded).
      unsigned qi = atomicAdd(&P.hdr->queue_head, 1u);
      for (;;) {
        int idx = -1;
        if (!broken && qi < ntasks) {  // (the wait returns false once the kernel aborts)
          if (wait_relaxed_ge(P, P.qslot + qi, 0)) {
            idx = ld_relaxed(P.qslot + qi);
            qi = atomicAdd(&P.hdr->queue_head, 1u);
            // The sources were written by other CTAs' generic stores; the
            // bulk copies below read them through the async proxy.
            fence_acquire();
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
        }
        const TaskView v = view_of(P, idx >= 0 ? idx : 0);
        const int ngroups = idx >= 0 ? v.ngroups : 1;
        const __nv_bfloat16* Fd = v.row ? P.FdA : P.FdB;
        const int nt = v.row ? P.ntA : P.ntB;
        for (int gi = 0; gi < ngroups; ++gi) {
          const uint32_t h = gg & 1;
          // gdesc[h] and the tensor-memory half h are free once the
          // epilogue finished group gg - 2.
          if (gg >= 2) mbar_wait(&sm.gempty[h], ((gg >> 1) - 1) & 1u, broken);
          sm.gdesc[h] = make_int4(idx, gi, gi == ngroups - 1, 0);
          sm.gview[h] = v;
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.gready[h])) : "memory");
          const int nsl = idx >= 0 ? v.nslab : 1;
          for (int sl = 0; sl < nsl; ++sl) {
            const uint32_t pb = zz & 1;
            if (zz >= 2) mbar_wait(&sm.empty[pb], ((zz >> 1) - 1) & 1u, broken);
            if (idx < 0 || broken) {  // stop: a unit without copies
              sm.unit[pb] = 4;
              asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.full[pb])) : "memory");
              ++zz;
              break;
            }
            sm.unit[pb] = (sl == 0 ? 1 : 0) | (sl == nsl - 1 ? 2 : 0);
            const int t0 = (v.tgt0 + gi * kTcM) / T;
            const int ntg = min(kTcM / T, nt - t0);
            const uint32_t abytes = (uint32_t)ntg * 2048u;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(&sm.full[pb])),
                         "r"(abytes * kDigF + (uint32_t)(kDigD * 2048))
                         : "memory");
            const size_t cs = (size_t)v.c * (CK / kSlab) + v.s0 + sl;
#pragma unroll
            for (int a = 0; a < kDigF; ++a) {
              const unsigned char* src =
                  reinterpret_cast<const unsigned char*>(Fd) + ((cs * kDigF + a) * nt + t0) * 2048;
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                      smem_u32(sm.buf[pb].A[a])),
                  "l"(src), "r"(abytes), "r"(smem_u32(&sm.full[pb]))
                  : "memory");
            }
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                    smem_u32(sm.buf[pb].B)),
                "l"(source_block(P, v, sl)), "r"((uint32_t)(kDigD * 2048)), "r"(smem_u32(&sm.full[pb]))
                : "memory");
            ++zz;
          }
          ++gg;
          if (idx < 0 || broken) break;
        }
        if (idx < 0 || broken) break;
      }
      // Leave no bulk copy in flight: both buffers' last fills have landed
      // once their full barriers completed (bounded wait).
      bool gone = false;
      for (uint32_t pb = 0; pb < 2; ++pb) {
        const uint32_t uses = (zz + 1 - pb) / 2;
        if (uses > 0) mbar_wait(&sm.full[pb], (uses - 1) & 1u, gone);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t tmem = sm.tmem_base;
      uint32_t zz = 0, gg = 0;
      for (;;) {
        const uint32_t pb = zz & 1;
        mbar_wait(&sm.full[pb], (zz >> 1) & 1u, broken);
        const int f = broken ? 4 : sm.unit[pb];
        const uint32_t h = gg & 1;
        if (f & 4) {  // stop: wake the epilogue on the next group's barrier
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.gfull[h])) : "memory");
          break;
        }
        if ((f & 1) && gg >= 2) mbar_wait(&sm.gempty[h], ((gg >> 1) - 1) & 1u, broken);
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < kSlab / 16; ++j) {
          const uint64_t db = umma_sdesc(smem_u32(sm.buf[pb].B) + (uint32_t)(2 * j) * 128u, 128u, 512u);
#pragma unroll
          for (int a = 0; a < kDigF; ++a) {
            const uint64_t da = umma_sdesc(smem_u32(sm.buf[pb].A[a]) + (uint32_t)(2 * j) * 128u, 128u, 512u);
            const uint32_t acc = ((f & 1) && j == 0 && a == 0) ? 0u : 1u;
            umma_bf16(tmem + (uint32_t)(256 * h + 32 * a), da, db, umma_idesc_bf16(kTcM, T * (kDigD - a)), acc);
          }
        }
        umma_commit(&sm.empty[pb]);
        if (f & 2) {
          umma_commit(&sm.gfull[h]);
          ++gg;
        }
        ++zz;
      }
    }
    __syncwarp();
  } else {  // epilogue warps
    const uint32_t tmem = sm.tmem_base;
    const int qd = warp & 3;          // tensor-memory lane quarter this warp may read
    const int rr = 32 * qd + lane;    // target line within the group
    const int eD = bound_exp(sigma);
    const int fexp_unit = fixed_unit_exp(sigma);
    uint32_t gg = 0, ntask_done = 0;
    for (;;) {
      const uint32_t h = gg & 1;
      mbar_wait(&sm.gready[h], (gg >> 1) & 1u, broken);
      mbar_wait(&sm.gfull[h], (gg >> 1) & 1u, broken);
      const int4 d = sm.gdesc[h];
      if (d.x < 0 || broken) break;
      tc_fence_after();
      const TaskView v = sm.gview[h];
      const int gi = d.y;
      const int tgt = v.tgt0 + gi * kTcM + rr;  // factor row = target line
      const bool rok = tgt < v.tgt_end;
      const signed char* fexp = v.row ? P.expA : P.expB;
      const int nch = v.row ? P.nchA : P.nchB;
      const int er = rok ? (int)fexp[(size_t)tgt * nch + v.c] : -100;
      const int ex = er + eD - 14 - fexp_unit;
      const float sc = ex >= -126 ? pow2f(min(ex, 127)) : 0.f;
      unsigned long long* plane = reinterpret_cast<unsigned long long*>(v.row ? P.Gc : P.Xc);
      // Both planes are indexed [source line][target line]: Gc by (source
      // row, target column), Xc by (source column, target row), so the 32
      // lanes of a warp (consecutive targets) update 256 contiguous bytes.
      // Source line = line0 + (q - lb).
      const size_t ostep = v.row ? (size_t)P.n : (size_t)P.m;
      const size_t obase = (size_t)v.t.line0 * ostep + tgt;
#pragma unroll 1
      for (int qb = v.lb; qb < v.lb + v.t.nLines; qb += 8) {
        float lv[kLevels][8];
#pragma unroll
        for (int l = 0; l < kLevels; ++l)
          tmem_ld(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(256 * h + T * l + qb), lv[l]);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          // levels 0..2 exactly, the rest (below 2^-24 of the total) in one fp32 sum
          float2 y = two_sum(lv[0][j], lv[1][j] * 0x1p-8f);
          const float2 y2 = two_sum(y.y, lv[2][j] * 0x1p-16f);
          const float tail = lv[3][j] * 0x1p-24f + lv[4][j] * 0x1p-32f + lv[5][j] * 0x1p-40f;
          y = two_sum(y.x, y2.x);
          y = two_sum(y.x, y.y + (y2.y + tail));
          const int q = qb - v.lb + j;
          if (rok && q < v.t.nLines)
            atomicAdd(plane + obase + (size_t)q * ostep, (unsigned long long)df_to_fixed(y, sc));
        }
      }
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.gempty[h])) : "memory");
      if (d.z) {  // the task's last group: count it per target
        // All 128 epilogue threads arrive on edone after their updates (an
        // arrive releases at CTA scope) and wait for its phase (bounded), so
        // that no thread arrives for the next task before this task's phase
        // is complete.  The counting warp's reductions release at GPU scope;
        // a release is cumulative over what its thread has observed, so it
        // publishes the updates of all 128 threads, and only that warp waits
        // for them to be performed.
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.edone)) : "memory");
        mbar_wait(&sm.edone, ntask_done & 1u, broken);
        if (warp == kEpiWarp0) {  // one warp counts the task's completion
          if (v.row) {
            const int nps = v.t.ps1 - v.t.ps0;
            const int tot = (v.t.t1 - v.t.t0) * nps;
            for (int e = lane; e < tot; e += 32) {
              const int t = v.t.t0 + e / nps, ps = v.t.ps0 + e % nps;
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
        ++ntask_done;
      }
      ++gg;
    }
  }
  if (broken) raise_timeout(P);
}

// -------------------------------------------------------------------- kernel
__global__ void __launch_bounds__(kThreads, 1) sweep_kernel(SweepParams P) {
  extern __shared__ __align__(1024) unsigned char sweep_smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sweep_smem_raw) + 1023) & ~uintptr_t(1023));
  ProdSmem& sm = *reinterpret_cast<ProdSmem*>(base);
  BandSmem& sb = *reinterpret_cast<BandSmem*>(base + kProdSmemBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float sigma = P.hdr->sigma;

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.empty[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.gfull[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;\n" ::"r"(smem_u32(&sm.gempty[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.gready[i])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;\n" ::"r"(smem_u32(&sm.edone)));
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
        sb.bag_done = I > 0 ? -1 : P.n;
        sb.far_done = -1;
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
      } else if (warp == kLoadWarp) {
        band_loader(P, sb, I, sigma);
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

// ------------------------------------------------------------ ready lists
// Every task of the plan (sweep_plan.h) is listed under each of its source
// bands at its ready step, the lists ordered by (band, step): a counting
// sort over the Mt x steps buckets.  After the scatter, bucket (I, s) holds
// the end of band I's entries up to step s, which is what the write-out
// warps read to enqueue.  The number of tasks serving each target is
// counted too.

__global__ void plan_count_kernel(Geom g, unsigned* bucket_cnt, unsigned* cnt_col, unsigned* cnt_row, int ncs,
                                  unsigned* ntasks) {
  const long long total = sweep::total_tasks(g);
  const int steps = g.n + T - 1;
  unsigned live = 0;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const Task t = sweep::decode(g, idx);
    if (t.type == sweep::kEmpty) continue;
    ++live;
    for (int b = t.srcBand0; b < t.srcBand1; ++b) atomicAdd(bucket_cnt + (size_t)b * steps + t.readyStep, 1u);
    if (t.type == sweep::kRowSlice || t.type == sweep::kRowChunk) {
      for (int tt = t.t0; tt < t.t1; ++tt)
        for (int ps = t.ps0; ps < t.ps1; ++ps) atomicSub(cnt_row + ((size_t)t.a * g.Nt + tt) * 4 + ps, 1u);
    } else {
      for (int b = t.t0; b < t.t1; ++b)
        for (int cs = t.cs0; cs < t.cs1; ++cs) atomicSub(cnt_col + (size_t)b * ncs + cs, 1u);
    }
  }
  live = __reduce_add_sync(0xffffffffu, live);
  if ((threadIdx.x & 31) == 0 && live) atomicAdd(ntasks, live);
}

// Exclusive scan of the bucket counts (one CTA).
__global__ void __launch_bounds__(1024) plan_scan_kernel(unsigned* bucket, long long nb) {
  __shared__ unsigned part[1024];
  const int tid = threadIdx.x;
  const long long per = (nb + 1023) / 1024;
  const long long b0 = tid * per, b1 = min(b0 + per, nb);
  unsigned s = 0;
  for (long long b = b0; b < b1; ++b) s += bucket[b];
  part[tid] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const unsigned x = tid >= o ? part[tid - o] : 0u;
    __syncthreads();
    part[tid] += x;
    __syncthreads();
  }
  unsigned run = tid ? part[tid - 1] : 0u;
  for (long long b = b0; b < b1; ++b) {
    const unsigned c = bucket[b];
    bucket[b] = run;
    run += c;
  }
}

__global__ void plan_scatter_kernel(Geom g, unsigned* bucket_off, int* list) {
  const long long total = sweep::total_tasks(g);
  const int steps = g.n + T - 1;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const Task t = sweep::decode(g, idx);
    if (t.type == sweep::kEmpty) continue;
    for (int b = t.srcBand0; b < t.srcBand1; ++b) {
      const unsigned pos = atomicAdd(bucket_off + (size_t)b * steps + t.readyStep, 1u);
      list[pos] = (int)idx;
    }
  }
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
  size_t plane, Gt, EB, GB, expA, expB, FdA, FdB, progress, qslot, cnt_col, cnt_row, buckets,
      ntasks, arrive, list, total;
  long long nbuckets;
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
  L.EB = off;
  off += align_up((size_t)g.Mt * g.Nt * kDigD * 2048);
  L.GB = off;
  off += align_up((size_t)g.Nt * g.Mt * kDigD * 2048);
  L.expA = off;
  off += align_up((size_t)n * nchA);
  L.expB = off;
  off += align_up((size_t)m * nchB);
  L.FdA = off;
  off += align_up(nchA * (CK / kSlab) * kDigF * ntA * 2048);
  L.FdB = off;
  off += align_up(nchB * (CK / kSlab) * kDigF * ntB * 2048);
  // From progress up to cnt_col: set to -1 before the solve; from cnt_col
  // up to list: zeroed.
  L.progress = off;
  off += align_up((size_t)g.Mt * sizeof(int));
  L.qslot = off;
  off += align_up((size_t)sweep::total_tasks(g) * sizeof(int));
  const size_t ncs = (size_t)((n + 7) / 8);
  L.cnt_col = off;
  off += align_up((size_t)g.Mt * ncs * sizeof(unsigned));
  L.cnt_row = off;
  off += align_up((size_t)g.Mt * g.Nt * 4 * sizeof(unsigned));
  L.nbuckets = (long long)g.Mt * (n + T - 1);
  L.buckets = off;
  off += align_up((size_t)L.nbuckets * sizeof(unsigned));
  L.ntasks = off;
  off += align_up(sizeof(unsigned));
  L.arrive = off;
  off += align_up((size_t)g.nCC * sizeof(unsigned));
  L.list = off;
  off += align_up((size_t)(g.nRS + g.nCS + g.nRC + sweep::kChunk * g.nCC) * sizeof(int));
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
  P.EB = reinterpret_cast<__nv_bfloat16*>(base + lay.EB);
  P.GB = reinterpret_cast<__nv_bfloat16*>(base + lay.GB);
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
  P.cnt_row = reinterpret_cast<unsigned*>(base + lay.cnt_row);
  P.rdy_end = reinterpret_cast<const unsigned*>(base + lay.buckets);
  P.rdy_list = reinterpret_cast<const int*>(base + lay.list);
  P.arrive = reinterpret_cast<unsigned*>(base + lay.arrive);
  P.qslot = reinterpret_cast<int*>(base + lay.qslot);
  P.qcap = (unsigned)sweep::total_tasks(P.geom);
  P.ntasks = reinterpret_cast<const unsigned*>(base + lay.ntasks);
  P.cc_base = P.geom.nRS + P.geom.nCS + P.geom.nRC;
  P.status = status_dev;
  P.m = m;
  P.n = n;
  P.Mt = P.geom.Mt;
  P.Nt = P.geom.Nt;
  P.ncs = (n + 7) / 8;
  P.bounded = al.bounded ? 1 : 0;
  P.lo = al.lo;
  P.hi = al.hi;

  // Zeroed state: status, header, the two planes, the counters, buckets and
  // arrivals; progress and the ready queue = -1.  (The source blocks need no clearing: the write-out warp
  // writes every entry a product reads along K, zeros past the matrix; lines
  // past the matrix only feed output columns that are never stored.)
  err = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(P.hdr, 0, sizeof(Header), stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(P.Xc, 0, 2 * lay.plane, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(base + lay.progress, 0xFF, lay.cnt_col - lay.progress, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(base + lay.cnt_col, 0, lay.list - lay.cnt_col, stream);
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
    plan_count_kernel<<<blocks, 256, 0, stream>>>(P.geom, bk, reinterpret_cast<unsigned*>(base + lay.cnt_col),
                                                  reinterpret_cast<unsigned*>(base + lay.cnt_row), P.ncs,
                                                  reinterpret_cast<unsigned*>(base + lay.ntasks));
    plan_scan_kernel<<<1, 1024, 0, stream>>>(bk, lay.nbuckets);
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
