// sweep_plan.h -- the task plan of the persistent band sweep (sweep.cu):
// which tensor-core product carries each delayed update, when its sources
// are complete, and which targets it serves.  Host and device share these
// functions: the device builds the per-band ready lists from them, and a host-side
// check (bakron_sweep_plan_check) verifies on the CPU that every delayed
// update is carried exactly once and before it is needed.
//
// "BaKron: Efficient Quantization with Kronecker-Factored Hessians":
//   App. B eq. (1): the updates from a finished set of entries to later
//     entries are one product L_B E L_A^T restricted to the later entries,
//     so they can be delayed and batched (Sec. 3.4, 3.5: the delayed,
//     batched updates of Algorithms 5 and 6);
//   Sec. 3.3: entry (i, j) affects only entries (p, q) with i <= p, j <= q.
//
// The matrix is cut into bands of T = 32 rows (band I: rows 32I .. 32I+31)
// and tiles of 32 columns.  A band is swept by one group of warps, one
// anti-diagonal of the band per step: at band step s, row p rounds column
// s - p.  With the row transform G = E L_A^T, the value rounded at (r, q) is
//   W0 + sum_{i < r} L_B[r, i] G[i, q]  +  sum_{j < q} E[r, j] L_A[q, j].
// Who adds which term, by the distance d between source and target:
//   row terms (same row, source tile j, target tile t = j + d):
//     d = 0, 1, 2   the band's own warps, as each error appears;
//     d >= 3        ROW_SLICE tasks (8 source rows x one source tile) up to
//                   tile 4 floor(j/4) + 6, ROW_CHUNK tasks (32 rows x a chunk
//                   of 4 source tiles) from tile 4h + 7 on (h = chunk);
//   column terms (same column, source band I', target band I = I' + d):
//     d = 0         the band's own warps;
//     d = 1         the band's own warps, from the published G of band
//                   I - 1 (staged by its loader warp);
//     d >= 2        COL_SLICE tasks (one source band x 8 columns) up to band
//                   4 floor(I'/4) + 5, COL_CHUNK tasks (a chunk of 4 source
//                   bands x one tile of columns) from band 4h' + 6 on.
// A task becomes ready when its source bands have passed a step (the last
// source entry rounded and written out); the band that completes it puts
// it into the ready queue.  Its targets are first needed kPrefetch steps
// before the first target entry is rounded.  In the reference schedule of
// the plan check, band I runs kLambda steps behind band I - 1, which leaves
// every task tens of steps between the two.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define SWEEP_HD __host__ __device__ __forceinline__
#else
#define SWEEP_HD inline
#endif

namespace bakron {
namespace sweep {

constexpr int kT = 32;         // band height and tile width
constexpr int kChunk = 4;      // tiles (bands) per chunk
constexpr int kSliceLines = 8; // rows (columns) of a slice task's source
constexpr int kRowAluTiles = 3;  // row terms with d < 3 tiles are the band's own
constexpr int kGroupsPerTask = 1;  // target groups (128 lines each) per chunk task
constexpr int kPrefetch = 16;  // band steps between loading a target's delayed sums and rounding it
constexpr int kLambda = 48;    // lag of band I behind band I - 1 in the plan check's reference schedule, in steps

enum TaskType : int { kEmpty = 0, kRowSlice = 1, kColSlice = 2, kRowChunk = 3, kColChunk = 4 };

struct Geom {
  int m, n, Mt, Nt;
  int rowParts, colParts;  // chunk task parts per (band, chunk) and per (chunk, column tile)
  long long nRS, nCS, nRC, nCC;  // canonical task counts per type
};

SWEEP_HD int cdiv(int a, int b) { return (a + b - 1) / b; }
SWEEP_HD int imin(int a, int b) { return a < b ? a : b; }
SWEEP_HD int imax(int a, int b) { return a > b ? a : b; }

SWEEP_HD Geom make_geom(int m, int n) {
  Geom g;
  g.m = m;
  g.n = n;
  g.Mt = cdiv(m, kT);
  g.Nt = cdiv(n, kT);
  // chunk 0 has the most targets: tiles (bands) from 7 (6) to the end
  const int rowGroups = imax(0, cdiv(g.Nt - 7, kChunk));
  const int colGroups = imax(0, cdiv(g.Mt - 6, kChunk));
  g.rowParts = cdiv(rowGroups, kGroupsPerTask);
  g.colParts = cdiv(colGroups, kGroupsPerTask);
  g.nRS = (long long)g.Mt * g.Nt * (kT / kSliceLines);
  g.nCS = (long long)g.Mt * g.Nt * (kT / kSliceLines);
  g.nRC = (long long)g.Mt * cdiv(g.Nt, kChunk) * g.rowParts;
  g.nCC = (long long)cdiv(g.Mt, kChunk) * g.Nt * g.colParts;
  return g;
}

SWEEP_HD long long total_tasks(const Geom& g) { return g.nRS + g.nCS + g.nRC + g.nCC; }

// A task: type, its parameters, the source band(s) it waits for, the
// threshold step, and its targets: tiles [t0, t1) of band `band` (row
// tasks, row slice `ps` or all four) or bands [t0, t1) at column slices
// [cs0, cs1) (column tasks).
struct Task {
  int type;
  int a, b, c;       // ROW_*: band, source tile (slice) or chunk, row slice (part)
                     // COL_*: source band (chunk), column tile, column slice (part)
  int srcBand0, srcBand1;  // bands [srcBand0, srcBand1) whose progress the task waits for
  int readyStep;     // they must have written out every step <= readyStep
  int t0, t1;        // target tiles (row tasks) or bands (column tasks), half-open
  int ps0, ps1;      // row tasks: target row slices [ps0, ps1)
  int cs0, cs1;      // column tasks: target column slices [cs0, cs1)
  int k0, kLen;      // source range along the product's depth: columns (row tasks), rows (column tasks)
  int line0, nLines; // source lines: rows (row tasks) or columns (column tasks)
};

// Decodes canonical task index idx (0 <= idx < total_tasks < 2^31, which
// the callers check).  Tasks whose targets or sources fall outside the
// matrix come back as kEmpty.  32-bit arithmetic throughout.
SWEEP_HD Task decode(const Geom& g, long long idx_in) {
  unsigned idx = (unsigned)idx_in;
  const unsigned Nt = (unsigned)g.Nt;
  Task t;
  t.type = kEmpty;
  t.a = t.b = t.c = 0;
  t.srcBand0 = t.srcBand1 = 0;
  t.readyStep = 0;
  t.t0 = t.t1 = 0;
  t.ps0 = t.ps1 = 0;
  t.cs0 = t.cs1 = 0;
  t.k0 = t.kLen = t.line0 = t.nLines = 0;
  const unsigned nps = kT / kSliceLines;
  if (idx < (unsigned)g.nRS) {
    const int ps = (int)(idx % nps);
    const unsigned rest = idx / nps;
    const int j = (int)(rest % Nt);
    const int I = (int)(rest / Nt);
    const int first = j + kRowAluTiles, last = imin(kChunk * (j / kChunk) + kChunk + kRowAluTiles - 1, g.Nt - 1);
    const int r0 = I * kT + kSliceLines * ps;
    if (first > last || r0 >= g.m) return t;
    t.type = kRowSlice;
    t.a = I; t.b = j; t.c = ps;
    t.srcBand0 = I; t.srcBand1 = I + 1;
    t.readyStep = imin(kT * j + kT - 1, g.n - 1) + kSliceLines * ps + kSliceLines - 1;
    t.t0 = first; t.t1 = last + 1;
    t.ps0 = ps; t.ps1 = ps + 1;
    t.k0 = kT * j; t.kLen = imin(kT, g.n - kT * j);
    t.line0 = r0; t.nLines = imin(kSliceLines, g.m - r0);
    return t;
  }
  idx -= (unsigned)g.nRS;
  if (idx < (unsigned)g.nCS) {
    const int cs = (int)(idx % nps);
    const unsigned rest = idx / nps;
    const int J = (int)(rest % Nt);
    const int I = (int)(rest / Nt);
    const int first = I + 2, last = imin(kChunk * (I / kChunk) + kChunk + 1, g.Mt - 1);
    const int c0 = J * kT + kSliceLines * cs;
    if (first > last || c0 >= g.n) return t;
    t.type = kColSlice;
    t.a = I; t.b = J; t.c = cs;
    t.srcBand0 = I; t.srcBand1 = I + 1;
    t.readyStep = imin(c0 + kSliceLines, g.n) - 1 + kT - 1;
    t.t0 = first; t.t1 = last + 1;
    t.cs0 = J * (kT / kSliceLines) + cs; t.cs1 = t.cs0 + 1;
    t.k0 = kT * I; t.kLen = imin(kT, g.m - kT * I);
    t.line0 = c0; t.nLines = imin(kSliceLines, g.n - c0);
    return t;
  }
  idx -= (unsigned)g.nCS;
  if (idx < (unsigned)g.nRC) {
    const unsigned nch = (unsigned)cdiv(g.Nt, kChunk);
    const int part = (int)(idx % (unsigned)g.rowParts);
    const unsigned rest = idx / (unsigned)g.rowParts;
    const int h = (int)(rest % nch);
    const int I = (int)(rest / nch);
    const int first = kChunk * h + kChunk + kRowAluTiles;  // 4h + 7
    const int g0 = part * kGroupsPerTask;
    const int t0 = first + kChunk * g0;
    if (t0 >= g.Nt) return t;
    t.type = kRowChunk;
    t.a = I; t.b = h; t.c = part;
    t.srcBand0 = I; t.srcBand1 = I + 1;
    t.readyStep = imin(kT * kChunk * (h + 1), g.n) - 1 + kT - 1;
    t.t0 = t0; t.t1 = imin(t0 + kChunk * kGroupsPerTask, g.Nt);
    t.ps0 = 0; t.ps1 = (int)nps;
    t.k0 = kT * kChunk * h; t.kLen = imin(kT * kChunk, g.n - t.k0);
    t.line0 = kT * I; t.nLines = imin(kT, g.m - kT * I);
    return t;
  }
  idx -= (unsigned)g.nRC;
  if (idx < (unsigned)g.nCC) {
    const int part = (int)(idx % (unsigned)g.colParts);
    const unsigned rest = idx / (unsigned)g.colParts;
    const int J = (int)(rest % Nt);
    const int h = (int)(rest / Nt);
    const int first = kChunk * h + kChunk + 2;  // 4h + 6
    const int g0 = part * kGroupsPerTask;
    const int t0 = first + kChunk * g0;
    if (t0 >= g.Mt) return t;
    t.type = kColChunk;
    t.a = h; t.b = J; t.c = part;
    t.srcBand0 = kChunk * h; t.srcBand1 = imin(kChunk * h + kChunk, g.Mt);
    t.readyStep = imin(kT * J + kT, g.n) - 1 + kT - 1;
    t.t0 = t0; t.t1 = imin(t0 + kChunk * kGroupsPerTask, g.Mt);
    t.cs0 = J * (kT / kSliceLines);
    t.cs1 = imin(t.cs0 + kT / kSliceLines, cdiv(g.n, kSliceLines));
    t.k0 = kT * kChunk * h; t.kLen = imin(kT * kChunk, g.m - t.k0);
    t.line0 = kT * J; t.nLines = imin(kT, g.n - kT * J);
    return t;
  }
  return t;
}

// Ideal global time of a band step: band I runs kLambda steps behind I - 1.
SWEEP_HD long long ideal_time(int band, int step) { return (long long)band * kLambda + step; }

// Ideal time at which a task's sources are complete.
SWEEP_HD long long ready_time(const Task& t) { return ideal_time(t.srcBand1 - 1, t.readyStep); }

// Ideal time at which the band first needs the task's contribution (its
// earliest target entry, loaded kPrefetch steps before it is rounded).
SWEEP_HD long long need_time(const Task& t) {
  if (t.type == kRowSlice || t.type == kRowChunk)
    return ideal_time(t.a, kT * t.t0 + kSliceLines * t.ps0 - kPrefetch);
  return ideal_time(t.t0, kSliceLines * t.cs0 - kPrefetch);
}

}  // namespace sweep
}  // namespace bakron
