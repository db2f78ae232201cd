// gram.cu -- Kronecker factors from calibration samples on the tensor cores
// ("BaKron: Efficient Quantization with Kronecker-Factored Hessians",
// Sec. 4.2 and App. A.2: K-FAC factors E[a a^T], E[b b^T]; one Shampoo step
// E[|b|^2 a a^T], E[|a|^2 b b^T]; App. D: damping by 0.5 times the mean
// diagonal):
//     G <- beta G + alpha X diag(w) X^T
// for samples X (d features x N samples, bfloat16, feature-major) and
// optional per-sample weights w (fp32).
//
// A packing pass first rearranges X into 16 KB blocks of 128 rows x 64
// samples, each already in the tcgen05 core-matrix layout (K = samples), in
// one streaming read and write.  With weights it also writes the column
// operand w_t x_t split into two bf16 terms (hi = bf16(w x), lo = bf16(w x -
// hi), about 2^-17 relative left over), multiplied in two MMAs.  Each CTA of
// the Gram kernel then computes one 128 x 128 tile of the lower block
// triangle over all N samples: one thread loads each stage with 1-D bulk
// copies of 16 KB that complete on the stage's mbarrier (the row operand;
// the column operand unless the tile is diagonal and unweighted; its low
// half with weights), one
// thread issues an MMA of M = N = 128, K = 16 per 16 samples into tensor
// memory (fp32; every bf16 x bf16 product is exact there).  The fp32
// accumulation in tensor memory is restarted every kGSegSamples samples:
// after each segment four epilogue warps add the accumulator into a running
// fp32 sum kept in tensor memory (columns 128..255), 32 columns per round
// trip, while the MMAs wait, so the rounding of the tensor cores' long
// accumulation grows with the segment length instead of with N (the running
// sum adds one rounding per segment).  Two CTAs share an SM, so one
// multiplies while the other adds.  After the last segment the epilogue
// writes the tile and its mirror.
#include <cuda_bf16.h>

#include <algorithm>

#include "bakron.h"
#include "df.cuh"
#include "internal.h"
#include "tc.cuh"

namespace bakron {
namespace {

constexpr int kGT = 128;                 // output tile edge (tensor-memory lanes, MMA N)
constexpr int kGK = 64;                  // samples per stage: 8 groups of 8 (16 bytes)
constexpr int kGStages = 3;
constexpr int kGSegStages = 32;                 // stages per accumulation segment
constexpr int kGSegSamples = kGSegStages * 64;  // 2048 samples
constexpr int kGWarps = 8;
constexpr int kGThreads = kGWarps * 32;
constexpr uint32_t kGLbo = 128;              // stride of an 8-sample group within an 8-row block
constexpr uint32_t kGSbo = 128 * (kGK / 8);  // stride of an 8-row block: 1024 bytes
constexpr int kGTileBytes = kGT * kGK * 2;   // 16 KB
constexpr int kGChunks = kGT * (kGK / 8);    // 16-byte chunks per block: 1024

template <bool kW>
struct GramSmem {
  static constexpr int kStages = kGStages;
  alignas(128) unsigned char A[kStages][kGTileBytes];
  alignas(128) unsigned char B[kStages][kW ? 2 : 1][kGTileBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t seg_full;   // the MMAs of a segment are done (commit)
  uint64_t seg_empty;  // the epilogue has added the segment into the running sum (128 arrivals)
  uint32_t tmem_base;
};

// Packed samples: block (rb, kb) holds rows 128 rb .. +127 and samples
// 64 kb .. +63 as 16 KB in the tcgen05 core-matrix layout (K-major, no
// swizzle): chunk c (16 bytes, 8 samples) is row 8 (c / 64) + c % 8, sample
// group (c % 64) / 8, so that byte 16 c = (r/8) SBO + g LBO + (r%8) 16.
// Blocks are stored block-row-major, [rb][kb].
struct GramParams {
  const unsigned char* Xa;   // packed samples (row operand)
  const unsigned char* Xb;   // packed column operand: the samples, or w x's high part
  const unsigned char* Xl;   // low part of w x (weighted only)
  float* G;
  int32_t* status;
  int d, nkb;
  float alpha, beta;
};

__device__ __forceinline__ void gchunk(int c, int& r, int& g) {
  r = 8 * (c / 64) + (c % 8);
  g = (c % 64) / 8;
}

__device__ __forceinline__ void tri_index(int t, int& bi, int& bj) {
  int i = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
  while (i * (i + 1) / 2 > t) --i;
  while ((i + 1) * (i + 2) / 2 <= t) ++i;
  bi = i;
  bj = t - i * (i + 1) / 2;
}

// One thread per 16-byte chunk of the packed arrays: the samples (zeros
// outside the matrix) and, with weights, w_t x_t split into bf16 hi + lo.
__global__ void gram_pack_kernel(const uint16_t* X, int d, int N, int ldx, const float* w, int nkb,
                                 unsigned char* Xa, unsigned char* Xh, unsigned char* Xl) {
  const size_t total = (size_t)((d + kGT - 1) / kGT) * nkb * kGChunks;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t blk = idx / kGChunks;
    const int c = (int)(idx % kGChunks);
    const int rb = (int)(blk / nkb), kb = (int)(blk % nkb);
    int r, g;
    gchunk(c, r, g);
    const int row = rb * kGT + r, k = kb * kGK + 8 * g;
    uint32_t xv[4] = {0u, 0u, 0u, 0u};
    if (row < d && k + 8 <= N) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(X + (size_t)row * ldx + k));
      xv[0] = q.x, xv[1] = q.y, xv[2] = q.z, xv[3] = q.w;
    } else if (row < d) {
      for (int e = 0; e < 8 && k + e < N; ++e) xv[e / 2] |= (uint32_t)X[(size_t)row * ldx + k + e] << (16 * (e % 2));
    }
    reinterpret_cast<uint4*>(Xa)[idx] = make_uint4(xv[0], xv[1], xv[2], xv[3]);
    if (w) {
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k0 = k + 2 * e;
        const float w0 = (row < d && k0 < N) ? w[k0] : 0.f, w1 = (row < d && k0 + 1 < N) ? w[k0 + 1] : 0.f;
        const float p0 = w0 * __uint_as_float(xv[e] << 16), p1 = w1 * __uint_as_float(xv[e] & 0xFFFF0000u);
        const __nv_bfloat16 h0 = __float2bfloat16_rn(p0), h1 = __float2bfloat16_rn(p1);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(p0 - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(p1 - __bfloat162float(h1));
        hv[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        lv[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
      }
      reinterpret_cast<uint4*>(Xh)[idx] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      reinterpret_cast<uint4*>(Xl)[idx] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
  }
}

// A 1-D bulk copy global -> shared (the TMA engine, no tensor map), counted
// on the mbarrier's transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(mbar))
               : "memory");
}

template <bool kW>
__global__ void __launch_bounds__(kGThreads, 2) gram_kernel(GramParams P) {
  extern __shared__ __align__(1024) unsigned char g_smem_raw[];
  GramSmem<kW>& sm = *reinterpret_cast<GramSmem<kW>*>(g_smem_raw);
  int bi, bj;
  tri_index(blockIdx.x, bi, bj);
  const bool diag = bi == bj;
  const bool copy_b = kW || !diag;  // the diagonal tile without weights multiplies A by itself
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nz = P.nkb;
  bool broken = false;

  constexpr int kStages = GramSmem<kW>::kStages;
  const int nseg = (nz + kGSegStages - 1) / kGSegStages;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.empty[i])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&sm.seg_full)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;\n" ::"r"(smem_u32(&sm.seg_empty)));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {  // the accumulator at column 0, the running sum at column 128
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;\n" ::"r"(smem_u32(&sm.tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 1 && lane == 0) {  // the copy thread: one to three bulk copies of 16 KB per stage
    const uint32_t bytes = (uint32_t)kGTileBytes * (1u + (copy_b ? 1u : 0u) + (kW ? 1u : 0u));
    const size_t rowa = (size_t)bi * P.nkb, rowb = (size_t)bj * P.nkb;
    for (int z = 0; z < nz; ++z) {
      const int slot = z % kStages;
      if (z >= kStages) mbar_wait(&sm.empty[slot], (uint32_t)((z / kStages) - 1) & 1u, broken);
      if (broken) break;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(&sm.full[slot])),
                   "r"(bytes)
                   : "memory");
      bulk_g2s(sm.A[slot], P.Xa + (rowa + z) * kGTileBytes, kGTileBytes, &sm.full[slot]);
      if (copy_b) bulk_g2s(sm.B[slot][0], P.Xb + (rowb + z) * kGTileBytes, kGTileBytes, &sm.full[slot]);
      if (kW) bulk_g2s(sm.B[slot][kW ? 1 : 0], P.Xl + (rowb + z) * kGTileBytes, kGTileBytes, &sm.full[slot]);
    }
  } else if (warp == 0 && lane == 0) {  // the MMA thread
    constexpr uint32_t idesc = umma_idesc_bf16(kGT, kGT);
    for (int z = 0; z < nz; ++z) {
      const int slot = z % kStages;
      const int seg = z / kGSegStages, zs = z % kGSegStages;
      const uint32_t acc = tmem;
      // the accumulator is free once the epilogue added segment seg - 1
      if (zs == 0 && seg >= 1) mbar_wait(&sm.seg_empty, (uint32_t)(seg - 1) & 1u, broken);
      mbar_wait(&sm.full[slot], (uint32_t)(z / kStages) & 1u, broken);
      if (broken) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sm.A[slot]);
      const uint32_t b0 = copy_b ? smem_u32(sm.B[slot][0]) : a0;
#pragma unroll
      for (int j = 0; j < kGK / 16; ++j) {
        const uint32_t off = (uint32_t)(2 * j) * kGLbo;
        const uint64_t da = umma_sdesc(a0 + off, kGLbo, kGSbo);
        umma_bf16(acc, da, umma_sdesc(b0 + off, kGLbo, kGSbo), idesc, (zs > 0 || j > 0) ? 1u : 0u);
        if (kW) umma_bf16(acc, da, umma_sdesc(smem_u32(sm.B[slot][kW ? 1 : 0]) + off, kGLbo, kGSbo), idesc, 1u);
      }
      umma_commit(&sm.empty[slot]);
      if (zs == kGSegStages - 1 || z == nz - 1) umma_commit(&sm.seg_full);
    }
  }
  __syncwarp();

  if (warp >= 4) {  // epilogue: tensor-memory lane quarter warp - 4, one output row per thread
    const int q = warp - 4;
    const int r = 32 * q + lane;
    const int i = bi * kGT + r;
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    for (int seg = 0; seg < nseg; ++seg) {
      const bool last = seg == nseg - 1;
      mbar_wait(&sm.seg_full, (uint32_t)seg & 1u, broken);
      tc_fence_after();
#pragma unroll 1
      for (int c32 = 0; c32 < kGT / 32; ++c32) {
        // Running sum += this segment's sums (one fp32 rounding per segment),
        // 32 columns per round trip to tensor memory.
        float v[4][8], hi[4][8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tmem_ld(tmem + lanes + (uint32_t)(32 * c32 + 8 * k), v[k]);
          if (seg > 0) tmem_ld(tmem + lanes + (uint32_t)(kGT + 32 * c32 + 8 * k), hi[k]);
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int e = 0; e < 8; ++e) hi[k][e] = seg == 0 ? v[k][e] : hi[k][e] + v[k][e];
        if (!last) {
#pragma unroll
          for (int k = 0; k < 4; ++k) tmem_st(tmem + lanes + (uint32_t)(kGT + 32 * c32 + 8 * k), hi[k]);
          continue;
        }
        // Entry (i, j) and its mirror (j, i); a diagonal tile writes its lower
        // triangle and mirrors it, so G is exactly symmetric even where the
        // two triangles' products were rounded differently (weighted split).
        if (i < P.d && !broken) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = bj * kGT + 32 * c32 + 8 * k + e;
              if (j < P.d && !(diag && j > i)) {
                float g = P.alpha * hi[k][e];
                if (P.beta != 0.f) g = fmaf(P.beta, P.G[(size_t)i * P.d + j], g);
                P.G[(size_t)i * P.d + j] = g;
                if (j != i) P.G[(size_t)j * P.d + i] = g;  // the mirror (coalesced across the warp)
              }
            }
        }
      }
      if (!last) {
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        tc_fence_before();
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.seg_empty)) : "memory");
      }
    }
  }
  if (broken) atomicOr(P.status, BAKRON_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;\n" ::"r"(tmem));
}

__global__ void sq_norms_kernel(const uint16_t* Y, int m, int N, int ldy, float* w) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= N) return;
  float2 acc = make_float2(0.f, 0.f);  // double-float sum of exact squares
  for (int i = 0; i < m; ++i) {
    const float y = __uint_as_float((uint32_t)Y[(size_t)i * ldy + t] << 16);
    acc = df_add(acc, two_prod(y, y));
  }
  w[t] = acc.x + acc.y;
}

// G + rel * mean(diag G) * I; one CTA of 1024 threads, the trace in double-float.
__global__ void damp_kernel(float* G, int d, float rel) {
  __shared__ float2 red[32];
  float2 s = make_float2(0.f, 0.f);
  for (int i = threadIdx.x; i < d; i += blockDim.x) s = df_add(s, make_float2(G[(size_t)i * d + i], 0.f));
  for (int o = 16; o; o >>= 1)
    s = df_add(s, make_float2(__shfl_xor_sync(0xffffffffu, s.x, o), __shfl_xor_sync(0xffffffffu, s.y, o)));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  float2 tot = make_float2(0.f, 0.f);
  for (int k = 0; k < (int)(blockDim.x >> 5); ++k) tot = df_add(tot, red[k]);
  const float add = rel * __fdiv_rn(tot.x + tot.y, (float)d);
  __syncthreads();
  for (int i = threadIdx.x; i < d; i += blockDim.x) G[(size_t)i * d + i] += add;
}

}  // namespace

size_t gram_workspace_bytes(int64_t d, int64_t N, bool weighted) {
  const size_t blocks = (size_t)((d + kGT - 1) / kGT) * (size_t)((N + kGK - 1) / kGK);
  return blocks * kGTileBytes * (weighted ? 3 : 1);
}

cudaError_t gram_launch(const uint16_t* X, int d, int N, int ldx, const float* w, float alpha, float beta, float* G,
                        void* ws, int32_t* status_dev, cudaStream_t stream) {
  const int nb = (d + kGT - 1) / kGT;
  const int nkb = (N + kGK - 1) / kGK;
  const size_t plane = (size_t)nb * nkb * kGTileBytes;
  unsigned char* Xa = static_cast<unsigned char*>(ws);
  unsigned char* Xh = w ? Xa + plane : nullptr;
  unsigned char* Xl = w ? Xa + 2 * plane : nullptr;
  GramParams P{Xa, w ? Xh : Xa, Xl, G, status_dev, d, nkb, alpha, beta};
  const int tiles = nb * (nb + 1) / 2;
  cudaError_t e = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  const size_t chunks = plane / 16;
  const int pack_blocks = (int)std::min<size_t>((chunks + 255) / 256, 152 * 16);
  gram_pack_kernel<<<pack_blocks, 256, 0, stream>>>(X, d, N, ldx, w, nkb, Xa, Xh, Xl);
  if (w) {
    const size_t smem = sizeof(GramSmem<true>) + 1024;
    e = cudaFuncSetAttribute(gram_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gram_kernel<true><<<tiles, kGThreads, smem, stream>>>(P);
  } else {
    const size_t smem = sizeof(GramSmem<false>) + 1024;
    e = cudaFuncSetAttribute(gram_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gram_kernel<false><<<tiles, kGThreads, smem, stream>>>(P);
  }
  return cudaGetLastError();
}

cudaError_t sq_norms_launch(const uint16_t* Y, int m, int N, int ldy, float* w, cudaStream_t stream) {
  sq_norms_kernel<<<(N + 255) / 256, 256, 0, stream>>>(Y, m, N, ldy, w);
  return cudaGetLastError();
}

cudaError_t damp_launch(float* G, int d, float rel, cudaStream_t stream) {
  damp_kernel<<<1, 1024, 0, stream>>>(G, d, rel);
  return cudaGetLastError();
}

}  // namespace bakron
