// internal.h -- declarations shared by the translation units of libbakron.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bakron {

constexpr size_t kAlign = 256;

// A process-unique id of the calling thread's current CUDA context (the
// driver's cuCtxGetId, reached through the runtime's driver entry point, so
// the library does not link the driver library).  Per-device caches (side
// streams and events, the no-allocation scratch address) are keyed on it:
// after cudaDeviceReset the device's next primary context has a new id, and
// the caches are rebuilt instead of handing out handles or addresses of the
// destroyed context.
cudaError_t current_context_id(unsigned long long* id);

inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Per-kernel-class timing of one solve (diagnostics): CUDA events around
// every launch, read back after the stream is synchronized.
// 0: input check + offset, 1: tile solve, 2: mid push, 3: chunk push (the
// launch-per-step schedule), 4: the persistent sweep (set-up included).
constexpr int kKernelClasses = 5;
struct KernelTimer {
  double ms[kKernelClasses];
  int64_t launches[kKernelClasses];
  double flops[kKernelClasses];  // algorithmic flops (2 per multiply-add) of the class
};

// Integer alphabet of the rounding: {lo .. hi} when bounded, else Z.
struct Alphabet {
  bool bounded;
  int lo, hi;
};
// `bits` = 0: Z; 2..8: {-2^(bits-1) .. 2^(bits-1) - 1}.
inline Alphabet alphabet_from_bits(int bits) {
  return bits ? Alphabet{true, -(1 << (bits - 1)), (1 << (bits - 1)) - 1} : Alphabet{false, 0, 0};
}

// Scales of the alphabet: entry (i, j) has scale fp32(R[i][j / group] t[j]),
// R m x ceil(n / group) (group <= 0 or >= n: one scale per row), R or t null
// for ones.
struct Scales {
  const float* R;
  int group;
  const float* t;
};
inline Scales per_row(const float* s) { return Scales{s, 0, nullptr}; }

// quantize.cu (LB == nullptr: the output factor is the identity, row-wise GPTQ)
size_t quantize_workspace_bytes(int64_t m, int64_t n);
cudaError_t quantize_launch(const float* W, const float* LA, const float* LB, Scales sc,
                            Alphabet al, int m, int n, int32_t* V, float* Wq, void* ws,
                            int32_t* status_dev, cudaStream_t stream, KernelTimer* timer = nullptr);
// Host-only check of quantize_launch's schedule (see quantize.cu).
int wavefront_plan_check(int64_t m, int64_t n, bool colpush, int lag, int64_t* stats);

// sweep.cu (the persistent band sweep: one cooperative kernel per solve)
size_t sweep_workspace_bytes(int64_t m, int64_t n);
bool sweep_supported(int64_t m, int64_t n);
// kernel_ms: if given, the call synchronizes and reports the sweep kernel's
// own time (CUDA events around its launch).
cudaError_t sweep_launch(const float* W, const float* LA, const float* LB, Scales sc, Alphabet al, int m, int n,
                         int32_t* V, float* Wq, void* ws, int32_t* status_dev, cudaStream_t stream,
                         float* kernel_ms);
int sweep_plan_check(int64_t m, int64_t n, int64_t* stats);

// antidiag.cu (Algorithm 3, one launch per anti-diagonal; per-row scales)
size_t antidiag_workspace_bytes(int64_t m, int64_t n);
cudaError_t antidiag_launch(const float* W, const float* LA, const float* LB, const float* scales, Alphabet al,
                            int m, int n, int32_t* V, float* Wq, void* ws, int32_t* status_dev,
                            cudaStream_t stream);

// gram.cu (Kronecker factors from samples)
size_t gram_workspace_bytes(int64_t d, int64_t N, bool weighted);
cudaError_t gram_launch(const uint16_t* X, int d, int N, int ldx, const float* w, float alpha, float beta, float* G,
                        void* ws, int32_t* status_dev, cudaStream_t stream);
cudaError_t sq_norms_launch(const uint16_t* Y, int m, int N, int ldy, float* w, cudaStream_t stream);
cudaError_t damp_launch(float* G, int d, float rel, cudaStream_t stream);

// selftest.cu
cudaError_t wait_selftest_launch(int32_t* status_dev, cudaStream_t stream);

// scales.cu
// One scale per run of `group` columns of each row (group <= 0 or >= n: per
// row), m x ceil(n / group) outputs.
cudaError_t row_scales_launch(const float* W, int m, int n, int group, Alphabet al, int grid, float* scales,
                              cudaStream_t stream);
cudaError_t pack_codes_launch(const int32_t* V, int m, int n, int bits, uint8_t* out, cudaStream_t stream);

// prep.cu
size_t factor_workspace_bytes(int64_t d);
cudaError_t factor_launch(const float* H, int d, float* Lhat, void* ws, int32_t* info_dev,
                          cudaStream_t stream);

}  // namespace bakron
