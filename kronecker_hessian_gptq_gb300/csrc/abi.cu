// abi.cu -- the extern "C" entry points of libbakron.so (declared in bakron.h).
//
// Every entry point validates its arguments on the host and returns a
// bakron_status before enqueuing anything; device-side conditions go to the
// caller's device status words.
#include <cstdint>
#include <mutex>

#include "bakron.h"
#include "internal.h"

namespace bakron {

cudaError_t current_context_id(unsigned long long* id) {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static cudaError_t lookup = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    lookup = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q);
    if (lookup == cudaSuccess && q == cudaDriverEntryPointSuccess) get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (lookup == cudaSuccess) lookup = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q);
    if (lookup == cudaSuccess && q == cudaDriverEntryPointSuccess) get_id = reinterpret_cast<GetId>(f);
    if (lookup == cudaSuccess && (!get_current || !get_id)) lookup = cudaErrorSymbolNotFound;
  });
  if (lookup != cudaSuccess) return lookup;
  // Make the runtime create or bind the current device's primary context
  // first (cudaSetDevice initializes it).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  if (e != cudaSuccess) return e;
  void* ctx = nullptr;
  if (get_current(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
  return get_id(ctx, id) == 0 ? cudaSuccess : cudaErrorDeviceUninitialized;
}

}  // namespace bakron

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? BAKRON_OK : BAKRON_ERR_CUDA; }

constexpr int64_t kMaxElems = (int64_t)1 << 31;  // m * n and d * d limit (int indexing)

}  // namespace

extern "C" {

const char* bakron_status_string(int status) {
  switch (status) {
    case BAKRON_OK: return "BAKRON_OK";
    case BAKRON_ERR_INVALID_ARG: return "BAKRON_ERR_INVALID_ARG";
    case BAKRON_ERR_NOT_SPD: return "BAKRON_ERR_NOT_SPD";
    case BAKRON_ERR_CUDA: return "BAKRON_ERR_CUDA";
    case BAKRON_ERR_WORKSPACE: return "BAKRON_ERR_WORKSPACE";
    case BAKRON_ERR_TIMEOUT: return "BAKRON_ERR_TIMEOUT";
    default: return "BAKRON_ERR_UNKNOWN";
  }
}

int bakron_abi_version(void) { return BAKRON_ABI_VERSION; }

size_t bakron_factor_workspace_size(int64_t d) {
  if (d < 1 || d * d >= kMaxElems) return 0;
  return bakron::factor_workspace_bytes(d);
}

int bakron_factor(const float* H, int64_t d, float* Lhat, void* ws, size_t ws_bytes, int32_t* info_dev,
                  void* stream) {
  if (!H || !Lhat || !info_dev || d < 1 || d * d >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)H == (const void*)Lhat) return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::factor_workspace_bytes(d))
    return BAKRON_ERR_WORKSPACE;
  return from_cuda(bakron::factor_launch(H, (int)d, Lhat, ws, info_dev, (cudaStream_t)stream));
}

size_t bakron_prepare_workspace_size(int64_t m, int64_t n) {
  const size_t a = bakron_factor_workspace_size(n), b = bakron_factor_workspace_size(m);
  if (a == 0 || b == 0) return 0;
  return a > b ? a : b;
}

int bakron_prepare(const float* A, const float* B, int64_t m, int64_t n, float* LA, float* LB, void* ws,
                   size_t ws_bytes, int32_t* info_dev, void* stream) {
  if (!A || !B || !LA || !LB || !info_dev || m < 1 || n < 1) return BAKRON_ERR_INVALID_ARG;
  if (m * m >= kMaxElems || n * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)A == (const void*)LA || (const void*)B == (const void*)LB || LA == LB)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron_prepare_workspace_size(m, n))
    return BAKRON_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = bakron::factor_launch(A, (int)n, LA, ws, info_dev, s);
  if (e != cudaSuccess) return BAKRON_ERR_CUDA;
  return from_cuda(bakron::factor_launch(B, (int)m, LB, ws, info_dev + 1, s));
}

size_t bakron_quantize_workspace_size(int64_t m, int64_t n) {
  if (m < 1 || n < 1 || m * n >= kMaxElems) return 0;
  return bakron::quantize_workspace_bytes(m, n);
}

int bakron_quantize(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                    int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                    int32_t* status_dev, void* stream) {
  if (!W || !LA || !LB || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 0 || (bits >= 2 && bits <= 8))) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::quantize_workspace_bytes(m, n))
    return BAKRON_ERR_WORKSPACE;
  return from_cuda(bakron::quantize_launch(W, LA, LB, bakron::per_row(scales), bakron::alphabet_from_bits(bits), (int)m, (int)n, V, Wq, ws, status_dev,
                                           (cudaStream_t)stream));
}

int bakron_quantize_persistent(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                               int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                               int32_t* status_dev, void* stream) {
  if (!W || !LA || !LB || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems || !bakron::sweep_supported(m, n)) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 0 || (bits >= 2 && bits <= 8))) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::quantize_workspace_bytes(m, n))
    return BAKRON_ERR_WORKSPACE;
  return from_cuda(bakron::sweep_launch(W, LA, LB, bakron::per_row(scales), bakron::alphabet_from_bits(bits), (int)m,
                                        (int)n, V, Wq, ws, status_dev, (cudaStream_t)stream, nullptr));
}

size_t bakron_gptq_workspace_size(int64_t m, int64_t n) { return bakron_quantize_workspace_size(m, n); }

int bakron_gptq_quantize(const float* W, const float* LA, const float* scales, int bits, int64_t m, int64_t n,
                         int32_t* V, float* Wq, void* ws, size_t ws_bytes, int32_t* status_dev, void* stream) {
  if (!W || !LA || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 0 || (bits >= 2 && bits <= 8))) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::quantize_workspace_bytes(m, n))
    return BAKRON_ERR_WORKSPACE;
  // L_B = I: the solver skips every column term (nullptr output factor).
  return from_cuda(bakron::quantize_launch(W, LA, nullptr, bakron::per_row(scales), bakron::alphabet_from_bits(bits), (int)m, (int)n, V, Wq, ws, status_dev,
                                           (cudaStream_t)stream));
}

int bakron_quantize_range(const float* W, const float* LA, const float* LB, const float* scales, int lo, int hi,
                          int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                          int32_t* status_dev, void* stream) {
  if (!W || !LA || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!(lo < hi && lo <= 0 && hi >= 0 && lo >= -BAKRON_MAX_CODE && hi <= BAKRON_MAX_CODE))
    return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::quantize_workspace_bytes(m, n))
    return BAKRON_ERR_WORKSPACE;
  return from_cuda(bakron::quantize_launch(W, LA, LB, bakron::per_row(scales), bakron::Alphabet{true, lo, hi}, (int)m, (int)n, V, Wq,
                                           ws, status_dev, (cudaStream_t)stream));
}

int bakron_row_scales(const float* W, int64_t m, int64_t n, int64_t group, int lo, int hi, int grid, float* scales,
                      void* stream) {
  if (!W || !scales || m < 1 || n < 1 || m * n >= kMaxElems || group < 0) return BAKRON_ERR_INVALID_ARG;
  if (!(lo < 0 && hi > 0 && lo >= -BAKRON_MAX_CODE && hi <= BAKRON_MAX_CODE)) return BAKRON_ERR_INVALID_ARG;
  if (grid < 1 || grid > BAKRON_MAX_SCALE_GRID) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)W == (const void*)scales) return BAKRON_ERR_INVALID_ARG;
  const int g = (group == 0 || group > n) ? (int)n : (int)group;
  return from_cuda(bakron::row_scales_launch(W, (int)m, (int)n, g, bakron::Alphabet{true, lo, hi}, grid, scales,
                                             (cudaStream_t)stream));
}

int bakron_quantize_scaled(const float* W, const float* LA, const float* LB, const float* scales, int64_t group,
                           const float* col_scales, int lo, int hi, int64_t m, int64_t n, int32_t* V, float* Wq,
                           void* ws, size_t ws_bytes, int32_t* status_dev, void* stream) {
  if (!W || !LA || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems || group < 0) return BAKRON_ERR_INVALID_ARG;
  if (!(lo < hi && lo <= 0 && hi >= 0 && lo >= -BAKRON_MAX_CODE && hi <= BAKRON_MAX_CODE))
    return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::quantize_workspace_bytes(m, n))
    return BAKRON_ERR_WORKSPACE;
  const int g = (group == 0 || group > n) ? (int)n : (int)group;
  return from_cuda(bakron::quantize_launch(W, LA, LB, bakron::Scales{scales, g, col_scales},
                                           bakron::Alphabet{true, lo, hi}, (int)m, (int)n, V, Wq, ws, status_dev,
                                           (cudaStream_t)stream));
}

int bakron_pack_codes(const int32_t* V, int64_t m, int64_t n, int bits, uint8_t* out, void* stream) {
  if (!V || !out || m < 1 || n < 1 || m * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 2 || bits == 4 || bits == 8)) return BAKRON_ERR_INVALID_ARG;
  return from_cuda(bakron::pack_codes_launch(V, (int)m, (int)n, bits, out, (cudaStream_t)stream));
}

size_t bakron_antidiag_workspace_size(int64_t m, int64_t n) {
  if (m < 1 || n < 1 || m * n >= kMaxElems) return 0;
  return bakron::antidiag_workspace_bytes(m, n);
}

int bakron_antidiag_quantize(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                             int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                             int32_t* status_dev, void* stream) {
  if (!W || !LA || !LB || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 0 || (bits >= 2 && bits <= 8))) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::antidiag_workspace_bytes(m, n))
    return BAKRON_ERR_WORKSPACE;
  return from_cuda(bakron::antidiag_launch(W, LA, LB, scales, bakron::alphabet_from_bits(bits), (int)m, (int)n, V,
                                           Wq, ws, status_dev, (cudaStream_t)stream));
}

size_t bakron_gram_workspace_size(int64_t d, int64_t N, int weighted) {
  if (d < 1 || N < 1 || d * d >= kMaxElems || N >= kMaxElems) return 0;
  return bakron::gram_workspace_bytes(d, N, weighted != 0);
}

int bakron_gram(const void* X, int64_t d, int64_t N, int64_t ldx, const float* w, float alpha, float beta, float* G,
                void* ws, size_t ws_bytes, int32_t* status_dev, void* stream) {
  if (!X || !G || !status_dev || d < 1 || N < 1 || ldx < N || ldx % 8 != 0) return BAKRON_ERR_INVALID_ARG;
  if (d * d >= kMaxElems || d * ldx >= ((int64_t)1 << 40) || N >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!aligned(X, 16) || (w && !aligned(w, 16)) || (const void*)G == X) return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::gram_workspace_bytes(d, N, w != nullptr))
    return BAKRON_ERR_WORKSPACE;
  return from_cuda(bakron::gram_launch(static_cast<const uint16_t*>(X), (int)d, (int)N, (int)ldx, w, alpha, beta, G,
                                       ws, status_dev, (cudaStream_t)stream));
}

int bakron_sq_norms(const void* Y, int64_t m, int64_t N, int64_t ldy, float* w, void* stream) {
  if (!Y || !w || m < 1 || N < 1 || ldy < N || N >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  return from_cuda(bakron::sq_norms_launch(static_cast<const uint16_t*>(Y), (int)m, (int)N, (int)ldy, w,
                                           (cudaStream_t)stream));
}

int bakron_damp(float* G, int64_t d, float rel, void* stream) {
  if (!G || d < 1 || d * d >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  return from_cuda(bakron::damp_launch(G, (int)d, rel, (cudaStream_t)stream));
}

int bakron_selftest_wait_timeout(int32_t* status_dev, void* stream) {
  if (!status_dev) return BAKRON_ERR_INVALID_ARG;
  return from_cuda(bakron::wait_selftest_launch(status_dev, (cudaStream_t)stream));
}

int bakron_sweep_plan_check(int64_t m, int64_t n, int64_t* stats) {
  if (!stats || m < 1 || n < 1 || m * n >= kMaxElems || !bakron::sweep_supported(m, n)) return BAKRON_ERR_INVALID_ARG;
  return bakron::sweep_plan_check(m, n, stats) == 0 ? BAKRON_OK : 1;
}

int bakron_wavefront_plan_check(int64_t m, int64_t n, int colpush, int lag, int64_t* stats) {
  if (!stats || m < 1 || n < 1 || m > (int64_t)1 << 15 || n > (int64_t)1 << 15 || lag < 1 || (colpush != 0 && colpush != 1))
    return BAKRON_ERR_INVALID_ARG;
  return bakron::wavefront_plan_check(m, n, colpush != 0, lag, stats) == 0 ? BAKRON_OK : 1;
}

int bakron_quantize_profile(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                            int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                            int32_t* status_dev, void* stream, double* kernel_ms, int64_t* kernel_launches,
                            double* kernel_flops) {
  if (!kernel_ms || !kernel_launches || !kernel_flops) return BAKRON_ERR_INVALID_ARG;
  if (!W || !LA || !LB || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 0 || (bits >= 2 && bits <= 8))) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, bakron::kAlign) || ws_bytes < bakron::quantize_workspace_bytes(m, n))
    return BAKRON_ERR_WORKSPACE;
  bakron::KernelTimer t;
  cudaError_t e = bakron::quantize_launch(W, LA, LB, bakron::per_row(scales), bakron::alphabet_from_bits(bits), (int)m, (int)n, V, Wq, ws, status_dev,
                                          (cudaStream_t)stream, &t);
  if (e != cudaSuccess) return BAKRON_ERR_CUDA;
  for (int c = 0; c < bakron::kKernelClasses; ++c) {
    kernel_ms[c] = t.ms[c];
    kernel_launches[c] = t.launches[c];
    kernel_flops[c] = t.flops[c];
  }
  return BAKRON_OK;
}

size_t bakron_quantize_host_workspace_size(int64_t m, int64_t n) {
  if (m < 1 || n < 1 || m * n >= kMaxElems) return 0;
  using bakron::align_up;
  const size_t mn = (size_t)m * (size_t)n;
  return align_up(mn * 4) * 3 + align_up((size_t)n * n * 4) + align_up((size_t)m * m * 4) +
         align_up((size_t)m * 4) + align_up(4) + bakron::quantize_workspace_bytes(m, n);
}

int bakron_quantize_host(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                         int64_t m, int64_t n, int32_t* V, float* Wq, void* dev_ws, size_t dev_ws_bytes,
                         int32_t* status_host, void* stream) {
  if (!W || !LA || !LB || !V || !Wq || !status_host) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= kMaxElems) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 0 || (bits >= 2 && bits <= 8))) return BAKRON_ERR_INVALID_ARG;
  if (!dev_ws || !aligned(dev_ws, bakron::kAlign) || dev_ws_bytes < bakron_quantize_host_workspace_size(m, n))
    return BAKRON_ERR_WORKSPACE;
  using bakron::align_up;
  const size_t mn = (size_t)m * (size_t)n;
  char* p = static_cast<char*>(dev_ws);
  float* dW = reinterpret_cast<float*>(p);
  p += align_up(mn * 4);
  int32_t* dV = reinterpret_cast<int32_t*>(p);
  p += align_up(mn * 4);
  float* dWq = reinterpret_cast<float*>(p);
  p += align_up(mn * 4);
  float* dLA = reinterpret_cast<float*>(p);
  p += align_up((size_t)n * n * 4);
  float* dLB = reinterpret_cast<float*>(p);
  p += align_up((size_t)m * m * 4);
  float* dS = reinterpret_cast<float*>(p);
  p += align_up((size_t)m * 4);
  int32_t* dStatus = reinterpret_cast<int32_t*>(p);
  p += align_up(4);
  void* qws = p;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(dW, W, mn * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dLA, LA, (size_t)n * n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dLB, LB, (size_t)m * m * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && scales) e = cudaMemcpyAsync(dS, scales, (size_t)m * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return BAKRON_ERR_CUDA;
  e = bakron::quantize_launch(dW, dLA, dLB, bakron::per_row(scales ? dS : nullptr), bakron::alphabet_from_bits(bits), (int)m, (int)n, dV, dWq, qws, dStatus,
                              s);
  if (e != cudaSuccess) return BAKRON_ERR_CUDA;
  e = cudaMemcpyAsync(V, dV, mn * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(Wq, dWq, mn * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(status_host, dStatus, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return from_cuda(e);
}

}  // extern "C"
