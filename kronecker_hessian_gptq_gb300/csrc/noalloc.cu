// noalloc.cu -- bakron_quantize for callers that cannot allocate device memory.
//
// The solve needs scratch space (the double-float state planes and a small
// header).  bakron_quantize takes it from the caller.  Some callers cannot
// provide it: a plugin running inside a host application whose device memory
// is entirely owned by another allocator, or a latency-critical path that
// must not call cudaMalloc, which can synchronize the whole device.  For them
// this file keeps one fixed scratch area in a file-scope device array and
// hands it to the ordinary solve.  The array is part of the library's device
// image: every GPU that loads the library holds it until the process exits.
//
// The paper has no counterpart to this; it is an interface convenience only.
#include <mutex>

#include "bakron.h"
#include "internal.h"

namespace {

static_assert(BAKRON_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size keeps 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[BAKRON_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
struct ScratchAddress {
  void* ptr = nullptr;              // device address of the array
  unsigned long long ctx_id = 0;    // context it belongs to (0: none yet)
};
ScratchAddress g_scratch_address[kMaxDevices];  // per device ordinal
std::mutex g_scratch_mutex;

// Device address of the array on the current device.  The name
// g_noalloc_scratch in host code is only a host-side stand-in for the symbol,
// so the real address is asked from the runtime once per device, with that
// device current, and cached together with the id of the context it belongs
// to; a new context on the device (after cudaDeviceReset) looks it up again.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  e = bakron::current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddress& a = g_scratch_address[dev];
  if (a.ptr == nullptr || a.ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    a.ptr = p;
    a.ctx_id = ctx;
  }
  *out = a.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" int bakron_quantize_noalloc(const float* W, const float* LA, const float* LB, const float* scales,
                                       int bits, int64_t m, int64_t n, int32_t* V, float* Wq,
                                       int32_t* status_dev, void* stream) {
  if (!W || !LA || !LB || !V || !Wq || !status_dev) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m * n >= ((int64_t)1 << 31)) return BAKRON_ERR_INVALID_ARG;
  if (!(bits == 0 || (bits >= 2 && bits <= 8))) return BAKRON_ERR_INVALID_ARG;
  if ((const void*)Wq == (const void*)W || (const void*)V == (const void*)W || (void*)V == (void*)Wq)
    return BAKRON_ERR_INVALID_ARG;
  if (bakron::quantize_workspace_bytes(m, n) > (size_t)BAKRON_NOALLOC_SCRATCH_BYTES) return BAKRON_ERR_WORKSPACE;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return BAKRON_ERR_CUDA;
  // The solve initializes every scratch byte it reads (status word, header
  // and state planes), so what an earlier call left there does not matter.
  cudaError_t e = bakron::quantize_launch(W, LA, LB, bakron::per_row(scales), bakron::alphabet_from_bits(bits), (int)m, (int)n, V, Wq, ws, status_dev,
                                          (cudaStream_t)stream);
  return e == cudaSuccess ? BAKRON_OK : BAKRON_ERR_CUDA;
}
