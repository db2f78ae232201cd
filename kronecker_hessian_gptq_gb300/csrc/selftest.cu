// selftest.cu -- the device-side timeout path, exercised on purpose.
//
// The tensor-core kernels wait on mbarriers with a bounded wait (tc.cuh:
// mbar_wait gives up after 2^28 cycles, about 0.1 s) and report
// BAKRON_DEV_TIMEOUT instead of hanging.  This kernel runs the same wait on
// an mbarrier that nothing ever arrives on, so the wait must run out; the
// host then reads the status word, and the context stays usable.  Nothing
// faults, traps or hangs: one thread spins for the bounded time and returns.
#include "bakron.h"
#include "internal.h"
#include "tc.cuh"

namespace bakron {
namespace {

__global__ void wait_selftest_kernel(int32_t* status) {
  __shared__ uint64_t mbar;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&mbar)));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool broken = false;
    mbar_wait(&mbar, 0u, broken);  // phase 0 never completes: no thread arrives
    if (broken) atomicOr(status, BAKRON_DEV_TIMEOUT);
  }
}

}  // namespace

cudaError_t wait_selftest_launch(int32_t* status_dev, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status_dev);
  return cudaGetLastError();
}

}  // namespace bakron
