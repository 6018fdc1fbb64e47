// Device self-test of the bounded-wait failure path (no fault, no hang): every wait in
// the kernels of this library gives up after a fixed time, records a site code in the
// device status word, raises its CTA's abort flag and returns, so that the context stays
// usable.  This kernel makes a wait run out on purpose: thread 0 waits for a phase that
// needs two arrivals but gets one; a thread of the second warp, which starts its own
// wait half a second later on a barrier nothing arrives on, must leave through the abort
// flag (before its own time limit), so the site code recorded is the first thread's.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace oattn {
namespace {

constexpr unsigned int kErrSelfTest = 0x1F0;  // site code of the self-test's wait

__global__ void selftest_wait_kernel(unsigned int* status, int* flags) {
  __shared__ uint64_t bar[2];
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 2);
    mbar_init(&bar[1], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &s_abort;
  if (threadIdx.x == 0) {
    mbar_arrive(&bar[0]);  // one of the two arrivals phase 0 needs
    const bool ok = mbar_wait(&bar[0], 0, abort, status, kErrSelfTest);
    if (flags != nullptr) flags[0] = ok ? 1 : 0;
  } else if (threadIdx.x == 32) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 500000000ull) __nanosleep(1000000);
    const bool ok = mbar_wait(&bar[1], 0, abort, status, kErrWaitFull);
    if (flags != nullptr) flags[1] = ok ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned int* status, int* flags, cudaStream_t st) {
  selftest_wait_kernel<<<1, 64, 0, st>>>(status, flags);
  return cudaGetLastError();
}

}  // namespace oattn
