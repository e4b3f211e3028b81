// A bounded wait that runs out, on purpose and harmlessly (include/ttt_kernels.h,
// ttt_k_wait_limit_probe).  Every kernel's spin-waits go through mbar_wait
// (ptx.cuh): after the wait limit it raises the CTA's abort flag, records a
// code in the caller's error word and returns false, and every other waiter of
// the CTA stops at its next check of the flag.  This kernel makes two threads
// wait on an mbarrier phase that nothing completes, so that a test can check
// that mechanism and that the context stays usable afterwards.  Nothing traps
// and every loop is bounded by time.
#include "ttt.h"
#include "ttt_kernels.h"
#include "ptx.cuh"

namespace ttt {
namespace {

constexpr uint64_t kLateStartNs = 100000000ull;  // the second waiter starts 100 ms later

__global__ void __launch_bounds__(64, 1) wait_limit_kernel(int* err, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (lane == 0) {
    if (warp == 1) {  // start late, so that warp 0's limit runs out first
      const uint64_t s = globaltimer();
      while (globaltimer() - s < kLateStartNs) __nanosleep(1000);
    }
    const uint64_t t0 = globaltimer();
    const bool ok = mbar_wait(&bar, 0, &abort_flag, err, warp == 0 ? DERR_TIMEOUT_EPILOGUE : DERR_TIMEOUT_MMA);
    status[2 * warp] = ok ? 1 : 0;
    status[2 * warp + 1] = (int)((globaltimer() - t0) / 1000000ull);  // milliseconds waited
  }
}

}  // namespace
}  // namespace ttt

extern "C" int ttt_k_wait_limit_probe(int32_t* err, int32_t* status, void* stream) {
  if (!err || !status) return TTT_ERR_ARG;
  ttt::wait_limit_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(err, status);
  return cudaGetLastError() == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}
