// Self-test of the bounded waits (vq_wait_selftest).
//
// The pipelined projection kernels never spin without a limit: every wait on
// one of their mbarriers gives up after kWaitTimeoutCycles, records
// kErrWaitTimeout in a status word and lets the block wind down, and a wait
// that sees another warp's abort flag gives up at once. This kernel runs those
// same helpers (wait_or_abort, wait_bounded) in one block against a barrier
// that completes and a barrier that nothing ever arrives at, and reports what
// each wait returned and how long it took, so that a test can check on the GPU
// that a stuck pipeline ends with an error status instead of a hang.
#include "vq_gemm.cuh"

namespace vq {
namespace {

// report[0]  1 if the wait on the completed barrier succeeded
// report[1]  its duration in SM cycles
// report[2]  1 if the wait on the barrier nothing arrives at succeeded (expect 0)
// report[3]  its duration (expect about kWaitTimeoutCycles)
// report[4]  the block's abort flag after it (expect 1)
// report[5]  1 if a second warp's wait on that barrier succeeded (expect 0)
// report[6]  its duration (short: it sees the abort flag)
// report[7]  the duration of the teardown wait on that barrier (wait_bounded)
// status[0]  OR of the flags of the two aborting waits; status[1] of the teardown wait
__global__ void __launch_bounds__(64) wait_selftest_kernel(int32_t* status, long long* report) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const uint32_t never = smem_addr(&bars[0]), done = smem_addr(&bars[1]);
  if (threadIdx.x == 0) {
    mbar_init(never, 1);
    mbar_init(done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(done);                 // completes phase 0 of `done`
    long long t0 = clock64();
    bool ok = wait_or_abort(done, 0u, &abort_flag, status);
    report[0] = ok;
    report[1] = clock64() - t0;
    t0 = clock64();
    ok = wait_or_abort(never, 0u, &abort_flag, status);
    report[2] = ok;
    report[3] = clock64() - t0;
    report[4] = abort_flag;
  }
  __syncthreads();
  if (threadIdx.x == 32) {
    long long t0 = clock64();
    const bool ok = wait_or_abort(never, 0u, &abort_flag, status);
    report[5] = ok;
    report[6] = clock64() - t0;
    t0 = clock64();
    wait_bounded(never, 0u, status + 1);
    report[7] = clock64() - t0;
  }
}

}  // namespace
}  // namespace vq

extern "C" int vq_wait_selftest(int32_t* status, int64_t* report, void* stream) {
  if (!status || !report) return VQ_EINVAL;
  if (((uintptr_t)status & 3u) || ((uintptr_t)report & 7u)) return VQ_EALIGN;
  int rc = vq::num_sms_current_device(nullptr);
  if (rc) return rc;
  vq::wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      status, reinterpret_cast<long long*>(report));
  return cudaGetLastError() == cudaSuccess ? VQ_OK : VQ_ECUDA;
}
