// Self-test of the failure-detection path: a bounded mbarrier wait that no
// arrival ever completes.  Every wait in the library's kernels gives up after
// a time limit, sets the device status word to DSI_ERR_TIMEOUT and lets its
// CTA drain and exit; this kernel runs exactly that path on purpose, so a
// test can check that the status reaches the host and that the context stays
// usable afterwards.  It faults nothing and ends on its own.
#include "kernels.h"
#include "tc_common.cuh"

namespace dsi {
using namespace tc;

namespace {

__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(uint64_t limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);        // one arrival expected; none is ever made
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  volatile int* ab = &abort_flag;
  // the warp-uniform form the kernels use before collective instructions
  const bool ok = warp_wait(&bar, 0, ab, err, limit_ns);
  (void)ok;
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, int* err, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, err);
  note_launch();
  return cudaGetLastError();
}

}  // namespace dsi
