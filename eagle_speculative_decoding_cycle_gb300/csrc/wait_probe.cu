// Failure-detection probe: runs the library's bounded device waits on conditions that
// nothing will ever satisfy, so a test can check that each wait gives up after its time
// limit, latches the timeout code in the status word the host reads, and returns with the
// context still usable. No fault, trap or unbounded loop is involved: both waits stop on
// %globaltimer.
#include "../../include/eagle.h"
#include "../../include/eagle_ops.h"
#include "common.cuh"
#include "tc_common.cuh"

namespace {
using namespace eagle;

__global__ void wait_probe_k(int kind, const unsigned* counter, int* err, int* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  bool ok;
  if (kind == 0) {
    // the TMA/MMA pipelines' wait: an mbarrier phase that no thread or copy completes
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
  } else {
    // the split-tile owner's wait: a counter that nothing increments
    ok = grid_wait(counter, 1u, &abort_flag, err, false);
  }
  *result = ok ? 1 : 0;
}

}  // namespace

extern "C" int eagle_op_wait_probe(void* stream, int kind, const unsigned* d_counter, int* d_err, int* d_result) {
  if ((kind != 0 && kind != 1) || !d_err || !d_result || (kind == 1 && !d_counter)) return EAGLE_EINVAL;
  wait_probe_k<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(kind, d_counter, d_err, d_result);
  return cudaGetLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ECUDA;
}
