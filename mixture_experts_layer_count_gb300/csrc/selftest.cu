// selftest.cu -- gbmoe_selftest_bounded_wait: the bounded mbarrier wait that
// every pipeline wait of the GEMM kernels goes through (mbar_wait in
// ptx.cuh), run on a barrier that nothing ever completes.  The wait has to
// give up after its time limit and report GBMOE_ERR_TIMEOUT through the
// caller's error word, leaving the context usable -- the failure path of a
// stalled pipeline, exercised without a stalled pipeline.
#include <cstdint>

#include "gbmoe.h"
#include "kernels.h"
#include "ptx.cuh"

namespace gbmoe {
namespace {

__global__ void bounded_wait_selftest_kernel(int32_t *err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // phase 0 of a barrier that expects one arrival and gets none never
  // completes: the wait returns false once limit_ns has passed
  if (threadIdx.x == 0 && !mbar_wait(b, 0, limit_ns)) set_err(err, GBMOE_ERR_TIMEOUT);
}

}  // namespace
}  // namespace gbmoe

extern "C" gbmoe_status_t gbmoe_selftest_bounded_wait(int32_t *err_word, int limit_us,
                                                      gbmoe_stream_t stream) {
  using namespace gbmoe;
  if (!err_word || limit_us < 1 || limit_us > 1000000) return GBMOE_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(
      err_word, (uint64_t)limit_us * 1000ull);
  return status_from_cuda(cudaGetLastError());
}
