// gq_selftest.cu -- a check of the library's bounded waits that needs no
// fault: one warp waits on an mbarrier that nothing completes, through the
// same helper the GEMMs or the aggregation use, with a short limit, and the
// code it reports lands in the caller's status word.  The pages have no
// counterpart; this is how the failure path is tested without hanging or
// faulting a GPU.
#include "gq_common.cuh"
#include "gq_internal.cuh"
#include "gq_sm100.cuh"

namespace gq {
namespace {

// helper 0: the GEMMs' wait (abort flag + status word); 1: the aggregation's
// (warp-wide verdict, then the status word).  complete != 0 makes lane 0
// arrive first, so the wait succeeds and the status stays as it was.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int helper, int complete, long long limit, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int lane = threadIdx.x;
  if (lane == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
  }
  fence_barrier_init();
  __syncwarp();
  if (complete && lane == 0) mbar_arrive(&bar);
  __syncwarp();
  if (helper == 0) {
    mbar_wait(&bar, 0, &abort_flag, status, kWaitCodeSelfTest, limit);
  } else {
    const bool ok = __all_sync(FULL, mbar_wait_u32(smem_u32(&bar), 0, limit));
    if (!ok && lane == 0) atomicCAS(status, 0, kWaitCodeSelfTest);
  }
}

}  // namespace
}  // namespace gq

extern "C" int gq_selftest_bounded_wait(int helper, int complete, long long limit_cycles, int* dev_status,
                                        gq_stream stream) {
  using namespace gq;
  if (dev_status == nullptr || !(helper == 0 || helper == 1)) return GQ_ERR_INVALID_ARG;
  if (limit_cycles < 1000 || limit_cycles > 2000000000LL) return GQ_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(helper, complete, limit_cycles, dev_status);
  return launch_status();
}
