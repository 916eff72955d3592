// Self-test of the bounded device waits (failure detection without a fault).
//
// Every tcgen05 kernel of the library waits on mbarriers through
// sm100::mbar_wait, which gives up after kWaitLimitNs of wall time; the
// kernel then records BD_ERR_TIMEOUT in the caller's status word, stops
// issuing work, frees its tensor memory and returns, so the context stays
// usable.  This kernel takes that path on purpose: one CTA allocates tensor
// memory the way those kernels do, then waits on a barrier that nothing ever
// arrives at.  No copy and no MMA is in flight at the wait, so nothing is left
// running when the kernel unwinds.
#include "bd_common.cuh"
#include "bd_sm100.cuh"

namespace bd {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(int32_t *dev_status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // phase 0 of `bar` never completes: the bounded wait must give up
  if (threadIdx.x == 32 && !mbar_wait(smem_u32(&bar), 0)) flag_error(dev_status, BD_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

}  // namespace
}  // namespace bd

BD_API bd_status bd_debug_wait_timeout_selftest(int32_t *dev_status, void *stream) {
  if (!dev_status) return BD_ERR_INVALID_ARG;
  if (!bd::preload_all()) return BD_ERR_CUDA;
  bd::wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
  bd::count_launches(1);
  return bd::launch_status();
}
