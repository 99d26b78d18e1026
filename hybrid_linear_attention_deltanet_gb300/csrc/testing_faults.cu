// Fault test hook: the library's two kinds of bounded wait -- an mbarrier
// try-wait and a poll of a ready flag in global memory (the handoff between
// the per-chunk workers and the state pass of the fused prefill) -- run on
// something that never completes, so that the wait gives up after its limit,
// records GDN_ERR_TIMEOUT in the device status word and returns.  Nothing
// traps, hangs or faults; the context stays usable.
#include "../../include/gdn_testing.h"
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace sm100;

// a ready flag that nothing ever sets
__device__ uint32_t g_never_set_flag = 0;

__global__ void bounded_wait_kernel(int32_t which, uint64_t limit_ns, unsigned* status,
                                    uint32_t* flag) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  bool ok = true;
  if (which == 0) {
    mbar_init(&bar, 1);   // expects one arrival, which never comes
    fence_barrier_init();
    ok = mbar_wait(&bar, 0, limit_ns);
  } else {
    const uint64_t t0 = globaltimer_ns();
    ok = false;
    do {
      if (ld_relaxed_gpu(flag) != 0u) {
        fence_acq_rel_gpu();
        ok = true;
        break;
      }
      __nanosleep(64);
    } while (globaltimer_ns() - t0 < limit_ns);
  }
  if (!ok) flag_status(status, GDN_ERR_TIMEOUT);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_testing_bounded_wait(int32_t which, int64_t limit_ns, gdn_stream_t stream) {
  if ((which != 0 && which != 1) || limit_ns < 0 || limit_ns > 2000000000LL)
    return GDN_ERR_INVALID_ARG;
  unsigned* status = status_ptr();
  uint32_t* flag = nullptr;
  if (!status || cudaGetSymbolAddress((void**)&flag, g_never_set_flag) != cudaSuccess)
    return GDN_ERR_CUDA;
  bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(which, (uint64_t)limit_ns, status,
                                                           flag);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
