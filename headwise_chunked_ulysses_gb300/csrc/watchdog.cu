// Self-test of the failure detection every kernel of the library relies on.
//
// Each mbarrier wait in the kernels is bounded (ptx.cuh): when a wait runs
// past its limit the thread raises the CTA's abort flag, writes a timeout
// code into the device status word and returns, the kernel skips the rest of
// its work and exits, and upipe_sync_status() reports UPIPE_ETIMEOUT.  The
// layer kernels never reach that path in a correct run, so this file gives a
// kernel that does, on purpose and safely: one CTA initialises an mbarrier
// that nothing ever arrives on and waits on it with a short limit, first with
// the per-thread form of the wait, then (second launch) with the
// warp-collective form.  No copy, bulk transfer or tensor-core operation is
// issued, so nothing is in flight when the waits give up; the kernel returns
// after at most `limit` SM clocks plus one polling interval.
//
// Built unless UPIPE_SELFTEST is defined to 0; without it the entry point
// returns UPIPE_EUNSUPPORTED.
#include "ptx.cuh"
#include "upipe.h"
#include "upipe_internal.h"

#ifndef UPIPE_SELFTEST
#define UPIPE_SELFTEST 1
#endif

namespace upipe {
namespace {

constexpr int kSiteSelftest = 0x7E;  // status word site id of the self-test waits

#if UPIPE_SELFTEST
__global__ void __launch_bounds__(64) watchdog_selftest_kernel(int* status, long long limit, int warp_form) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival would complete phase 0; none comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Watch w{&abort_flag, status};
  const bool ok = warp_form ? mbar_wait_warp(&bar, 0, w, kSiteSelftest + 1, limit)
                            : mbar_wait(&bar, 0, w, kSiteSelftest, limit);
  (void)ok;  // false: the wait gave up (or saw another thread give up)
  __syncthreads();
}
#endif

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" int upipe_watchdog_selftest(long long limit_cycles, int warp_form, void* stream) {
#if UPIPE_SELFTEST
  if (limit_cycles < 1000 || limit_cycles > 1000000000LL) return UPIPE_EINVAL;
  if (warp_form != 0 && warp_form != 1) return UPIPE_EINVAL;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  int* status = device_status_word();
  if (!status) return UPIPE_ECUDA;
  watchdog_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_cycles, warp_form);
  return cudaGetLastError() == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
#else
  (void)limit_cycles;
  (void)warp_form;
  (void)stream;
  return UPIPE_EUNSUPPORTED;
#endif
}
