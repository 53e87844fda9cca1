// Check of the bounded-wait failure path that every pipeline kernel relies on.
//
// The tensor-core kernels never wait without a bound: each mbarrier wait gives
// up after a limit of %globaltimer time, every lane of the waiting warp agrees
// on the outcome (warp_wait), and the kernel then sets PA_DEVERR_WAIT in the
// device error word and unwinds instead of hanging. Making one of those waits
// run out inside a real pipeline would need a stalled copy or MMA, which is not
// something to provoke on a shared GPU. This kernel runs the same wait code on
// an mbarrier that nothing ever completes, with nothing in flight, and takes
// the same failure branch, so the host can check that the bound ends the wait,
// that the warp agrees and that the error bit reaches pa_get_device_error.
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace pa {
namespace {

// One warp. Phase 0 of the barrier is completed by lane 0 itself and must be
// seen; phase 1 is never completed, so its wait runs out after limit_ns.
// report[0]: 1 when the completed phase was seen by the warp;
// report[1]: lanes whose own wait on phase 1 gave up (32 expected);
// report[2]: 1 when the warp agreed on the failure (warp_wait returned false);
// report[3]: nanoseconds lane 0 spent in the failed wait.
__global__ void bounded_wait_check_kernel(unsigned long long limit_ns, int64_t *report, unsigned int *err) {
    __shared__ __align__(8) uint64_t bar;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::mbar_fence_init();
    }
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(&bar);            // completes phase 0
    const bool seen = sm100::warp_wait(&bar, 0, limit_ns);

    const unsigned long long t0 = sm100::globaltimer_ns();
    const bool own = sm100::mbar_wait(&bar, 1, limit_ns);
    const unsigned long long t1 = sm100::globaltimer_ns();
    const unsigned gave_up = __popc(__ballot_sync(0xffffffffu, !own));
    const bool agreed = sm100::warp_wait(&bar, 1, limit_ns);
    if (!agreed && lane == 0) raise_error(err, PA_DEVERR_WAIT);   // the pipeline kernels' failure branch
    if (lane == 0 && report) {
        report[0] = seen ? 1 : 0;
        report[1] = gave_up;
        report[2] = agreed ? 0 : 1;
        report[3] = (int64_t)(t1 - t0);
    }
}

}  // namespace

int launch_bounded_wait_check(unsigned long long limit_ns, int64_t *report, unsigned int *err,
                              cudaStream_t stream) {
    bounded_wait_check_kernel<<<1, 32, 0, stream>>>(limit_ns, report, err);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace pa
