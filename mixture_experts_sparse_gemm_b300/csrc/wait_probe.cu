// Probe of the failure path of the bounded device-side waits (moe_wait_probe).
//
// The tensor-core kernels wait in two ways: on an mbarrier phase (the ring of
// shared-memory stages and the TMEM accumulators) and on a counter in global
// memory that other CTAs advance (the down tiles of the fused expert launch wait
// for the up tiles that write their rows).  Both give up after the wait limit,
// record kErrWaitTimeout in the device error word and return, so a stalled
// kernel ends instead of hanging and the host learns of it through
// moe_check_device_error.  This kernel runs exactly those two routines, so the
// give-up path can be exercised on purpose without stalling a real layer:
//   1. wait until *flag >= target (the caller decides whether anything ever sets it);
//   2. if that succeeded, arrive on a fresh mbarrier, whose phase then completes;
//      either way, wait on that phase with the abort flag cleared -- after a failed
//      counter wait nothing arrives, so this wait gives up too.
// A satisfied flag gives two successful waits and no error; an unsatisfied one
// gives two timeouts, each after the limit.
#include "tc_common.cuh"

namespace moe {
namespace {

__global__ void wait_probe_kernel(const int32_t *flag, int32_t target, uint64_t limit_ns, unsigned *err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    tc::mbar_init(tc::smem_u32(&bar), 1);
    tc::fence_mbarrier_init();
    abort_flag = 0;
    const bool ok = tc::wait_counter_bounded(flag, target, &abort_flag, err, limit_ns);
    if (ok) tc::mbar_arrive(tc::smem_u32(&bar));
    abort_flag = 0;
    (void)tc::wait_bounded(tc::smem_u32(&bar), 0, &abort_flag, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_probe(const int32_t *flag, int32_t target, uint64_t limit_ns, unsigned *err,
                              cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(flag, target, limit_ns, err);
    return cudaGetLastError();
}

}  // namespace moe
