// Test hook for the failure path of the bounded in-kernel waits: one warp
// holds TMEM, waits on an mbarrier that nothing arrives on with a short
// limit, gives up (raising FT_DEVERR_WAIT_TIMEOUT in the error word), frees
// the TMEM and returns - the unwinding every pipelined kernel here does when
// one of its waits gives up, without faulting, trapping or hanging.
#include "ft_common.cuh"
#include "ft_internal.h"

namespace ft {

__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_slot;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    // phase 0 never completes: the wait must give up after limit_ns
    const bool ok = mbar_wait_warp(&bar, 0u, err, limit_ns);
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
    (void)ok;
}

int launch_wait_timeout_probe(uint32_t* err, int64_t limit_ns, cudaStream_t s) {
    wait_timeout_probe_kernel<<<1, 32, 0, s>>>(err, static_cast<uint64_t>(limit_ns));
    return check_launch("wait_timeout_probe_kernel", dim3(1), dim3(32), 0);
}

}  // namespace ft
