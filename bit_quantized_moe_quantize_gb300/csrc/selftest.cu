// Test and measurement hooks.
//
// wait_timeout_probe_kernel - the failure path of the bounded in-kernel
// waits: one warp holds TMEM, waits on an mbarrier that nothing arrives on
// with a short limit, gives up (raising FT_DEVERR_WAIT_TIMEOUT in the error
// word), frees the TMEM and returns - the unwinding every pipelined kernel
// here does when one of its waits gives up, without faulting, trapping or
// hanging.
//
// stream_read_kernel - a plain streaming read of n 16-byte words (four
// independent 16-byte loads per thread in flight, grid of 4 CTAs of 512
// threads per SM): the time the memory system needs to deliver a buffer of
// that size to the SMs at all, against which a bandwidth-bound kernel of the
// same size is judged.
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

__global__ void __launch_bounds__(512) stream_read_kernel(const uint4* __restrict__ w, int64_t n16, uint32_t* sink) {
    uint32_t acc = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = __ldg(w + i), b = __ldg(w + i + stride), c = __ldg(w + i + 2 * stride), d = __ldg(w + i + 3 * stride);
        acc += a.x ^ b.y ^ c.z ^ d.w;
    }
    for (; i < n16; i += stride) acc += __ldg(w + i).x;
    if (acc == 0x9E3779B9u) sink[0] = acc;   // keeps the loads; practically never taken
}

int launch_stream_read(const void* buf, int64_t n16, uint32_t* sink, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(4 * sm_count())), block(512);
    stream_read_kernel<<<grid, block, 0, s>>>(static_cast<const uint4*>(buf), n16, sink);
    return check_launch("stream_read_kernel", grid, block, 0);
}

int launch_wait_timeout_probe(uint32_t* err, int64_t limit_ns, cudaStream_t s) {
    wait_timeout_probe_kernel<<<1, 32, 0, s>>>(err, static_cast<uint64_t>(limit_ns));
    return check_launch("wait_timeout_probe_kernel", dim3(1), dim3(32), 0);
}

}  // namespace ft
