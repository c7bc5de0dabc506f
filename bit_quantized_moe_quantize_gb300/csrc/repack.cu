// One-time repack of Q4_0 expert weights from the stored array of 18-byte
// blocks (fp16 d, 16 nibble bytes) into a structure of arrays: the nibble
// bytes of every block, 16 per block in block order (16-byte aligned rows of
// any length), then the fp16 scales in block order.  An export for consumers
// that want the nibbles and scales apart (TMA boxes of whole 16-byte chunks,
// scale vectors); the matmul kernels read the stored layout directly.
//
// HBM-bound byte move: 18 bytes read and 18 written per block.  One thread
// per block: nine 2-byte loads (blocks are only 2-byte aligned), one 16-byte
// store of the nibbles and one 2-byte store of the scale.
#include "ft_common.cuh"
#include "ft_internal.h"

namespace ft {

__global__ void __launch_bounds__(256) repack_q4_0_soa_kernel(const uint16_t* __restrict__ blocks,
                                                              uint4* __restrict__ qs, uint16_t* __restrict__ d,
                                                              int64_t n_blocks) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < n_blocks; b += stride) {
        const uint16_t* src = blocks + b * (Q4_0_BYTES / 2);
        uint32_t h[Q4_0_BYTES / 2];
#pragma unroll
        for (int i = 0; i < Q4_0_BYTES / 2; ++i) h[i] = __ldg(src + i);
        d[b] = static_cast<uint16_t>(h[0]);
        qs[b] = make_uint4(h[1] | (h[2] << 16), h[3] | (h[4] << 16), h[5] | (h[6] << 16), h[7] | (h[8] << 16));
    }
}

int launch_repack_q4_0_soa(const void* blocks, void* qs, void* d, int64_t n_blocks, cudaStream_t s) {
    if (n_blocks == 0) return FT_OK;
    const int threads = 256;
    const int64_t want = (n_blocks + threads - 1) / threads;
    const dim3 grid(static_cast<unsigned>(want < 0x7FFFFFFF ? want : 0x7FFFFFFF));
    repack_q4_0_soa_kernel<<<grid, threads, 0, s>>>(static_cast<const uint16_t*>(blocks), static_cast<uint4*>(qs),
                                                    static_cast<uint16_t*>(d), n_blocks);
    return check_launch("repack_q4_0_soa_kernel", grid, dim3(threads), 0);
}

}  // namespace ft
