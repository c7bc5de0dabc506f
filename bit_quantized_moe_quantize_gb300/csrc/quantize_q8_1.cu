// Activation quantizer: fp16 rows -> Q8_1 blocks (quantize_row_q8_1 on
// FreeToken PR #185, "Fix"; format restated in ft_moe.h).
//
// HBM-bound: 2 bytes read and 1.125 bytes written per value.  Eight lanes
// own one 32-value block (four values each, one 8-byte load per lane); the
// block's amax and integer sum are reduced with 3 shuffle steps inside the
// 8-lane group.  The flat block index runs on grid.x with a grid-stride loop,
// so neither tokens nor tokens * blocks is bound by a 65535 grid dimension
// (the limit quantize_row_q8_1 tiles around on FreeToken PR #185, "Fix").
//
// Bit-exactness: amax is exact, d = amax / 127 and x / d are IEEE fp32
// divisions (__fdiv_rn), q = roundf (half away from zero), s = d * sum(q) is
// one fp32 multiply, and both are rounded to fp16 with __float2half_rn.
#include <cuda_fp16.h>

#include "ft_common.cuh"
#include "ft_internal.h"

namespace ft {

__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const uint2* __restrict__ x, uint8_t* __restrict__ out,
                                                            int64_t n_blocks) {
    const int64_t total = n_blocks * 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint32_t lane = lane_id();
    const uint32_t group_mask = 0xFFu << (lane & 24u);
    const uint32_t sub = lane & 7u;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t blk = i >> 3;
        const uint2 raw = __ldg(x + i);   // values 4*sub .. 4*sub+3 of block blk
        const __half2 h01 = *reinterpret_cast<const __half2*>(&raw.x);
        const __half2 h23 = *reinterpret_cast<const __half2*>(&raw.y);
        const float v[4] = {__low2float(h01), __high2float(h01), __low2float(h23), __high2float(h23)};
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(group_mask, amax, o));
        const float d = __fdiv_rn(amax, 127.0f);
        int q[4];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int qi = 0;
            if (amax != 0.0f) {
                qi = static_cast<int>(roundf(__fdiv_rn(v[j], d)));
                qi = min(127, max(-127, qi));
            }
            q[j] = qi;
            sum += qi;
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(group_mask, sum, o);
        uint8_t* ob = out + blk * Q8_1_BYTES;
        const uint32_t packed = (static_cast<uint32_t>(q[0]) & 0xFFu) | ((static_cast<uint32_t>(q[1]) & 0xFFu) << 8) |
                                ((static_cast<uint32_t>(q[2]) & 0xFFu) << 16) |
                                ((static_cast<uint32_t>(q[3]) & 0xFFu) << 24);
        *reinterpret_cast<uint32_t*>(ob + 4 + 4 * sub) = packed;
        if (sub == 0) {
            const __half hd = __float2half_rn(d);
            const __half hs = __float2half_rn(__fmul_rn(d, static_cast<float>(sum)));
            const uint32_t ds = static_cast<uint32_t>(__half_as_ushort(hd)) |
                                (static_cast<uint32_t>(__half_as_ushort(hs)) << 16);
            *reinterpret_cast<uint32_t*>(ob) = ds;
        }
    }
}

int launch_quantize_q8_1(const void* x, void* act, int64_t tokens, int64_t ncols, cudaStream_t s) {
    const int64_t n_blocks = tokens * (ncols / QK);
    if (n_blocks == 0) return FT_OK;
    const int threads = 256;
    // one thread per 8-byte load: every load of the batch is issued at once
    // (grid.x up to 2^31 - 1; larger batches take the grid-stride loop)
    const int64_t want = (n_blocks * 8 + threads - 1) / threads;
    const int64_t cap = 0x7FFFFFFF;
    const dim3 grid(static_cast<unsigned>(want < cap ? want : cap));
    quantize_q8_1_kernel<<<grid, threads, 0, s>>>(static_cast<const uint2*>(x), static_cast<uint8_t*>(act),
                                                  n_blocks);
    return check_launch("quantize_q8_1_kernel", grid, dim3(threads), 0);
}

}  // namespace ft
