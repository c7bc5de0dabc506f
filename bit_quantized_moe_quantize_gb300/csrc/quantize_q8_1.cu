// Activation quantizer: fp16 rows -> Q8_1 blocks (quantize_row_q8_1 on
// FreeToken PR #185, "Fix"; format restated in ft_moe.h).
//
// HBM-bound: 2 bytes read and 1.125 bytes written per value.  Two layouts of
// the same arithmetic:
//  - quantize_q8_1_block_kernel, for batches of at least two 256-thread CTAs
//    per SM (and x 16-byte aligned): one thread owns a whole 32-value block (four 16-byte loads, 64
//    bytes in flight per thread), so amax and the code sum need no shuffles;
//  - quantize_q8_1_kernel, for small batches: eight lanes own one block (one
//    8-byte load each, amax and sum reduced with 3 shuffle steps), which puts
//    8x more threads on a batch of a few tokens.
// The flat block index runs on grid.x with a grid-stride loop, so neither
// tokens nor tokens * blocks is bound by a 65535 grid dimension (the limit
// quantize_row_q8_1 tiles around on FreeToken PR #185, "Fix").
//
// Bit-exactness: amax is exact, d = amax / 127 is an IEEE fp32 division
// (__fdiv_rn), q = roundf(x / d) with the quotient of an IEEE division (see
// q8_codes), s = d * sum(q) is one fp32 multiply, and both are rounded to fp16
// with __float2half_rn.
#include <cuda_fp16.h>

#include "ft_common.cuh"
#include "ft_internal.h"
#include "q8_1_math.cuh"

namespace ft {

// value i (0..31) of a block held as four 16-byte words of fp16
__device__ __forceinline__ float half_of(const uint4 (&raw)[4], int i) {
    const uint4 r = raw[i >> 3];
    const uint32_t w = (i & 6) == 0 ? r.x : (i & 6) == 2 ? r.y : (i & 6) == 4 ? r.z : r.w;
    const __half2 h = *reinterpret_cast<const __half2*>(&w);
    return (i & 1) ? __high2float(h) : __low2float(h);
}

__global__ void __launch_bounds__(256) quantize_q8_1_block_kernel(const uint4* __restrict__ x,
                                                                  uint32_t* __restrict__ out, int64_t n_blocks) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; blk < n_blocks; blk += stride) {
        uint4 raw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) raw[c] = __ldg(x + blk * 4 + c);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(half_of(raw, i)));
        const float d = __fdiv_rn(amax, 127.0f);
        // q8_codes, written out over the raw halves (no 32-value array): the
        // codes from the reciprocal first; if any value lands near a tie (or
        // d < 1e-36), the block is redone with the division for those values
        const bool fast = d >= 1.0e-36f;
        const float rd = __frcp_rn(d);
        uint32_t packed[8];
        int sum = 0;
        bool slow = !fast;
#pragma unroll
        for (int i = 0; i < 8; ++i) packed[i] = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float y = __fmul_rn(half_of(raw, i), rd);
            const float t = fabsf(y);
            slow |= fabsf((t - truncf(t)) - 0.5f) < 4.0e-5f;
            const int qi = amax != 0.0f ? min(127, max(-127, static_cast<int>(roundf(y)))) : 0;
            sum += qi;
            packed[i >> 2] |= (static_cast<uint32_t>(qi) & 0xFFu) << (8 * (i & 3));
        }
        if (slow) {
            // reloaded (from L1 / L2) rather than kept: holding the 32 values
            // across the common path would double the registers
            uint4 raw2[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) raw2[c] = __ldg(x + blk * 4 + c);
            sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) packed[i] = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float v = half_of(raw2, i);
                float y = __fmul_rn(v, rd);
                const float t = fabsf(y);
                if (!fast || fabsf((t - truncf(t)) - 0.5f) < 4.0e-5f) y = __fdiv_rn(v, d);
                const int qi = amax != 0.0f ? min(127, max(-127, static_cast<int>(roundf(y)))) : 0;
                sum += qi;
                packed[i >> 2] |= (static_cast<uint32_t>(qi) & 0xFFu) << (8 * (i & 3));
            }
        }
        uint32_t* ob = out + blk * (Q8_1_BYTES / 4);
        ob[0] = q8_header(d, sum);
#pragma unroll
        for (int i = 0; i < 8; ++i) ob[1 + i] = packed[i];
    }
}

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
        q8_codes<4>(v, amax, d, q);
        uint32_t packed = 0;
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sum += q[j];
            packed |= (static_cast<uint32_t>(q[j]) & 0xFFu) << (8 * j);
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(group_mask, sum, o);
        uint8_t* ob = out + blk * Q8_1_BYTES;
        *reinterpret_cast<uint32_t*>(ob + 4 + 4 * sub) = packed;
        if (sub == 0) *reinterpret_cast<uint32_t*>(ob) = q8_header(d, sum);
    }
}

int launch_quantize_q8_1(const void* x, void* act, int64_t tokens, int64_t ncols, cudaStream_t s) {
    const int64_t n_blocks = tokens * (ncols / QK);
    if (n_blocks == 0) return FT_OK;
    const int threads = 256;
    const int64_t cap = 0x7FFFFFFF;
    const bool x16 = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;   // 16-byte loads need it
    if (x16 && n_blocks >= 2 * static_cast<int64_t>(threads) * sm_count()) {
        // one thread per block, every block of the batch in flight at once
        // (grid.x up to 2^31 - 1; larger batches take the grid-stride loop)
        const int64_t want = (n_blocks + threads - 1) / threads;
        const dim3 grid(static_cast<unsigned>(want < cap ? want : cap));
        quantize_q8_1_block_kernel<<<grid, threads, 0, s>>>(static_cast<const uint4*>(x),
                                                             static_cast<uint32_t*>(act), n_blocks);
        return check_launch("quantize_q8_1_block_kernel", grid, dim3(threads), 0);
    }
    const int64_t want = (n_blocks * 8 + threads - 1) / threads;
    const dim3 grid(static_cast<unsigned>(want < cap ? want : cap));
    quantize_q8_1_kernel<<<grid, threads, 0, s>>>(static_cast<const uint2*>(x), static_cast<uint8_t*>(act),
                                                  n_blocks);
    return check_launch("quantize_q8_1_kernel", grid, dim3(threads), 0);
}

// ---------------------------------------------------------------------------
// Gated activation + Q8_1 requantization: the step between the two expert
// layers (gelu_tanh_and_mul right after the routed matmul on FreeToken PR
// #185, "Problem"; SiLU*up between layer 1 and layer 2 on
// nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6).  h [rows][2 I] fp32, gate half
// then up half -> [rows][I/32] Q8_1 of a = act(gate) * up.  a lives only in
// registers: no fp32 or fp16 copy of it is written and read back by a
// separate quantizer.
//
// Both activations are g * sigmoid(z) in fp32: z = g for SiLU, and
// z = 2 sqrt(2/pi) (g + 0.044715 g^3) for the tanh form of GELU, since
// (1 + tanh(y)) / 2 = 1 / (1 + exp(-2 y)); the sigmoid form has no
// cancellation where tanh(y) approaches -1.  The exponential and the
// division are the fast hardware forms (__expf, __fdividef): relative error
// about 1e-6 for |z| <= 20, so a code can differ from that of the exactly
// computed a only where a / d lies within ~1e-4 of a rounding boundary, and
// where the exact a is below 2^-126 |g| (exp(-z) past 2^126) the result is 0,
// in blocks whose fp16 scale is 0 anyway or whose codes there are 0.
//
// HBM-bound: 8 bytes read and 1.125 bytes written per output value.  Eight
// lanes own one block (four gate and four up values each, one 16-byte load
// per half); each thread loads its kActUnroll units before it uses any, so
// 32 * kActUnroll bytes per thread are in flight.

constexpr int kActUnroll = 1;

__global__ void __launch_bounds__(256) act_mul_quantize_q8_1_kernel(const float4* __restrict__ h,
                                                                    uint8_t* __restrict__ out, int64_t n_blocks,
                                                                    uint32_t nb_row, int kind) {
    const int64_t total = n_blocks * 8;
    const uint32_t lane = lane_id();
    const uint32_t group_mask = 0xFFu << (lane & 24u);
    const uint32_t sub = lane & 7u;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * (256 * kActUnroll) + threadIdx.x;
    // block (row r, column block b) of the first unit; unit u is 32 u blocks on
    int64_t r = (i0 >> 3) / nb_row;
    uint32_t b = static_cast<uint32_t>((i0 >> 3) - r * nb_row);
    float4 g[kActUnroll], up[kActUnroll];
#pragma unroll
    for (int u = 0; u < kActUnroll; ++u) {
        if (i0 + u * 256 < total) {
            // float4 index of the gate quad: row r holds 16 nb_row float4s
            const int64_t gi = r * (16 * static_cast<int64_t>(nb_row)) + 8 * static_cast<int64_t>(b) + sub;
            g[u] = __ldg(h + gi);
            up[u] = __ldg(h + gi + 8 * static_cast<int64_t>(nb_row));
        } else {
            g[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            up[u] = g[u];
        }
        b += 32;
        while (b >= nb_row) {
            b -= nb_row;
            ++r;
        }
    }
#pragma unroll
    for (int u = 0; u < kActUnroll; ++u) {
        const int64_t i = i0 + u * 256;
        const float v[4] = {act_mul(g[u].x, up[u].x, kind), act_mul(g[u].y, up[u].y, kind),
                            act_mul(g[u].z, up[u].z, kind), act_mul(g[u].w, up[u].w, kind)};
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(group_mask, amax, o));
        const float d = __fdiv_rn(amax, 127.0f);
        int q[4];
        q8_codes<4>(v, amax, d, q);
        uint32_t packed = 0;
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sum += q[j];
            packed |= (static_cast<uint32_t>(q[j]) & 0xFFu) << (8 * j);
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(group_mask, sum, o);
        if (i < total) {
            uint8_t* ob = out + (i >> 3) * Q8_1_BYTES;
            *reinterpret_cast<uint32_t*>(ob + 4 + 4 * sub) = packed;
            if (sub == 0) *reinterpret_cast<uint32_t*>(ob) = q8_header(d, sum);
        }
    }
}

int launch_act_mul_quantize_q8_1(const float* h, void* act, int64_t rows, int64_t n_inter, int kind,
                                 cudaStream_t s) {
    const int64_t nb_row = n_inter / QK;
    const int64_t n_blocks = rows * nb_row;
    if (n_blocks == 0) return FT_OK;
    const int64_t per_cta = 256 * kActUnroll;
    const int64_t want = (n_blocks * 8 + per_cta - 1) / per_cta;
    if (want > 0x7FFFFFFF) return fail(FT_ERR_SIZE, "rows * n_inter too large for one launch");
    const dim3 grid(static_cast<unsigned>(want));
    act_mul_quantize_q8_1_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(h), static_cast<uint8_t*>(act),
                                                      n_blocks, static_cast<uint32_t>(nb_row), kind);
    return check_launch("act_mul_quantize_q8_1_kernel", grid, dim3(256), 0);
}

}  // namespace ft
