// Per-block Q8_1 arithmetic shared by the activation quantizer, the
// activation/requantize step and the tensor-core path's fused layer-1
// epilogue, so that all three produce the same codes from the same values:
// the codes of a block from its amax and d, the packed (d, s) header, and the
// gated activation g -> act(g) * up.
#pragma once

#include <cuda_fp16.h>

#include "ft_common.cuh"

namespace ft {

// Codes of N values of one block: round(v / d) clamped to [-127, 127],
// exactly as the IEEE quotient rounds.  v * rcp(d) lies within
// 2^-23 |v / d| (<= 1.6e-5 for |v / d| <= 127.5) of v / d, whose fp32
// rounding moves it by at most 4e-6 more, so both round to the same integer
// unless v * rcp(d) is within 4e-5 of a half integer.  All N values go
// through the reciprocal; only if one of them lands that near a tie (or
// d < 1e-36, where rcp(d) may overflow) do those take the division: one
// rarely taken branch per N values.  amax == 0 gives all-zero codes.
template <int N>
__device__ __forceinline__ void q8_codes(const float (&v)[N], float amax, float d, int (&q)[N]) {
    const bool fast = d >= 1.0e-36f;
    const float rd = __frcp_rn(d);
    float y[N];
    bool slow = !fast;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        y[j] = __fmul_rn(v[j], rd);
        const float t = fabsf(y[j]);
        slow |= fabsf((t - truncf(t)) - 0.5f) < 4.0e-5f;
    }
    if (slow) {
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const float t = fabsf(y[j]);
            if (!fast || fabsf((t - truncf(t)) - 0.5f) < 4.0e-5f) y[j] = __fdiv_rn(v[j], d);
        }
    }
#pragma unroll
    for (int j = 0; j < N; ++j)
        q[j] = amax != 0.0f ? min(127, max(-127, static_cast<int>(roundf(y[j])))) : 0;
}

__device__ __forceinline__ uint32_t q8_header(float d, int sum) {
    const __half hd = __float2half_rn(d);
    const __half hs = __float2half_rn(__fmul_rn(d, static_cast<float>(sum)));
    return static_cast<uint32_t>(__half_as_ushort(hd)) | (static_cast<uint32_t>(__half_as_ushort(hs)) << 16);
}

// The gated activation of one value: act(g) * up, both activations as
// g * sigmoid(z) in fp32: z = g for SiLU, and z = 2 sqrt(2/pi) (g + 0.044715
// g^3) for the tanh form of GELU, since (1 + tanh(y)) / 2 = 1 / (1 + exp(-2 y)).
__device__ __forceinline__ float act_mul(float g, float up, int kind) {
    const float z = kind == FT_ACT_SILU ? g : 1.5957691216057308f * fmaf(0.044715f * g, g * g, g);
    return __fdividef(g, 1.0f + __expf(-z)) * up;
}

}  // namespace ft
