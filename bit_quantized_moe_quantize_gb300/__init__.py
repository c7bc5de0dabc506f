"""GB300 (sm_103a) routed Q4_0 x Q8_1 MoE expert matmul.

The computation lives in ``libft_moe.so`` (hand-written CUDA, C ABI in
``include/ft_moe.h``); this package is its thin Python binding plus the seeded
synthetic-input generator used by the tests and the benchmark.

    act = quantize_q8_1(x_fp16)                       # fp16 [T, K] -> Q8_1
    out = moe_q4_0_q8_1(weights_q4_0, act, topk_ids)  # fp32 [T, k, N]
    out = moe_q4_0_fp16(weights_q4_0, x_fp16, topk_ids)  # the same, from fp16 (one launch when decoding)
    a2 = act_mul_quantize_q8_1(out, ACT_SILU)         # Q8_1 of silu(gate) * up per slot
    y, h, a2 = moe_ffn_q4_0_q8_1(w13, w2, act, topk_ids, ACT_SILU)   # both expert layers
"""

from ._lib import (ACT_GELU_TANH, ACT_SILU, FT_DEVERR_BAD_EXPERT_ID, FT_DEVERR_WAIT_TIMEOUT,
                   FT_DEVERR_WORKSPACE_GUARD, FT_PATH_AUTO, FT_PATH_GEMM, FT_PATH_GEMV, FT_PATH_GEMV_DP4A, FtError,
                   act_mul_quantize_q8_1, block_dots, debug_stream_read, debug_wait_timeout, ffn_reserve, last_error, load,
                   moe_ffn_q4_0_q8_1, moe_gguf_q8_1, moe_q4_0_fp16, moe_q4_0_q8_1, moe_q4_0_q8_1_act, moe_q4_0_q8_1_ep,
                   moe_q4_0_q8_1_slots, profile_enable,
                   profile_read, quantize_q8_1, read_device_error, repack_q4_0_soa, release, reserve, route_offsets, selected_path,
                   set_path, workspace_bytes, WEIGHT_TYPES)

__all__ = [
    "ACT_GELU_TANH", "ACT_SILU", "WEIGHT_TYPES", "moe_gguf_q8_1", "repack_q4_0_soa", "act_mul_quantize_q8_1", "moe_ffn_q4_0_q8_1", "moe_q4_0_q8_1_act", "ffn_reserve", "moe_q4_0_fp16", "FT_DEVERR_BAD_EXPERT_ID", "FT_DEVERR_WAIT_TIMEOUT", "FT_DEVERR_WORKSPACE_GUARD", "debug_wait_timeout", "debug_stream_read", "FT_PATH_AUTO", "FT_PATH_GEMM", "FT_PATH_GEMV", "FT_PATH_GEMV_DP4A", "FtError",
    "block_dots", "last_error", "load", "moe_q4_0_q8_1", "moe_q4_0_q8_1_ep", "moe_q4_0_q8_1_slots", "profile_enable", "profile_read", "quantize_q8_1", "read_device_error", "release", "reserve",
    "route_offsets", "selected_path", "set_path", "workspace_bytes",
]
