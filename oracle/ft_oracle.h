/*
 * CPU oracle for the routed Q4_0 x Q8_1 MoE expert matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this code.  It shares no source, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Plain, slow, obviously correct C: loops in the order of the definitions,
 * fp64 accumulation, fp32 only where the activation quantizer's definition
 * fixes single precision.  Functions and their pins:
 *
 *   oracle_half_to_double / oracle_float_to_half   pinned to numpy float16
 *   oracle_quantize_q4_0                           pinned: nearest-level brute
 *                                                  force, hand blocks
 *   oracle_quantize_q8_1                           pinned: hand blocks, error
 *                                                  bound, numpy fp32 replay
 *   oracle_route                                   pinned: stable argsort
 *   oracle_block_dot / oracle_moe_*                pinned: hand blocks, fp64
 *                                                  dequant brute force, numpy
 *                                                  einsum of decoded operands,
 *                                                  split invariance
 *   oracle_moe_slots_q4_0_q8_1                     pinned: numpy einsum of decoded
 *                                                  operands; replicated token rows
 *                                                  give oracle_moe_q4_0_q8_1 bit for bit
 *   oracle_moe_ep_q4_0_q8_1                        pinned: the shards of a partition
 *                                                  of the experts sum to
 *                                                  oracle_moe_q4_0_q8_1 bit for bit;
 *                                                  hand-checked masking
 *   oracle_act_mul / _quantize_q8_1                pinned: 50-digit mpmath values, torch
 *                                                  activations, the exact
 *                                                  GELU x*Phi(x) within the tanh
 *                                                  form's error, f(x) - f(-x) = x,
 *                                                  gate/up order, hand values; the
 *                                                  quantizer replayed in numpy fp32
 *
 * Byte layouts (GGUF block formats; the pages serve GGUF Q4_0 checkpoints but
 * do not print the formats):
 *   Q4_0 block, 18 B: fp16 d, then 16 bytes qs; weight j (j < 16) is the low
 *       nibble of qs[j], weight j+16 its high nibble; value = (q - 8) * d.
 *   Q8_1 block, 36 B: fp16 d, fp16 s, then 32 int8 q; value = q * d,
 *       s = d * sum(q).
 *   weights [E][N][K/32] Q4_0, activations [T][K/32] Q8_1,
 *   topk_ids [T][k] int32 (slot s = t*k + j), out [T][k][N] fp32.
 *   gated activation: h [rows][2 * n_inter] fp32 (gate | up), a [rows][n_inter].
 */
#ifndef FT_ORACLE_H
#define FT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

double   oracle_half_to_double(uint16_t h);
uint16_t oracle_float_to_half(float f);

void oracle_quantize_q4_0(const float* w, int64_t n_blocks, uint8_t* out);
void oracle_dequantize_q4_0(const uint8_t* blocks, int64_t n_blocks, double* out);

void oracle_quantize_q8_1(const uint16_t* x_fp16, int64_t tokens, int64_t ncols, uint8_t* out);
void oracle_dequantize_q8_1(const uint8_t* blocks, int64_t n_blocks, double* out);

#define ORACLE_ACT_SILU 0
#define ORACLE_ACT_GELU_TANH 1
void oracle_act_mul(const float* h, int64_t rows, int64_t n_inter, int32_t kind, float* a);
void oracle_act_mul_quantize_q8_1(const float* h, int64_t rows, int64_t n_inter, int32_t kind, uint8_t* out);

int64_t oracle_route(const int32_t* topk_ids, int64_t n_slots, int32_t n_experts,
                     int32_t* counts, int32_t* offsets, int32_t* perm);

int32_t oracle_block_dot(const uint8_t* w_block, const uint8_t* a_block);

void oracle_moe_q4_0_q8_1(const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                          float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                          int64_t nrows, int64_t ncols);

void oracle_moe_slots_q4_0_q8_1(const uint8_t* weights, const uint8_t* act_slots, const int32_t* topk_ids,
                                float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                                int64_t nrows, int64_t ncols);

void oracle_moe_ep_q4_0_q8_1(const uint8_t* weights_local, const uint8_t* act, const int32_t* topk_ids,
                             float* out, int64_t tokens, int32_t top_k, int32_t n_global,
                             int32_t expert_start, int32_t n_local, int64_t nrows, int64_t ncols);

void oracle_moe_sample(const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                       int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                       int64_t ncols, const int64_t* slots, const int64_t* rows, int64_t n,
                       double* out);

void oracle_moe_block_dots(const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                           int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                           int64_t ncols, int32_t* dots);

void oracle_moe_dequant_bruteforce(const uint8_t* weights, const uint8_t* act,
                                   const int32_t* topk_ids, int64_t tokens, int32_t top_k,
                                   int32_t n_experts, int64_t nrows, int64_t ncols, double* out);

#ifdef __cplusplus
}
#endif
#endif
