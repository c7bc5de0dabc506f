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
 *   oracle_dequantize_gguf / _gguf_block_dot /     pinned: hand blocks per type, an
 *   oracle_moe_gguf_q8_1                           independent numpy decode + einsum,
 *                                                  Q4_0 equal to oracle_moe_q4_0_q8_1
 *                                                  bit for bit, the offset term within
 *                                                  the fp16 rounding of s; K-quants:
 *                                                  hand-packed super-blocks, a numpy
 *                                                  decoder, the plain dequantized dot,
 *                                                  unit-scale Q4_K = eight Q4_1 blocks;
 *                                                  Q2_K / Q3_K / Q6_K: hand-built
 *                                                  super-blocks, numpy decoders,
 *                                                  the plain dequantized dot
 *   oracle_repack_q4_0_soa                         pinned: numpy slicing of the
 *                                                  block bytes, hand block
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
 * Other GGUF weight types with 32-weight blocks (weight i = q_i d + c):
 *   Q4_1 20 B: fp16 d, fp16 m, 16 B qs (nibbles as Q4_0); q_i = nibble, c = m
 *   Q5_0 22 B: fp16 d, 4 B qh (little-endian), 16 B qs; q_i = nibble_i |
 *       (bit i of qh) << 4, minus 16; c = 0
 *   Q5_1 24 B: fp16 d, fp16 m, 4 B qh, 16 B qs; q_i = nibble_i | (bit i) << 4;
 *       c = m
 *   Q8_0 34 B: fp16 d, 32 int8 q; c = 0
 * K-quants, 256 weights per super-block, eight sub-blocks of 32 (weight l of
 * sub-block j = d * sc_j * q_l - dmin * m_j, 6-bit sc_j and m_j):
 *   Q4_K 144 B: fp16 d, fp16 dmin, 12 B scales/mins, 128 B nibbles
 *   Q5_K 176 B: fp16 d, fp16 dmin, 12 B scales/mins, 32 B qh, 128 B nibbles
 *   Q6_K 210 B: 128 B low nibbles, 64 B 2-bit high parts, 16 int8 scales (one
 *       per 16 weights), fp16 d; level = 6-bit value - 32, weight = d scale q
 *   Q2_K  84 B: 16 scale bytes (scale | min << 4 per 16 weights), 64 B of
 *       2-bit codes, fp16 d, fp16 dmin; weight = d scale q - dmin min
 *   Q3_K 110 B: 32 B hmask (third bits), 64 B of 2-bit codes, 12 B of sixteen
 *       packed 6-bit scales, fp16 d; weight = d (scale - 32) q, q in [-4, 3]
 *   (oracle_dequantize_gguf counts super-blocks for these; ncols % 256 == 0)
 *   weights [E][N][K/32] blocks of the type.
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

/* GGUF weight types with 32-weight blocks (GGML type numbers). */
#define ORACLE_GGUF_Q4_0 2
#define ORACLE_GGUF_Q4_1 3
#define ORACLE_GGUF_Q5_0 6
#define ORACLE_GGUF_Q5_1 7
#define ORACLE_GGUF_Q8_0 8
#define ORACLE_GGUF_Q4_K 12
#define ORACLE_GGUF_Q5_K 13
#define ORACLE_GGUF_Q6_K 14
#define ORACLE_GGUF_Q2_K 10
#define ORACLE_GGUF_Q3_K 11
int32_t oracle_gguf_block_bytes(int32_t type);
void oracle_dequantize_gguf(int32_t type, const uint8_t* blocks, int64_t n_blocks, double* out);
int32_t oracle_gguf_block_dot(int32_t type, const uint8_t* w_block, const uint8_t* a_block);
void oracle_moe_gguf_q8_1(int32_t type, const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                          float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                          int64_t nrows, int64_t ncols);

void oracle_repack_q4_0_soa(const uint8_t* blocks, int64_t n_blocks, uint8_t* qs, uint16_t* d);

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
