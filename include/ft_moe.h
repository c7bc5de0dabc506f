/*
 * ft_moe.h - C ABI of the GB300 (sm_103a) routed Q4_0 x Q8_1 MoE expert matmul.
 *
 * What it computes.  For every flat (token, top-k) slot s = t * top_k + j of a
 * batch, with expert e = topk_ids[s], and every weight row r of that expert:
 *
 *     out[s][r] = sum_b  d_w[e][r][b] * d_a[t][b] * sum_{i<32} (q_w[e][r][b][i] - 8) * q_a[t][b][i]
 *
 * the dot product of the routed expert's Q4_0 weight rows with the token's
 * Q8_1 activation (moe_vec_q4_0_q8_1 over the flat (token, top-k) index:
 * FreeToken PR #185, "launch GGUF MoE GEMV token axis on grid.x, not grid.z",
 * sections "Problem" and "Fix"), in both the per-slot GEMV form and the
 * expert-grouped GEMM form keyed by expert_offsets with a leading 0
 * (nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 4).  The per-block integer dots
 * are exact; the scale products are accumulated in fp32.
 *
 * Formats (GGUF blocks of 32 values, little-endian):
 *   Q4_0, 18 bytes: fp16 d, then 16 bytes qs; value j < 16 is the low nibble
 *         of qs[j], value j + 16 its high nibble; weight = (q - 8) * d.
 *   Q8_1, 36 bytes: fp16 d, fp16 s, then 32 int8 q; activation = q * d and
 *         s = d * sum(q) (stored for format fidelity; the dot does not use it).
 *
 * Layouts (all row-major, contiguous):
 *   weights  [n_experts][nrows][ncols/32] Q4_0 blocks (18 B each)
 *   act      [tokens][ncols/32] Q8_1 blocks (36 B each)
 *   topk_ids [tokens][top_k] int32
 *   out      [tokens][top_k][nrows] fp32
 *
 * Conventions shared by every entry point.
 *   - Pointers are DEVICE pointers on the current CUDA device unless stated.
 *     The caller owns every buffer it passes; the library owns only its
 *     workspace (see ft_moe_reserve).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All work is stream-ordered; no entry point below synchronizes
 *     except ft_moe_read_device_error and ft_moe_release.
 *   - Every size product is computed in 64-bit; no launch places the slot or
 *     token count on grid.y or grid.z, so tokens * top_k is not capped at
 *     65535 (FreeToken PR #185, "Problem"; mlxcel PR #652, "Summary").
 *   - Argument errors are reported before anything is launched.  After every
 *     kernel launch the library checks the launch status and, on failure,
 *     returns FT_ERR_LAUNCH with the kernel name and grid in ft_last_error()
 *     (FreeToken PR #185: FT_MOE_VEC_LAUNCH_CHECK, "Fix").
 *   - Expert ids outside [0, n_experts) never fault: the slot is left out of
 *     the routing, its output row is zeroed and FT_DEVERR_BAD_EXPERT_ID is
 *     raised in the device error word.
 *   - Route + matmul issue a fixed number of launches, allocate nothing once
 *     the workspace is reserved and read nothing back to the host, so they can
 *     be captured in a CUDA graph (nvfp4-megamoe-kernel CURRENT_BUG.md,
 *     "Cudagraph Constraints").
 */
#ifndef FT_MOE_H
#define FT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FT_MOE_ABI_VERSION 1

#if defined(__GNUC__)
#define FT_API __attribute__((visibility("default")))
#else
#define FT_API
#endif

typedef enum {
    FT_OK = 0,
    FT_ERR_ARG = 1,          /* null pointer, bad count, bad top_k, ncols % 32 != 0 ...   */
    FT_ERR_SIZE = 2,         /* a size product overflows, or exceeds a documented limit */
    FT_ERR_ALIGN = 3,        /* a pointer misses its required alignment                 */
    FT_ERR_LAUNCH = 4,       /* a kernel launch was rejected; see ft_last_error()       */
    FT_ERR_WORKSPACE = 5,    /* workspace too small while the stream is being captured  */
    FT_ERR_CUDA = 6,         /* a CUDA runtime call failed; see ft_last_error()         */
    FT_ERR_DEVICE_FLAG = 7   /* ft_moe_read_device_error found a raised device flag     */
} ft_status;

/* Bits of the device error word. */
#define FT_DEVERR_BAD_EXPERT_ID 0x1u   /* a topk id was outside [0, n_experts)           */
#define FT_DEVERR_WAIT_TIMEOUT  0x2u   /* a bounded in-kernel wait gave up (never expected) */
#define FT_DEVERR_WORKSPACE_GUARD 0x4u /* a guard block between workspace regions was overwritten */

/* Path selection for ft_moe_q4_0_q8_1 (ft_moe_set_path). */
#define FT_PATH_AUTO 0   /* chosen on the host from tokens*top_k, n_experts and the shape */
#define FT_PATH_GEMV 1   /* per-slot GEMV on CUDA cores                                  */
#define FT_PATH_GEMM 2   /* expert-grouped GEMM on the tcgen05 tensor cores              */
#define FT_PATH_GEMV_DP4A 3 /* the GEMV path, every slot tile on the dp4a CUDA-core kernels
                               (no mma.sync tiles; for comparison and tests)                */

/* Weight block types of ft_moe_gguf_q8_1: the GGUF types whose blocks hold
 * 32 weights (GGML type numbers).  Weight i of a block = q_i * d + c:
 *   Q4_0 18 B: fp16 d, 16 B nibbles (weight j<16: low nibble of byte j, j+16:
 *        its high nibble); q_i = nibble - 8, c = 0
 *   Q4_1 20 B: fp16 d, fp16 m, 16 B nibbles as Q4_0; q_i = nibble, c = m
 *   Q5_0 22 B: fp16 d, 4 B qh (little-endian uint32), 16 B nibbles;
 *        q_i = (nibble_i | (bit i of qh) << 4) - 16, c = 0
 *   Q5_1 24 B: fp16 d, fp16 m, 4 B qh, 16 B nibbles; q_i = nibble_i |
 *        (bit i of qh) << 4, c = m
 *   Q8_0 34 B: fp16 d, 32 int8 q_i, c = 0 */
#define FT_TYPE_Q4_0 2
#define FT_TYPE_Q4_1 3
#define FT_TYPE_Q5_0 6
#define FT_TYPE_Q5_1 7
#define FT_TYPE_Q8_0 8
/* K-quants: 256 weights per super-block, eight sub-blocks of 32; weight l of
 * sub-block j = d * sc_j * q_l - dmin * m_j with 6-bit sc_j, m_j packed in 12
 * bytes (j < 4: low 6 bits of bytes j and j + 4; j >= 4: low / high nibble of
 * byte j + 4 with the top two bits of byte j - 4 / j above it).  Sub-block j
 * takes nibble byte 32 * (j / 2) + l, low nibble for even j, high for odd j.
 *   Q4_K 144 B: fp16 d, fp16 dmin, 12 B scales/mins, 128 B nibbles
 *   Q5_K 176 B: fp16 d, fp16 dmin, 12 B scales/mins, 32 B qh (bit j of qh[l]
 *        is the 5th bit of weight l of sub-block j), 128 B nibbles */
#define FT_TYPE_Q4_K 12
#define FT_TYPE_Q5_K 13
/*   Q6_K 210 B: 128 B low nibbles, 64 B 2-bit high parts, 16 int8 scales (one
 *        per 16 weights), fp16 d last.  Sub-block j = 4 h + k takes nibble byte
 *        64 h + 32 (k % 2) + l (high nibble for k >= 2) and bits 2k, 2k + 1 of
 *        byte 128 + 32 h + l; level = that 6-bit value - 32; weight l uses
 *        scale 8 h + 2 k (l < 16) or 8 h + 2 k + 1: weight = d * scale * level */
#define FT_TYPE_Q6_K 14
/*   Q2_K  84 B: 16 scale bytes (scale | min << 4, one per 16 weights), 64 B of
 *        2-bit codes, fp16 d, fp16 dmin; weight = d scale q - dmin min
 *   Q3_K 110 B: 32 B hmask, 64 B of 2-bit codes, 12 B of sixteen packed 6-bit
 *        scales, fp16 d; bit j of hmask[l] is the third bit of weight l of
 *        sub-block j, q = (code | third bit << 2) - 4, weight = d (scale - 32) q.
 *        Scale g: low four bits from byte g % 8 (low nibble for g < 8, high for
 *        g >= 8), top two from bits 2 (g / 4) of byte 8 + g % 4.
 *   In both, sub-block j = 4 h + k takes bits 2k of code byte 32 h + l and
 *   scale groups 2j (weights < 16) and 2j + 1. */
#define FT_TYPE_Q2_K 10
#define FT_TYPE_Q3_K 11

/* Gated activations of ft_act_mul_quantize_q8_1 / ft_moe_ffn_q4_0_q8_1. */
#define FT_ACT_SILU 0        /* silu(g) = g / (1 + exp(-g))                              */
#define FT_ACT_GELU_TANH 1   /* g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))            */

/* Documented limits. */
#define FT_MAX_EXPERTS 4096
#define FT_MAX_NCOLS   65536

/*
 * ft_quantize_q8_1 - fp16 activations -> Q8_1 blocks (quantize_row_q8_1 on
 * FreeToken PR #185, "Fix").  Per 32-block of a row, in IEEE fp32 with
 * round-to-nearest: amax = max |x|, d = amax / 127, q = round-half-away(x / d)
 * (0 when amax == 0), s = d * sum(q); d and s stored as fp16 (round to
 * nearest even).  The result is bit-identical to the CPU oracle.
 *
 *   x_fp16    device, [tokens][ncols] fp16, 4-byte aligned
 *   act_q8_1  device, [tokens][ncols/32] Q8_1 (36 B each), 4-byte aligned
 *   tokens    >= 0 (0 is a no-op); ncols > 0, ncols % 32 == 0
 * Errors: FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_ALIGN, FT_ERR_LAUNCH.
 */
FT_API int ft_quantize_q8_1(const void* x_fp16, void* act_q8_1, int64_t tokens, int64_t ncols,
                     void* stream);

/*
 * ft_moe_route_offsets - stable counting sort of the tokens*top_k slots by
 * expert id (the expert_offsets of nvfp4-megamoe-kernel CURRENT_BUG.md,
 * Bug 4, with the searchsorted(right=True) slot-to-expert map of Bug 2).
 *
 *   topk_ids  device, [tokens][top_k] int32
 *   counts    device, [n_experts] int32 out: slots routed to each expert
 *   offsets   device, [n_experts + 1] int32 out: offsets[0] = 0,
 *             offsets[e+1] = offsets[e] + counts[e]; offsets[n_experts] is the
 *             number of slots with a valid id
 *   perm      device, [tokens*top_k] int32 out: perm[offsets[e] + r] is the
 *             r-th slot (ascending slot order) routed to e; entries at and past
 *             offsets[n_experts] are -1.  Unique, hence bit-comparable.
 *   dev_err   device uint32 or NULL; bad ids OR FT_DEVERR_BAD_EXPERT_ID into
 *             it (NULL: the library's own word, read by ft_moe_read_device_error)
 * Needs 1 <= top_k <= n_experts <= FT_MAX_EXPERTS and tokens*top_k < 2^31.
 * Uses the library workspace (reserved or grown on demand outside capture).
 * Errors: FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_WORKSPACE, FT_ERR_CUDA, FT_ERR_LAUNCH.
 */
FT_API int ft_moe_route_offsets(const int32_t* topk_ids, int64_t tokens, int32_t top_k,
                         int32_t n_experts, int32_t* counts, int32_t* offsets, int32_t* perm,
                         uint32_t* dev_err, void* stream);

/*
 * ft_moe_route_offsets_noalloc - the same routing as ft_moe_route_offsets,
 * for callers that are not allowed to allocate device memory: a runtime
 * whose memory planner owns every byte of the GPU after start-up, a plugin
 * running inside another framework's allocator, or a latency-critical loop
 * that cannot afford cudaMalloc's implicit device synchronization.  This
 * entry point has no counterpart on the pages; it exists only for them.
 *
 * Nothing is allocated, by this call or any earlier one: the per-chunk
 * histogram scratch lives in one fixed array of FT_ROUTE_NOALLOC_SCRATCH_WORDS
 * int32 (1 MiB) compiled into the library, which every GPU that loads the
 * library holds until the process exits.  The scratch needs
 * ceil(tokens*top_k / 256) * n_experts words; larger problems are rejected
 * with FT_ERR_SIZE before anything runs (use ft_moe_route_offsets for them).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for the life
 * of the process; make that first call before any stream capture.  A
 * cudaDeviceReset (or any teardown of the device's primary context) makes the
 * kept address stale, so after one this entry point must not be used again in
 * the same process.  All calls share the one array and nothing in it
 * needs to start at zero (every histogram entry is written before it is
 * read), so calls that overlap on the GPU - on different streams, or from
 * different host threads - race with each other and must be serialized by
 * the caller.  Arguments, outputs and the other errors are those of
 * ft_moe_route_offsets; with dev_err == NULL bad-id flags are dropped.
 */
#define FT_ROUTE_NOALLOC_SCRATCH_WORDS (1 << 18)
FT_API int ft_moe_route_offsets_noalloc(const int32_t* topk_ids, int64_t tokens, int32_t top_k,
                                        int32_t n_experts, int32_t* counts, int32_t* offsets,
                                        int32_t* perm, uint32_t* dev_err, void* stream);

/*
 * ft_moe_q4_0_q8_1 - the routed expert matmul defined at the top of this file.
 * Routes internally (into the workspace), then runs the GEMV or the grouped
 * GEMM path (FT_PATH_AUTO decides on the host, without reading the device:
 * the GEMM from 40 routed slots per expert on average where the GEMV runs
 * its 16-slot mma.sync tiles, else from 16).
 *
 *   weights   device, Q4_0 [n_experts][nrows][ncols/32]; 16-byte aligned
 *   act       device, Q8_1 [tokens][ncols/32] (from ft_quantize_q8_1); 16-byte aligned
 *   topk_ids  device, int32 [tokens][top_k]
 *   out       device, fp32 [tokens][top_k][nrows]; every element is written
 *             (rows of slots with a bad expert id are written as 0)
 * Needs ncols % 32 == 0, 0 < ncols <= FT_MAX_NCOLS, nrows > 0,
 * 1 <= top_k <= n_experts <= FT_MAX_EXPERTS, tokens*top_k < 2^31.
 * The tensor-core path additionally needs ncols % 256 == 0; other shapes take
 * the GEMV path (a forced FT_PATH_GEMM on such a shape returns FT_ERR_ARG).
 * Errors: FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_ALIGN, FT_ERR_WORKSPACE, FT_ERR_CUDA,
 * FT_ERR_LAUNCH.
 */
FT_API int ft_moe_q4_0_q8_1(const void* weights, const void* act, const int32_t* topk_ids, float* out,
                     int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                     int64_t ncols, void* stream);

/*
 * ft_moe_q4_0_fp16 - the whole hot path from fp16 activations: exactly
 *   ft_moe_q4_0_q8_1(weights, ft_quantize_q8_1(x_fp16), topk_ids, out)
 * (quantize_row_q8_1 then moe_vec_q4_0_q8_1 over the flat slots, FreeToken
 * PR #185, "Fix" and "Problem").  A decode-sized batch on the GEMV path (at
 * most 512 slots, 1024 experts, ncols % 256 == 0, x_fp16 16-byte aligned,
 * and at most 256 activation blocks per CTA's slot group) runs as one
 * kernel launch in which every CTA routes the slots and quantizes the
 * activation rows it needs itself (the stable slot order and
 * the quantizer's arithmetic, so the out bits are those of the two calls);
 * any other batch quantizes into library workspace (counted by
 * ft_moe_workspace_bytes and ft_moe_reserve) and takes the usual path.
 *
 *   x_fp16    device, fp16 [tokens][ncols], 8-byte aligned
 *   weights, topk_ids, out, tokens, top_k, n_experts, nrows, ncols as for
 *   ft_moe_q4_0_q8_1.
 * Bad expert ids: zero output rows and the device error flag, as there.
 * Errors: those of ft_quantize_q8_1 and ft_moe_q4_0_q8_1.
 */
FT_API int ft_moe_q4_0_fp16(const void* weights, const void* x_fp16, const int32_t* topk_ids, float* out,
                            int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols,
                            void* stream);

/*
 * ft_moe_q4_0_q8_1_slots - the same matmul with one activation row per routed
 * slot instead of one per token: the input of the second expert layer, which
 * runs on the first layer's output after SiLU*up, one row per routed slot
 * (nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6).
 *   out[s][r] = sum_b d_w[e][r][b] * d_a[s][b] * sum_i (q_w - 8) * q_a[s][b][i],
 *   e = topk_ids[s], s = t * top_k + j.
 *
 *   act_slots device, Q8_1 [tokens*top_k][ncols/32]; row s belongs to slot s;
 *             16-byte aligned
 * Every other argument, the layouts, the path choice, the workspace and the
 * errors are those of ft_moe_q4_0_q8_1.
 */
FT_API int ft_moe_q4_0_q8_1_slots(const void* weights, const void* act_slots, const int32_t* topk_ids,
                                  float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                                  int64_t nrows, int64_t ncols, void* stream);

/*
 * ft_moe_q4_0_q8_1_ep - the matmul on one expert-parallel shard: topk_ids
 * hold global expert ids, the shard holds experts [expert_start,
 * expert_start + n_experts_local) of n_experts_global, a slot routed to one
 * of them is computed with local expert id - expert_start, and every other
 * slot's output row is written as 0 (nvfp4-megamoe-kernel CURRENT_BUG.md,
 * Bug 8: global ids remapped by experts_start_idx, non-local tokens masked),
 * so the outputs of shards that partition the experts add up to the full
 * result.  Only ids outside [0, n_experts_global) raise
 * FT_DEVERR_BAD_EXPERT_ID.
 *
 *   weights_local  device, Q4_0 [n_experts_local][nrows][ncols/32]; 16-byte aligned
 *   act, topk_ids, out, tokens, top_k, nrows, ncols as for ft_moe_q4_0_q8_1
 * Needs 1 <= top_k <= n_experts_global <= FT_MAX_EXPERTS, n_experts_local >= 1,
 * 0 <= expert_start and expert_start + n_experts_local <= n_experts_global.
 * Errors as for ft_moe_q4_0_q8_1.  The path choice and the tile plans assume
 * the slots spread evenly over the global experts.
 */
FT_API int ft_moe_q4_0_q8_1_ep(const void* weights_local, const void* act, const int32_t* topk_ids,
                               float* out, int64_t tokens, int32_t top_k, int32_t n_experts_global,
                               int32_t expert_start, int32_t n_experts_local, int64_t nrows,
                               int64_t ncols, void* stream);

/*
 * ft_moe_gguf_q8_1 - the routed matmul with expert weights of a GGUF type
 * (FT_TYPE_*; the per-type launchers of moe_vec.cuh on FreeToken PR #185,
 * "Notes"):
 *   out[s][r] = sum_b d_w d_a sum_i q_i q_a[i] + c d_a sum_i q_a[i]
 * per 32-weight block b of row r of expert topk_ids[s] and activation block b
 * of the slot's token, with q_i, c as in the FT_TYPE_* list (c = 0 for Q4_0,
 * Q5_0, Q8_0) and the exact sum of the activation codes (the dequantized
 * activation is d_a q_a; the stored fp16 s, that sum rounded, is not used); for the
 * K-quants, per sub-block b, d sc_b d_a sum_i q_i q_a[i] - dmin m_b d_a sum_i q_a[i]
 * (Q6_K, Q3_K: d d_a (sc_lo sum_{i<16} q_i q_a[i] + sc_hi sum_{i>=16} q_i q_a[i]);
 * Q2_K adds - dmin d_a (min_lo sum_{i<16} q_a[i] + min_hi sum_{i>=16} q_a[i])).
 *
 *   wtype     FT_TYPE_Q4_0 (exactly ft_moe_q4_0_q8_1), FT_TYPE_Q4_1,
 *             FT_TYPE_Q5_0, FT_TYPE_Q5_1, FT_TYPE_Q8_0, FT_TYPE_Q2_K,
 *             FT_TYPE_Q3_K, FT_TYPE_Q4_K, FT_TYPE_Q5_K or FT_TYPE_Q6_K (the
 *             K-quants need ncols % 256 == 0)
 *   weights   device, [n_experts][nrows][ncols/32] blocks of wtype
 *             ([ncols/256] super-blocks for the K-quants); 16-byte aligned
 *   act, topk_ids, out, tokens, top_k, n_experts, nrows, ncols as for
 *   ft_moe_q4_0_q8_1.
 * Q4_0 and Q4_K take either path by the rule of ft_moe_q4_0_q8_1 (Q4_K on the
 * tensor cores: one 144-byte super-block per row and stage, its sub-block
 * scales and mins applied in the drain); the other types always take the
 * GEMV path, and ft_moe_set_path(FT_PATH_GEMM) makes them fail with
 * FT_ERR_ARG.  On the GEMV path, batches with more than 4 slots per expert of
 * Q4_0, Q4_1, Q8_0 and Q4_K run tiles of 8 or 16 slots on mma.sync (exact
 * integer block dots; each block's or sub-block's scale and offset applied
 * after its two MMAs, as the dp4a kernels do).
 * ft_moe_gguf_selected_path tells which path a shape takes.
 * Errors as for ft_moe_q4_0_q8_1, plus FT_ERR_ARG for an unknown wtype.
 */
FT_API int ft_moe_gguf_q8_1(int32_t wtype, const void* weights, const void* act, const int32_t* topk_ids,
                            float* out, int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                            int64_t ncols, void* stream);

/*
 * ft_repack_q4_0_soa - one-time export of Q4_0 weights as a structure of
 * arrays (the SoA weight repack export next to the per-type launchers of
 * moe_vec.cuh, FreeToken PR #185, "Notes"): for block b of the stored array
 *   qs[16 b .. 16 b + 15] = its 16 nibble bytes (block bytes 2..17)
 *   d[b]                  = its fp16 scale (block bytes 0..1)
 * Bytes move unchanged.  The matmul entry points read the stored layout; this
 * is for consumers that want nibbles and scales apart.
 *
 *   weights   device, n_blocks Q4_0 blocks (e.g. [E][N][K/32]), 2-byte aligned
 *   qs        device, uint8 [n_blocks][16] out, 16-byte aligned
 *   d         device, fp16 [n_blocks] out, 2-byte aligned
 *   n_blocks  >= 0 (0 is a no-op)
 * Errors: FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_ALIGN, FT_ERR_LAUNCH.
 */
FT_API int ft_repack_q4_0_soa(const void* weights, void* qs, void* d, int64_t n_blocks, void* stream);

/*
 * ft_act_mul_quantize_q8_1 - the step between the two expert layers, fused:
 * the gated activation of the gate half of each row times its up half,
 * requantized to Q8_1 (gelu_tanh_and_mul right after the routed matmul on
 * FreeToken PR #185, "Problem"; SiLU*up between layer 1 and layer 2 on
 * nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6).  Per row r and column i < I:
 *   a[r][i] = act(h[r][i]) * h[r][I + i]      (fp32, never stored)
 * then each 32-block of a row is quantized as ft_quantize_q8_1 does.
 * The activation is computed in fp32 to within a few ulps of the exact value
 * (the CPU oracle takes it in fp64 and rounds once), so a Q8_1 code may differ
 * by 1 from the oracle's where a / d lies that close to a rounding boundary.
 *
 *   h         device, fp32 [rows][2 * n_inter] (gate | up), 16-byte aligned
 *   act_q8_1  device, Q8_1 [rows][n_inter / 32], 4-byte aligned
 *   rows      >= 0 (0 is a no-op); n_inter > 0, n_inter % 32 == 0
 *   act_kind  FT_ACT_SILU or FT_ACT_GELU_TANH
 * Errors: FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_ALIGN, FT_ERR_LAUNCH.
 */
FT_API int ft_act_mul_quantize_q8_1(const float* h, void* act_q8_1, int64_t rows, int64_t n_inter,
                                    int32_t act_kind, void* stream);

/*
 * ft_moe_q4_0_q8_1_act - layer 1 of the routed MoE block with the gated
 * activation and the Q8_1 requantization fused into it (gelu_tanh_and_mul
 * right after the routed matmul on FreeToken PR #185, "Problem"; SiLU*up
 * between layer 1 and layer 2 on nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6):
 *   act_mid = ft_act_mul_quantize_q8_1(ft_moe_q4_0_q8_1(w13, act))
 * without the fp32 layer-1 result in memory on the tensor-core path: each
 * tile there holds 64 gate rows and the 64 matching up rows of one expert,
 * and its epilogue writes the Q8_1 blocks of act(gate) * up for its slots.
 * On the GEMV path the layer-1 result goes to library workspace
 * (tokens * top_k * 2 n_inter fp32) and the activation step reads it there.
 * The per-element arithmetic is that of the two calls it replaces, so the
 * result equals theirs bit for bit on the same path.
 *
 *   w13       device, Q4_0 [n_experts][2 * n_inter][hidden / 32]: rows
 *             [0, n_inter) of an expert are its gate rows, [n_inter, 2 n_inter)
 *             its up rows; 16-byte aligned
 *   act       device, Q8_1 [tokens][hidden / 32]; 16-byte aligned
 *   topk_ids  device, int32 [tokens][top_k]
 *   act_mid   device, Q8_1 [tokens * top_k][n_inter / 32] out; 4-byte aligned
 *   n_inter   positive multiple of 32; the limits of ft_moe_q4_0_q8_1 apply
 *             to the matmul with nrows = 2 n_inter, ncols = hidden
 *   act_kind  FT_ACT_SILU or FT_ACT_GELU_TANH
 * Slots with a bad expert id get zero act_mid rows (and the device error
 * flag).  Errors: those of ft_moe_q4_0_q8_1 and ft_act_mul_quantize_q8_1.
 */
FT_API int ft_moe_q4_0_q8_1_act(const void* w13, const void* act, const int32_t* topk_ids, void* act_mid,
                                int64_t tokens, int32_t top_k, int32_t n_experts, int64_t n_inter, int64_t hidden,
                                int32_t act_kind, void* stream);

/*
 * ft_moe_ffn_q4_0_q8_1 - both expert layers of the routed MoE block, per
 * slot, on `stream` (layer 1 -> activation -> layer 2 on
 * nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6).  With h != NULL, three steps:
 *   h       = ft_moe_q4_0_q8_1(w13, act)           gate and up rows in one matmul
 *   act_mid = ft_act_mul_quantize_q8_1(h)          per slot row
 *   out     = ft_moe_q4_0_q8_1_slots(w2, act_mid)
 * with h == NULL, two: act_mid = ft_moe_q4_0_q8_1_act(w13, act), then the
 * same layer 2 (act_mid and out equal those of the three steps bit for bit).
 * The weighted sum over a token's top_k slots is left to the caller.
 *
 *   w13       device, Q4_0 [n_experts][2 * n_inter][hidden / 32]: rows
 *             [0, n_inter) of an expert are its gate rows, [n_inter, 2 n_inter)
 *             its up rows; 16-byte aligned
 *   w2        device, Q4_0 [n_experts][hidden][n_inter / 32]; 16-byte aligned
 *   act       device, Q8_1 [tokens][hidden / 32]; 16-byte aligned
 *   topk_ids  device, int32 [tokens][top_k]
 *   h         device, fp32 [tokens][top_k][2 * n_inter] out (scratch the
 *             caller owns; holds the layer-1 result afterwards); 16-byte
 *             aligned; or NULL: layer 1 with the activation fused
 *   act_mid   device, Q8_1 [tokens * top_k][n_inter / 32] out (scratch the
 *             caller owns; holds the layer-2 input afterwards); 16-byte aligned
 *   out       device, fp32 [tokens][top_k][hidden] out
 * Needs hidden and n_inter positive multiples of 32 and the limits of
 * ft_moe_q4_0_q8_1 for both matmuls.  Slots with a bad expert id get zero h,
 * act_mid and out rows.  Errors: those of the three steps.
 */
FT_API int ft_moe_ffn_q4_0_q8_1(const void* w13, const void* w2, const void* act, const int32_t* topk_ids,
                                float* h, void* act_mid, float* out, int64_t tokens, int32_t top_k,
                                int32_t n_experts, int64_t hidden, int64_t n_inter, int32_t act_kind,
                                void* stream);

/*
 * ft_moe_ffn_reserve - ft_moe_reserve for both expert layers: allocates the
 * current device's workspace for ft_moe_ffn_q4_0_q8_1 (h given or NULL) and
 * ft_moe_q4_0_q8_1_act at up to these sizes, so that they can be captured
 * in a CUDA graph.  Errors: FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_CUDA.
 */
FT_API int ft_moe_ffn_reserve(int64_t max_tokens, int32_t max_top_k, int32_t n_experts, int64_t hidden,
                              int64_t n_inter);

/*
 * ft_moe_workspace_bytes - bytes of library workspace that one
 * ft_moe_q4_0_q8_1 / ft_moe_route_offsets call of this shape needs.
 * Returns 0 for invalid arguments.
 */
FT_API size_t ft_moe_workspace_bytes(int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                              int64_t ncols);

/*
 * ft_moe_reserve - allocate (cudaMalloc) the workspace of the current device
 * for shapes up to these maxima.  Call it before capturing a stream; inside a
 * capture the library never allocates and returns FT_ERR_WORKSPACE instead.
 * Outside capture a call that needs more grows the workspace by itself
 * (cudaFree + cudaMalloc, which synchronize the device).
 * Errors: FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_CUDA.
 */
FT_API int ft_moe_reserve(int64_t max_tokens, int32_t max_top_k, int32_t n_experts, int64_t nrows,
                   int64_t ncols);

/* ft_moe_release - free the current device's workspace (synchronizes). */
FT_API int ft_moe_release(void);

/*
 * ft_moe_read_device_error - synchronize `stream`, read the library's device
 * error word of the current device into *flags_out and clear it.  It also
 * checks the 256-byte guard blocks that separate the workspace regions (they
 * are filled with a fixed pattern when the workspace is allocated): a
 * changed guard adds FT_DEVERR_WORKSPACE_GUARD and is refilled.  Returns
 * FT_OK when no flag was raised, FT_ERR_DEVICE_FLAG otherwise.  Not for use
 * inside a stream capture.
 */
FT_API int ft_moe_read_device_error(void* stream, uint32_t* flags_out);

/*
 * ft_debug_wait_timeout - test hook for the failure path of the bounded
 * in-kernel waits.  Launches one small kernel on `stream` that allocates TMEM,
 * waits on an mbarrier that nothing ever arrives on (the same bounded wait the
 * matmul kernels use, here with a limit of limit_ns nanoseconds), raises
 * FT_DEVERR_WAIT_TIMEOUT in the library's device error word when the wait
 * gives up, frees its TMEM and returns.  The context stays usable: read the
 * flag with ft_moe_read_device_error, then keep calling the library.
 *   limit_ns  in [1000, 1000000000]
 * Uses the library workspace (its error word).  The pages have no counterpart.
 * Errors: FT_ERR_ARG, FT_ERR_WORKSPACE, FT_ERR_CUDA, FT_ERR_LAUNCH.
 */
FT_API int ft_debug_wait_timeout(int64_t limit_ns, void* stream);

/*
 * ft_debug_stream_read - measurement hook: a plain streaming read of `bytes`
 * bytes of `buf` on `stream` (four independent 16-byte loads in flight per
 * thread, four 512-thread CTAs per SM, nothing written), so that a caller can
 * time how long the memory system takes to deliver a buffer of that size at
 * all; a bandwidth-bound kernel reading the same number of bytes is judged
 * against that time as well as against the copy peak of large buffers.
 *   buf    device, 16-byte aligned; bytes a multiple of 16 (0 is a no-op)
 * Uses the library workspace.  The pages have no counterpart.
 * Errors: FT_ERR_ARG, FT_ERR_ALIGN, FT_ERR_WORKSPACE, FT_ERR_CUDA, FT_ERR_LAUNCH.
 */
FT_API int ft_debug_stream_read(const void* buf, int64_t bytes, void* stream);

/*
 * ft_moe_set_path - force the path of later ft_moe_q4_0_q8_1 calls in this
 * process (FT_PATH_AUTO / FT_PATH_GEMV / FT_PATH_GEMM / FT_PATH_GEMV_DP4A);
 * returns the previous setting, or -1 for an unknown value.  The environment
 * variable FT_MOE_PATH (auto|gemv|gemm|gemv_dp4a) sets the initial value.
 */
FT_API int ft_moe_set_path(int32_t path);

/* ft_moe_selected_path - the path ft_moe_q4_0_q8_1 would take for this shape
 * under the current setting (FT_PATH_GEMV or FT_PATH_GEMM), or -1. */
FT_API int ft_moe_selected_path(int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                         int64_t ncols);

/* ft_moe_gguf_selected_path - the same for ft_moe_gguf_q8_1 with weights of
 * FT_TYPE_* wtype (-1 also for an unknown type or ncols not a whole number
 * of its blocks). */
FT_API int ft_moe_gguf_selected_path(int32_t wtype, int64_t tokens, int32_t top_k, int32_t n_experts,
                                     int64_t nrows, int64_t ncols);

/*
 * ft_moe_block_dots - diagnostic: run the selected path in a mode that writes
 * every per-block integer dot instead of the scaled sum:
 *   dots  device, int32 [tokens*top_k][nrows][ncols/32]
 *         dots[s][r][b] = sum_i (q_w[e][r][b][i] - 8) * q_a[t][b][i]
 *         (0 for slots with a bad id).
 * Same arguments and errors as ft_moe_q4_0_q8_1, plus FT_ERR_SIZE when the
 * dots array would exceed 2^31 elements.  For tests on small shapes.
 */
FT_API int ft_moe_block_dots(const void* weights, const void* act, const int32_t* topk_ids,
                      int32_t* dots, int64_t tokens, int32_t top_k, int32_t n_experts,
                      int64_t nrows, int64_t ncols, void* stream);

/*
 * Profiling.  ft_profile_enable(max_calls) starts recording, on the stream
 * each call launches on, CUDA events around the quantizer kernel and, in each
 * later matmul call, around its preparation (routing, plus on the tensor-core
 * path the gather of the routed activations into the MMA operand layout) and
 * around its matmul kernel (up to max_calls calls; 0 stops recording).  It
 * allocates the events, so call it outside stream capture.  ft_profile_read
 * synchronizes on the recorded events and returns the summed times
 * (milliseconds) as quantize_ms, route_ms (the preparation) and matmul_ms
 * (the matmul kernel alone), the number of calls recorded and the number of
 * kernels this library launched since recording started, then resets the
 * totals.  Per-process state, meant for benchmarks.
 */
FT_API int ft_profile_enable(int32_t max_calls);
FT_API int ft_profile_read(double* quantize_ms, double* route_ms, double* matmul_ms, int64_t* n_calls,
                           int64_t* n_launches);

/* ft_last_error - message of the last failing call on this host thread
 * (empty string if none).  The pointer stays valid until the next call on the
 * same thread. */
FT_API const char* ft_last_error(void);

/* ft_abi_version - FT_MOE_ABI_VERSION of the loaded library. */
FT_API int ft_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FT_MOE_H */
