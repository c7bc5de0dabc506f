// Host-side internals shared by the translation units of libft_moe.so.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ft {

// Status plus a message recorded for ft_last_error().
int fail(int status, const char* fmt, ...);

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Sets the dynamic shared-memory limit of a kernel once per device and size.
int set_smem_limit(const void* kernel, int bytes);

// Profiling hooks (no-ops unless ft_profile_enable is active).
enum ProfPoint { kProfQuantBegin, kProfQuantEnd, kProfRouteBegin, kProfMatmulBegin, kProfMatmulEnd };
void prof_mark(ProfPoint p, cudaStream_t s);
void prof_count_launch();

// Checks cudaGetLastError() after a launch; on failure records the kernel
// name and geometry and returns FT_ERR_LAUNCH.
int check_launch(const char* kernel, dim3 grid, dim3 block, size_t smem);

// Test hook: a kernel whose bounded wait must give up after limit_ns.
int launch_wait_timeout_probe(uint32_t* err, int64_t limit_ns, cudaStream_t s);
// Measurement hook: a plain streaming read of n16 16-byte words of buf.
int launch_stream_read(const void* buf, int64_t n16, uint32_t* sink, cudaStream_t s);

// ------------------------------------------------------------ quantizer
int launch_quantize_q8_1(const void* x, void* act, int64_t tokens, int64_t ncols, cudaStream_t s);
int launch_act_mul_quantize_q8_1(const float* h, void* act, int64_t rows, int64_t n_inter, int kind, cudaStream_t s);
int launch_repack_q4_0_soa(const void* blocks, void* qs, void* d, int64_t n_blocks, cudaStream_t s);

// ---------------------------------------------------------------- router
constexpr int kRouteChunk = 256;          // slots per warp-chunk
constexpr int kRouteWarps = 8;            // warp-chunks per CTA

struct RouteBuffers {
    int32_t* counts;       // [E]
    int32_t* offsets;      // [E+1]
    int32_t* perm;         // [S]
    int32_t* hist;         // [nchunks][E] scratch
    int32_t* tiles_gemv;   // [E+1] or nullptr
    int32_t* tiles_gemm;   // [E+1] or nullptr
    uint32_t* err;
    // Expert-parallel shard: ids are global, the routed experts are
    // [expert_start, expert_start + n_experts) of n_global (0 = n_experts);
    // other valid ids are left out (zero rows, no error), ids outside
    // [0, n_global) raise FT_DEVERR_BAD_EXPERT_ID.
    int32_t expert_start;
    int32_t n_global;
};

inline int64_t route_chunks(int64_t n_slots) { return (n_slots + kRouteChunk - 1) / kRouteChunk; }

// Launches the three routing kernels.  When zero_rows != nullptr the rows of
// slots with a bad expert id are zeroed there (row_words 4-byte words each).
int launch_route(const int32_t* ids, int64_t n_slots, int32_t n_experts, const RouteBuffers& b,
                 int32_t gemv_group, int32_t gemm_group, uint32_t* zero_rows, int64_t row_words, cudaStream_t s);

// ------------------------------------------------------------------ GEMV
struct GemvPlan {
    int group;            // slots per tile (1, 2, 4 or 8)
    int row_warps;        // row-per-lane kernel: row groups of 32 per CTA (0: the block-per-lane kernel)
    int ksplit;           // row-per-lane kernel: warps that share a row group
    int64_t min_tiles;    // slot tiles the batch has at least (ceil(S / group))
    int rows;             // weight rows per stage (8 * rows per warp)
    int lanes_per_row;    // rows per warp per stage (1, 2 or 4)
    int stages;           // depth of the bulk-copy ring
    int64_t grid_x;       // slot-tile upper bound
    int64_t row_tiles;    // grid.y: CTAs per slot tile
    int64_t rows_per_cta;
    size_t smem;
    // Q4_0 tiles of `mma` groups of 8 slots on mma.sync (moe_gemv_mma.cu; 0:
    // the dp4a kernels); row_warps (warps of 16 rows there), stages and smem
    // then describe that kernel
    int mma;
};

// mean: routed slots per expert on average (decides the slots per tile);
// mma: Q4_0 tiles with more than 4 slots may run on the mma.sync kernel
GemvPlan plan_gemv(int64_t n_slots, int32_t n_experts, int64_t nrows, int64_t ncols, double mean,
                   int wtype = FT_TYPE_Q4_0, bool mma = true);
// bytes of one stored block of a FT_TYPE_* weight type (0: unknown type) and
// the weights it holds (32, or 256 for the K-quant super-blocks)
int weight_block_bytes(int wtype);
int weight_block_values(int wtype);
// Row-per-lane GEMV kernel: bytes of a row's 256 weights of a FT_TYPE_* type
// and their pitch in a shared-memory box (0: the type does not run there).
int row_box_bytes(int wtype);
int row_box_pitch(int wtype);

int launch_gemv(const GemvPlan& plan, const uint8_t* weights, const uint8_t* act, const int32_t* perm,
                const int32_t* offsets, const int32_t* tiles, float* out, int32_t* dots, uint32_t* err,
                int64_t n_slots, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols, cudaStream_t s,
                int wtype = FT_TYPE_Q4_0);

// The decode step in one launch (moe_decode.cu): the row-per-lane GEMV with
// the routing and the activation quantizer done per CTA, from fp16 x
// [tokens][ncols] and the ids; Q4_0 weights.  gemv_fused_ok: whether the plan
// and sizes allow it (and it pays off).
bool gemv_fused_ok(const GemvPlan& plan, int64_t n_slots, int32_t n_experts, int64_t ncols);
int launch_gemv_fused(const GemvPlan& plan, const uint8_t* weights, const uint16_t* x, const int32_t* ids,
                      float* out, uint32_t* err, int64_t n_slots, int32_t top_k, int32_t n_experts, int64_t nrows,
                      int64_t ncols, cudaStream_t s);

// ------------------------------------------------------------------ GEMM
constexpr int kGemmBN = 128;   // slots per tile
constexpr int kGemmBM = 128;   // weight rows per tile

// Slot-tile width (32 or 128) the tensor-core path uses for this batch; the
// router's GEMM tile prefix must be built with the same width.
int gemm_tile_width(double mean_slots_per_expert);

inline int64_t gemm_rows(int64_t n_slots) { return (n_slots + kGemmBN - 1) / kGemmBN * kGemmBN; }

// xh: [S_pad][ncols] fp16 and da: [S_pad][ncols/32] fp16 workspace for the
// routed activations in router order, S_pad = gemm_rows(S): written by
// launch_gather (zero past the routed slots), then read by the GEMM's TMA.
// sa != nullptr (Q4_K weights): also the exact d_a * sum(q_a) of every block, [S_pad][ncols/32] fp32.
int launch_gather(const uint8_t* act, const int32_t* perm, const int32_t* offsets, int32_t n_experts, int32_t top_k,
                  int64_t nb, int64_t n_slots, uint16_t* xh, uint16_t* da, cudaStream_t s, float* sa = nullptr);
// Layer 1 with the gated activation fused into the epilogue: the weights
// hold n_inter gate rows then n_inter up rows per expert (nrows = 2 n_inter),
// and instead of out the kernel writes act_mid [S][n_inter / 32] Q8_1 rows of
// act(gate) * up (kind: FT_ACT_*).
struct ActFuse {
    uint8_t* act_mid;
    int64_t n_inter;
    int32_t kind;
};

int launch_gemm(const uint8_t* weights, const uint8_t* act, const int32_t* perm, const int32_t* offsets,
                const int32_t* tiles, float* out, int32_t* dots, uint32_t* err, int64_t n_slots, int32_t top_k,
                int32_t n_experts, int64_t nrows, int64_t ncols, uint16_t* xh, uint16_t* da, int tile_width,
                cudaStream_t s, const ActFuse* af = nullptr, const float* sa = nullptr);

}  // namespace ft
