// The decode step of the routed Q4_0 x Q8_1 expert matmul in one launch:
// the row-per-lane GEMV kernel (gemv_rows.cuh) instantiated FUSED, so that
// each CTA routes the batch's few slots itself and quantizes its slots' fp16
// activation rows into shared memory, in place of the quantizer and router
// launches before the matmul (quantize_row_q8_1 and moe_vec_q4_0_q8_1 on
// FreeToken PR #185; the slot order of the stable counting sort with
// expert_offsets, nvfp4-megamoe-kernel CURRENT_BUG.md, Bugs 2 and 4).  The
// kernel's main loop, and so its arithmetic, is the routed kernel's.
#include "gemv_rows.cuh"

namespace ft {

// Every CTA quantizes its G slots' rows itself, so the one launch pays off
// only while that is small next to the CTA's weight stream: at most 256
// blocks of 32 values per CTA (G = 8 slots of 4096 columns took 1.8x the two
// launches on the 8-expert 14336 x 4096 layer at 32 tokens).
constexpr int64_t kFuseMaxStagedBlocks = 256;

bool gemv_fused_ok(const GemvPlan& plan, int64_t n_slots, int32_t n_experts, int64_t ncols) {
    if (plan.row_warps <= 0 || plan.mma || n_slots > kFuseMaxSlots || n_experts > kFuseMaxExperts) return false;
    if (static_cast<int64_t>(plan.group) * (ncols / QK) > kFuseMaxStagedBlocks) return false;
    const size_t ring = static_cast<size_t>(plan.stages) * RowBox<FT_TYPE_Q4_0>::PITCH * 32 * plan.row_warps;
    return gemv_fused_scratch_bytes(n_slots, n_experts) <= ring;
}

int launch_gemv_fused(const GemvPlan& plan, const uint8_t* weights, const uint16_t* x, const int32_t* ids,
                      float* out, uint32_t* err, int64_t n_slots, int32_t top_k, int32_t n_experts, int64_t nrows,
                      int64_t ncols, cudaStream_t s) {
    if (plan.grid_x == 0) return FT_OK;
    if (!gemv_fused_ok(plan, n_slots, n_experts, ncols)) return fail(FT_ERR_ARG, "shape outside the one-launch decode step");
    GemvArgs a{};
    a.weights = weights;
    a.out = out;
    a.err = err;
    a.nrows = nrows;
    a.nb = static_cast<int32_t>(ncols / QK);
    a.top_k = top_k;
    a.n_experts = n_experts;
    a.stages = plan.stages;
    a.rows_per_cta = plan.rows_per_cta;
    a.row_warps = plan.row_warps;
    a.ksplit = plan.ksplit;
    a.x = x;
    a.ids = ids;
    a.n_slots = n_slots;
    constexpr int bytes = RowBox<FT_TYPE_Q4_0>::BYTES, pitch = RowBox<FT_TYPE_Q4_0>::PITCH;
    const uint64_t row_bytes = static_cast<uint64_t>(a.nb / 8) * bytes;
    CUtensorMap wmap;
    if (int st = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, weights, row_bytes / 2,
                           static_cast<uint64_t>(n_experts) * nrows, row_bytes, pitch / 2, 32 * plan.row_warps,
                           CU_TENSOR_MAP_SWIZZLE_NONE, "weights"))
        return st;
    switch (plan.group) {
        case 1: return launch_gemv_rows<FT_TYPE_Q4_0, 1, false, true>(plan, wmap, a, s);
        case 2: return launch_gemv_rows<FT_TYPE_Q4_0, 2, false, true>(plan, wmap, a, s);
        case 4: return launch_gemv_rows<FT_TYPE_Q4_0, 4, false, true>(plan, wmap, a, s);
        default: return launch_gemv_rows<FT_TYPE_Q4_0, 8, false, true>(plan, wmap, a, s);
    }
}

}  // namespace ft
