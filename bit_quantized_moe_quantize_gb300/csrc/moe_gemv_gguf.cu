// The block-per-lane GEMV kernel instantiated for the GGUF weight types other
// than Q4_0 (Q4_1, Q5_0, Q5_1, Q8_0, Q2_K..Q6_K: the per-type launchers of
// moe_vec.cuh on FreeToken PR #185, "Notes"), in a translation unit of its
// own so that the library's sources compile in parallel (the row-per-lane
// kernel's instances are in moe_gemv_rows_gguf.cu).  No block dots (a Q4_0
// diagnostic).
#include "gemv_blocks.cuh"

namespace ft {

template <int WT>
static int launch_gemv_type(const GemvPlan& plan, const GemvArgs& a, cudaStream_t s) {
    switch (plan.group) {
        case 1: return launch_gemv_rw<WT, 1, false>(plan, a, s);
        case 2: return launch_gemv_rw<WT, 2, false>(plan, a, s);
        case 4: return launch_gemv_rw<WT, 4, false>(plan, a, s);
        default: return launch_gemv_rw<WT, 8, false>(plan, a, s);
    }
}

int launch_gemv_gguf(int wtype, const GemvPlan& plan, const GemvArgs& a, cudaStream_t s) {
    switch (wtype) {
        case FT_TYPE_Q4_1: return launch_gemv_type<FT_TYPE_Q4_1>(plan, a, s);
        case FT_TYPE_Q5_0: return launch_gemv_type<FT_TYPE_Q5_0>(plan, a, s);
        case FT_TYPE_Q5_1: return launch_gemv_type<FT_TYPE_Q5_1>(plan, a, s);
        case FT_TYPE_Q8_0: return launch_gemv_type<FT_TYPE_Q8_0>(plan, a, s);
        case FT_TYPE_Q4_K: return launch_gemv_type<FT_TYPE_Q4_K>(plan, a, s);
        case FT_TYPE_Q5_K: return launch_gemv_type<FT_TYPE_Q5_K>(plan, a, s);
        case FT_TYPE_Q6_K: return launch_gemv_type<FT_TYPE_Q6_K>(plan, a, s);
        case FT_TYPE_Q2_K: return launch_gemv_type<FT_TYPE_Q2_K>(plan, a, s);
        case FT_TYPE_Q3_K: return launch_gemv_type<FT_TYPE_Q3_K>(plan, a, s);
        default: return fail(FT_ERR_ARG, "unknown weight type %d", wtype);
    }
}

}  // namespace ft
