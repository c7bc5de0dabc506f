// The row-per-lane GEMV kernel (gemv_rows.cuh) instantiated for the GGUF
// weight types other than Q4_0 that it runs (Q4_1, Q5_0, Q5_1, Q8_0, Q4_K,
// Q5_K: the per-type launchers of moe_vec.cuh on FreeToken PR #185, "Notes"),
// in a translation unit of its own so that the library's sources compile in
// parallel.
#include "gemv_rows.cuh"

namespace ft {

int launch_gemv_rows_gguf(int wtype, const GemvPlan& plan, const CUtensorMap& wmap, const GemvArgs& a,
                          cudaStream_t s) {
    switch (wtype) {
        case FT_TYPE_Q4_1: return launch_gemv_rows_type<FT_TYPE_Q4_1>(plan, wmap, a, s);
        case FT_TYPE_Q5_0: return launch_gemv_rows_type<FT_TYPE_Q5_0>(plan, wmap, a, s);
        case FT_TYPE_Q5_1: return launch_gemv_rows_type<FT_TYPE_Q5_1>(plan, wmap, a, s);
        case FT_TYPE_Q8_0: return launch_gemv_rows_type<FT_TYPE_Q8_0>(plan, wmap, a, s);
        case FT_TYPE_Q4_K: return launch_gemv_rows_type<FT_TYPE_Q4_K>(plan, wmap, a, s);
        case FT_TYPE_Q5_K: return launch_gemv_rows_type<FT_TYPE_Q5_K>(plan, wmap, a, s);
        default: return fail(FT_ERR_ARG, "weight type %d has no row-per-lane kernel", wtype);
    }
}

}  // namespace ft
