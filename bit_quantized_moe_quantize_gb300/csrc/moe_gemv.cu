// GEMV path of the routed Q4_0 x Q8_1 expert matmul (moe_vec_q4_0_q8_1 on
// FreeToken PR #185) and of its other GGUF weight types, for batches with few
// slots per expert (decode): the plan (plan_gemv) and the launch
// (launch_gemv) of three kernels:
//  - moe_gemv_mma_kernel (moe_gemv_mma.cu): Q4_0, Q4_1, Q8_0, Q4_K rows of
//    whole 256-weight runs with more than 4 slots per expert on average;
//    tiles of 8 or 16 slots on mma.sync, one CTA per SM over a weighted
//    split of (tile, 16-row group) units;
//  - moe_gemv_rows_kernel (gemv_rows.cuh): one weight row per lane, rows of
//    whole 256-weight runs of the types with 16-byte box rows, tiles of 1, 2,
//    4 or 8 slots;
//  - moe_gemv_kernel (gemv_blocks.cuh): one 32-weight block per lane, any row
//    length and every type.
//
// Launch geometry of the last two.  grid.x enumerates slot tiles: each is up
// to G slots of one expert taken from the router's permutation, so grid.x is
// bounded by ceil(S / G) + min(E, S) and can reach 2^31 - 1 (FreeToken PR
// #185, "Fix": the flat (token, top-k) index belongs on grid.x, never on
// grid.z).  The tile -> expert map is a binary search over the router's tile
// prefix, i.e. searchsorted(right=True) (nvfp4-megamoe-kernel CURRENT_BUG.md,
// Bug 2), so empty experts own no tile.  grid.y splits the expert's rows into
// contiguous ranges, sized from the SM count so that all CTAs stream at once
// (<= 65535).  Extra CTAs of the upper bound exit.
//
// Every kernel stages a tile's activation rows once per CTA and streams the
// tile's expert rows (contiguous, because an expert's rows are) through an
// mbarrier-tracked ring of TMA boxes or bulk copies, so each weight block is
// read once from shared memory for all the tile's slots and weight bytes
// leave HBM once per (expert, slot group).  Every block dot is the exact
// integer sum_i q_w[i] q_a[i] (minus level0 sum_i q_a[i]), scaled by d_w d_a
// in fp32 (plus the type's offset term).
#include <mutex>

#include <cuda_fp16.h>

#include "gemv_rows.cuh"

namespace ft {

int weight_block_bytes(int wtype) {
    switch (wtype) {
        case FT_TYPE_Q4_0: return WBlock<FT_TYPE_Q4_0>::bytes;
        case FT_TYPE_Q4_1: return WBlock<FT_TYPE_Q4_1>::bytes;
        case FT_TYPE_Q5_0: return WBlock<FT_TYPE_Q5_0>::bytes;
        case FT_TYPE_Q5_1: return WBlock<FT_TYPE_Q5_1>::bytes;
        case FT_TYPE_Q8_0: return WBlock<FT_TYPE_Q8_0>::bytes;
        case FT_TYPE_Q4_K: return WBlock<FT_TYPE_Q4_K>::bytes;
        case FT_TYPE_Q5_K: return WBlock<FT_TYPE_Q5_K>::bytes;
        case FT_TYPE_Q6_K: return WBlock<FT_TYPE_Q6_K>::bytes;
        case FT_TYPE_Q2_K: return WBlock<FT_TYPE_Q2_K>::bytes;
        case FT_TYPE_Q3_K: return WBlock<FT_TYPE_Q3_K>::bytes;
        default: return 0;
    }
}

int weight_block_values(int wtype) {
    return wtype == FT_TYPE_Q4_K || wtype == FT_TYPE_Q5_K || wtype == FT_TYPE_Q6_K || wtype == FT_TYPE_Q2_K ||
                   wtype == FT_TYPE_Q3_K
               ? 256
           : weight_block_bytes(wtype)                                            ? 32
                                                                                  : 0;
}

int row_box_bytes(int wtype) {
    switch (wtype) {
        case FT_TYPE_Q4_0: return RowBox<FT_TYPE_Q4_0>::BYTES;
        case FT_TYPE_Q4_1: return RowBox<FT_TYPE_Q4_1>::BYTES;
        case FT_TYPE_Q5_0: return RowBox<FT_TYPE_Q5_0>::BYTES;
        case FT_TYPE_Q5_1: return RowBox<FT_TYPE_Q5_1>::BYTES;
        case FT_TYPE_Q8_0: return RowBox<FT_TYPE_Q8_0>::BYTES;
        case FT_TYPE_Q4_K: return RowBox<FT_TYPE_Q4_K>::BYTES;
        case FT_TYPE_Q5_K: return RowBox<FT_TYPE_Q5_K>::BYTES;
        default: return 0;   // Q6_K, Q2_K, Q3_K: super-blocks not whole 16-byte chunks
    }
}

int row_box_pitch(int wtype) {
    switch (wtype) {
        case FT_TYPE_Q4_0: return RowBox<FT_TYPE_Q4_0>::PITCH;
        case FT_TYPE_Q4_1: return RowBox<FT_TYPE_Q4_1>::PITCH;
        case FT_TYPE_Q5_0: return RowBox<FT_TYPE_Q5_0>::PITCH;
        case FT_TYPE_Q5_1: return RowBox<FT_TYPE_Q5_1>::PITCH;
        case FT_TYPE_Q8_0: return RowBox<FT_TYPE_Q8_0>::PITCH;
        case FT_TYPE_Q4_K: return RowBox<FT_TYPE_Q4_K>::PITCH;
        case FT_TYPE_Q5_K: return RowBox<FT_TYPE_Q5_K>::PITCH;
        default: return 0;
    }
}

GemvPlan plan_gemv(int64_t n_slots, int32_t n_experts, int64_t nrows, int64_t ncols, double mean, int wtype,
                   bool mma) {
    // row bytes per 32 weights (144 / 8, 176 / 8 for Q4_K, Q5_K; Q6_K's 210 / 8
    // rounded up, enough for sizing the ring)
    const int block_bytes = (weight_block_bytes(wtype) * 32 + weight_block_values(wtype) - 1) / weight_block_values(wtype);
    GemvPlan p{};
    const int64_t nb = ncols / QK;
    p.group = mean <= 1.0 ? 1 : mean <= 2.0 ? 2 : mean <= 4.0 ? 4 : 8;
    if (ncols % 256 == 0 && row_box_pitch(wtype) > 0) {
        // row-per-lane kernel.  KS warps per row group so that the batch
        // keeps ~32 compute warps per SM busy, then as many row groups per CTA
        // (RW, RW * KS <= 8) as still leave two CTAs per SM; a ring of
        // 2 KS boxes when the K range is split, else as deep as ~110 KB allows;
        // grid.y sized so that every CTA is resident at once.
        // expected routed slots (an expert-parallel shard routes only its share)
        const double expect = mean * n_experts < static_cast<double>(n_slots) ? mean * n_experts : n_slots;
        const int64_t local = static_cast<int64_t>(expect + 0.999);
        const int64_t min_tiles = local > 0 ? (local + p.group - 1) / p.group : 1;
        const int64_t groups32 = (nrows + 31) / 32;
        const int64_t sms = sm_count();
        const int64_t n_ks = nb / 8;
        // (8-slot tiles hold ~134 registers per thread, so splitting them
        // further halves the CTAs an SM holds: keep those at ~16 warps)
        const int64_t target = (p.group >= 8 ? 16 : 32) * sms;
        const int64_t want = (target + min_tiles * groups32 - 1) / (min_tiles * groups32);
        int ks = 1;
        while (ks < want && ks < 8 && 2 * ks <= n_ks) ks *= 2;
        int rw = 1;
        for (int w = 4; w > 1; w >>= 1)
            if (w * ks <= 8 && min_tiles * ((groups32 + w - 1) / w) >= 2 * sms) {
                rw = w;
                break;
            }
        p.row_warps = rw;
        p.ksplit = ks;
        const size_t ring0 = gemv_rows_ring_offset(p.group, static_cast<int>(nb), rw, ks);
        const size_t stage = static_cast<size_t>(row_box_pitch(wtype)) * 32 * rw;
        int st;
        if (ks > 1) {
            st = 2 * ks;
        } else {
            const size_t budget = 110 * 1024;
            st = budget > ring0 ? static_cast<int>((budget - ring0) / stage) : 0;
        }
        st = st < 2 ? 2 : st > kMaxRowStages ? kMaxRowStages : st;
        p.stages = st;
        p.smem = ring0 + static_cast<size_t>(st) * stage;
        const int64_t ub = (n_slots + p.group - 1) / p.group + (n_experts < n_slots ? n_experts : n_slots);
        p.grid_x = ub < n_slots ? ub : n_slots;
        // grid.y (row blocks per slot tile) is set at launch from the kernel's
        // occupancy, so that every CTA is resident at once
        p.rows_per_cta = (nrows + 32 * rw - 1) / (32 * rw);   // row blocks per slot tile
        p.min_tiles = min_tiles;
        p.row_tiles = 0;
        if (mma && (wtype == FT_TYPE_Q4_0 || wtype == FT_TYPE_Q4_1 || wtype == FT_TYPE_Q8_0 || wtype == FT_TYPE_Q4_K) &&
            mean > 4.0) {
            // tiles on mma.sync: 16 slots (two groups of 8) where their staged
            // activation tile leaves room for a ring, else 8.  One CTA per SM
            // of RW warps of 16 rows (fewer when the batch has fewer row blocks
            // than SMs), RW chosen for a ring of at least 3 boxes where one
            // exists; at most 15, so that with the producer each scheduler runs
            // 4 warps and a thread may hold 128 registers (a 17th warp puts 5 on
            // one scheduler and caps them at 96)
            const size_t cap = 227 * 1024;
            const int64_t groups16 = (nrows + 15) / 16;
            for (int nt = 2; nt >= 1; --nt) {
                const int64_t tiles = (local + 8 * nt - 1) / (8 * nt);
                int best_rw = 0, best_st = 0;
                static const int kRowWarps[] = {15, 12, 8, 4, 2, 1};
                for (int need = 3; need >= 2 && best_rw == 0; --need)
                    for (int mrw : kRowWarps) {
                        // fewer rows per block only where the row blocks would not cover the SMs
                        if (mrw > 1 && tiles * ((groups16 + mrw - 1) / mrw) < sms) continue;
                        const size_t r0 = gemv_mma_smem(static_cast<int>(nb), nt, mrw, 0, wtype);
                        const size_t stg = static_cast<size_t>(row_box_pitch(wtype)) * 16 * mrw;
                        int st = cap > r0 ? static_cast<int>((cap - r0) / stg) : 0;
                        st = st > kMaxRowStages ? kMaxRowStages : st;
                        if (st >= need) {
                            best_rw = mrw;
                            best_st = st;
                            break;
                        }
                    }
                if (best_rw == 0) continue;
                p.mma = nt;
                p.group = 8 * nt;
                p.row_warps = best_rw;
                p.ksplit = 1;
                p.stages = best_st;
                p.smem = gemv_mma_smem(static_cast<int>(nb), nt, best_rw, best_st, wtype);
                p.min_tiles = tiles > 0 ? tiles : 1;
                const int64_t ub2 = (n_slots + p.group - 1) / p.group + (n_experts < n_slots ? n_experts : n_slots);
                p.grid_x = ub2 < n_slots ? ub2 : n_slots;
                p.rows_per_cta = (nrows + 16 * best_rw - 1) / (16 * best_rw);
                break;
            }
        }
        return p;
    }
    const int64_t row_bytes = nb * block_bytes;
    // rows per warp: a stage of 8 * RW rows of about 40 KB
    const int64_t rw = 40960 / (8 * row_bytes);
    p.lanes_per_row = rw >= 4 ? 4 : rw >= 2 ? 2 : 1;   // RW (rows per warp per stage)
    p.rows = 8 * p.lanes_per_row;
    const size_t act = gemv_act_bytes(p.group, static_cast<int>(nb));
    const size_t stage = gemv_stage_bytes(p.rows, static_cast<int>(nb), block_bytes);
    const size_t budget = 220 * 1024;
    int stages = static_cast<int>(budget > act ? (budget - act) / stage : 0);
    while (stages < 2 && p.group > 1) {                 // very long rows: fewer slots per tile
        p.group >>= 1;
        const size_t act2 = gemv_act_bytes(p.group, static_cast<int>(nb));
        stages = static_cast<int>(budget > act2 ? (budget - act2) / stage : 0);
    }
    // 0 stages: one stage of 8 rows does not fit; the host rejects the shape
    p.stages = stages < 0 ? 0 : stages > kMaxStages ? kMaxStages : stages;
    p.smem = gemv_act_bytes(p.group, static_cast<int>(nb)) + static_cast<size_t>(p.stages) * stage;
    const int64_t ub = (n_slots + p.group - 1) / p.group + (n_experts < n_slots ? n_experts : n_slots);
    p.grid_x = ub < n_slots ? ub : n_slots;
    // spread each slot tile's rows over enough CTAs that every SM streams
    const int64_t stages_total = (nrows + p.rows - 1) / p.rows;
    const int64_t ctas_per_sm = p.smem <= 110 * 1024 ? 2 : 1;
    const int64_t target = static_cast<int64_t>(sm_count()) * ctas_per_sm;
    const int64_t min_tiles = (n_slots + p.group - 1) / p.group;     // at least this many slot tiles exist
    int64_t y = min_tiles > 0 ? (target + min_tiles - 1) / min_tiles : 1;
    y = y < 1 ? 1 : y > stages_total ? stages_total : y;
    y = y > 65535 ? 65535 : y;
    p.row_tiles = y;
    p.rows_per_cta = (stages_total + y - 1) / y * p.rows;
    return p;
}

// CTAs of a kernel that fit on one SM at once (cached per device, kernel,
// block size and shared memory).
int resident_ctas(const void* kernel, int threads, size_t smem) {
    struct Entry {
        const void* k;
        int dev, threads;
        size_t smem;
        int n;
    };
    static Entry cache[64];
    static int n_cache = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_cache; ++i)
        if (cache[i].k == kernel && cache[i].dev == dev && cache[i].threads == threads && cache[i].smem == smem)
            return cache[i].n;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 1;
    }
    if (n_cache < 64) cache[n_cache++] = Entry{kernel, dev, threads, smem, n};
    return n;
}

int launch_gemv(const GemvPlan& plan, const uint8_t* weights, const uint8_t* act, const int32_t* perm,
                const int32_t* offsets, const int32_t* tiles, float* out, int32_t* dots, uint32_t* err,
                int64_t n_slots, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols, cudaStream_t s,
                int wtype) {
    if (plan.grid_x == 0) return FT_OK;
    GemvArgs a{};
    a.weights = weights;
    a.act = act;
    a.perm = perm;
    a.offsets = offsets;
    a.tiles = tiles;
    a.out = out;
    a.dots = dots;
    a.err = err;
    a.nrows = nrows;
    a.nb = static_cast<int32_t>(ncols / QK);
    a.top_k = top_k;
    a.n_experts = n_experts;
    a.stages = plan.stages;
    a.rows_per_cta = plan.rows_per_cta;
    a.bulk = ((ncols / weight_block_values(wtype) * weight_block_bytes(wtype)) % 16 == 0) &&
             ((reinterpret_cast<uintptr_t>(weights) & 15u) == 0);
    a.row_warps = plan.row_warps;
    a.ksplit = plan.ksplit;
    (void)n_slots;
    const bool dump = dots != nullptr;
    if (dump && wtype != FT_TYPE_Q4_0) return fail(FT_ERR_ARG, "weight type %d: block dots are Q4_0 only", wtype);
    if (plan.row_warps > 0) {
        // boxes of 256 weights x 32 RW rows, 16-bit elements (a Q8_0 box row is
        // 272 bytes, past the 256 elements a box dimension may hold in bytes)
        const int bytes = row_box_bytes(wtype), pitch = row_box_pitch(wtype);
        const uint64_t row_bytes = static_cast<uint64_t>(a.nb / 8) * bytes;
        CUtensorMap wmap;
        // (rows per box: 32 per row warp, 16 on the mma.sync kernel)
        if (int st = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, weights, row_bytes / 2,
                               static_cast<uint64_t>(n_experts) * nrows, row_bytes, pitch / 2,
                               (plan.mma ? 16 : 32) * plan.row_warps, CU_TENSOR_MAP_SWIZZLE_NONE, "weights"))
            return st;
        if (plan.mma) {
            CUtensorMap wmap16;
            if (int st = encode_2d(&wmap16, CU_TENSOR_MAP_DATA_TYPE_UINT16, weights, row_bytes / 2,
                                   static_cast<uint64_t>(n_experts) * nrows, row_bytes, pitch / 2, 16,
                                   CU_TENSOR_MAP_SWIZZLE_NONE, "weights"))
                return st;
            return launch_gemv_mma(plan, wmap, wmap16, a, dump, wtype, s);
        }
        if (wtype != FT_TYPE_Q4_0) return launch_gemv_rows_gguf(wtype, plan, wmap, a, s);
        switch (plan.group) {
            case 1: return dump ? launch_gemv_rows<FT_TYPE_Q4_0, 1, true>(plan, wmap, a, s) : launch_gemv_rows<FT_TYPE_Q4_0, 1, false>(plan, wmap, a, s);
            case 2: return dump ? launch_gemv_rows<FT_TYPE_Q4_0, 2, true>(plan, wmap, a, s) : launch_gemv_rows<FT_TYPE_Q4_0, 2, false>(plan, wmap, a, s);
            case 4: return dump ? launch_gemv_rows<FT_TYPE_Q4_0, 4, true>(plan, wmap, a, s) : launch_gemv_rows<FT_TYPE_Q4_0, 4, false>(plan, wmap, a, s);
            default: return dump ? launch_gemv_rows<FT_TYPE_Q4_0, 8, true>(plan, wmap, a, s) : launch_gemv_rows<FT_TYPE_Q4_0, 8, false>(plan, wmap, a, s);
        }
    }
    if (wtype != FT_TYPE_Q4_0) return launch_gemv_gguf(wtype, plan, a, s);
    switch (plan.group) {
        case 1: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 1, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 1, false>(plan, a, s);
        case 2: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 2, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 2, false>(plan, a, s);
        case 4: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 4, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 4, false>(plan, a, s);
        default: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 8, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 8, false>(plan, a, s);
    }
}

}  // namespace ft
