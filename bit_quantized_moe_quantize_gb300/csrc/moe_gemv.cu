// GEMV path of the routed Q4_0 x Q8_1 expert matmul (moe_vec_q4_0_q8_1 on
// FreeToken PR #185), for batches with few slots per expert (decode).  Two
// kernels share the launch geometry below: moe_gemv_rows_kernel (one weight
// row per lane; rows a multiple of 16 bytes) and moe_gemv_kernel (one block
// per lane; any row length).
//
// Launch geometry.  grid.x enumerates slot tiles: each is up to G slots of
// one expert taken from the router's permutation, so grid.x is bounded by
// ceil(S / G) + min(E, S) and can reach 2^31 - 1 (FreeToken PR #185, "Fix":
// the flat (token, top-k) index belongs on grid.x, never on grid.z).  The
// tile -> expert map is a binary search over the router's tile prefix, i.e.
// searchsorted(right=True) (nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 2), so
// empty experts own no tile.  grid.y splits the expert's rows into contiguous
// ranges, sized from the SM count so that all CTAs stream at once (<= 65535).
// Extra CTAs of the upper bound exit.
//
// Per CTA: the G activation rows are staged once in shared memory as 16-byte
// aligned int8 blocks plus fp32 scales and exact block sums; the row range's
// Q4_0 bytes (contiguous, because an expert's rows are) stream through a ring
// of up to four mbarrier-tracked bulk copies (cp.async.bulk) of ~40 KB, so
// several copies are in flight while the previous stage is computed.  Each
// weight block is read once from shared memory and dotted with all G slots,
// so weight bytes leave HBM once per (expert, slot group).
//
// Arithmetic: per block, sum_i q_w[i] * q_a[i] with dp4a on the raw nibbles,
// then minus 8 * sum_i q_a[i] (exact integer), so the block dot is bit-exact;
// it is scaled by d_w * d_a in fp32 and summed over the lane's blocks, then
// across lanes with shuffles.
#include <mutex>

#include <cuda_fp16.h>

#include "gemv_blocks.cuh"

namespace ft {

// Row-per-lane kernel's shared memory: mbarriers full/empty [kMaxRowStages]
// and red_full/red_empty [2] | slot ids int32[G] | qa [G][nb][32] | aux
// float2 [G][nb] | partial sums [2][ksplit-1][row warps][32][G] fp32 | ring of
// boxes (128-byte aligned, 144 x 32 * row warps bytes each).
constexpr int kMaxRowStages = 16;
__host__ __device__ inline size_t gemv_rows_qa_offset(int G) {
    return (8 * (2 * kMaxRowStages + 4) + static_cast<size_t>(G) * 4 + 15) / 16 * 16;
}
__host__ __device__ inline size_t gemv_rows_red_offset(int G, int nb) {
    return gemv_rows_qa_offset(G) + static_cast<size_t>(G) * nb * 40;
}
__host__ __device__ inline size_t gemv_rows_ring_offset(int G, int nb, int row_warps, int ksplit) {
    const size_t red = static_cast<size_t>(2) * (ksplit - 1) * row_warps * 32 * G * 4;
    return (gemv_rows_red_offset(G, nb) + red + 127) / 128 * 128;
}

// ---------------------------------------------------------------------------
// Row-per-lane kernel, for rows that are a whole number of 16-byte chunks
// (ncols % 256 == 0).  grid.x: slot tiles (G slots of one expert); grid.y:
// blocks of 32 RW weight rows of that expert (looping past 65535).  Lane l of
// a compute warp owns one row, so the lane keeps the G partial sums of its row
// in registers: no cross-lane reduction, and a warp's output store is 32
// consecutive floats.  The weights stream through a ring of TMA boxes of 8
// Q4_0 blocks (144 bytes) x 32 RW rows, refilled by a producer warp; in shared
// memory a row of the box is 9 16-byte chunks, an odd count, so the 32 lanes'
// 16-byte loads of their own rows never collide on a bank.  The G slots'
// activations are staged once per CTA and every read of them is the same
// address for the whole warp (a broadcast).
//
// When the batch has few tiles (one token), KS warps share each row group:
// warp (r, k) takes boxes k, k + KS, ... of row group r, so a CTA streams with
// KS times as many warps; warps k > 0 hand their partial sums to warp k = 0
// through shared memory (two mbarriers per parity, bounded waits), which adds
// them in order k = 0, 1, ..., KS-1, so the result does not depend on timing.
template <int G, bool DUMP>
__global__ void __launch_bounds__(288) moe_gemv_rows_kernel(const __grid_constant__ CUtensorMap wmap,
                                                             const GemvArgs a) {
    constexpr int KB = 8;                                 // blocks per box
    constexpr int BOX_ROW = KB * Q4_0_BYTES;              // 144
    const int32_t RW = a.row_warps, KS = a.ksplit;
    const int32_t n_compute = RW * KS;
    const int64_t t = blockIdx.x;
    const int32_t E = a.n_experts;
    if (t >= a.tiles[E]) return;
    const int32_t e = find_expert(a.tiles, E, t);
    const int64_t p0 = static_cast<int64_t>(a.offsets[e]) + (t - a.tiles[e]) * G;
    const int32_t ng = static_cast<int32_t>(min(static_cast<int64_t>(G), a.offsets[e + 1] - p0));
    const int32_t nb = a.nb;
    const int32_t n_ks = nb / KB;
    const int NS = a.stages;
    const int64_t n_groups = (a.nrows + 32 * RW - 1) / (32 * RW);
    const int64_t my_groups = blockIdx.y < n_groups ? (n_groups - 1 - blockIdx.y) / gridDim.y + 1 : 0;

    extern __shared__ __align__(128) uint8_t smem_rows[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_rows);
    uint64_t* empty = full + kMaxRowStages;
    uint64_t* red_full = empty + kMaxRowStages;           // [2]: partial sums of a row group written
    uint64_t* red_empty = red_full + 2;                   // [2]: ... and consumed
    int32_t* slot = reinterpret_cast<int32_t*>(smem_rows + 8 * (2 * kMaxRowStages + 4));
    uint4* qa = reinterpret_cast<uint4*>(smem_rows + gemv_rows_qa_offset(G));         // [G][nb][2] uint4
    float2* aux = reinterpret_cast<float2*>(qa + static_cast<size_t>(G) * nb * 2);  // [G][nb] {d_a, 8 sum q}
    float* red = reinterpret_cast<float*>(smem_rows + gemv_rows_red_offset(G, nb));   // [2][KS-1][RW][32][G]
    uint8_t* ring = smem_rows + gemv_rows_ring_offset(G, nb, RW, KS);
    const uint32_t stage_bytes = static_cast<uint32_t>(BOX_ROW * 32 * RW);

    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], RW);                     // the RW warps that read a box
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&red_full[i], RW * (KS - 1));
            mbar_init(&red_empty[i], RW);
        }
        fence_mbar_init();
    }
    if (threadIdx.x < G) slot[threadIdx.x] = threadIdx.x < ng ? a.perm[p0 + threadIdx.x] : 0;
    __syncthreads();

    // stage the G activation rows once: 32 int8 as two 16-byte chunks, and
    // {d_a, 8 * sum q} so that each block dot starts from -8 sum q
    for (int32_t i = threadIdx.x; i < G * nb; i += blockDim.x) {
        const int32_t g = i / nb, b = i - g * nb;
        uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
        float d = 0.0f;
        int sm = 0;
        if (g < ng) {
            const int64_t tok = slot[g] / a.top_k;
            const uint32_t* src = reinterpret_cast<const uint32_t*>(a.act + (tok * nb + b) * Q8_1_BYTES);
            const uint32_t ds = __ldg(src);
            q0 = make_uint4(__ldg(src + 1), __ldg(src + 2), __ldg(src + 3), __ldg(src + 4));
            q1 = make_uint4(__ldg(src + 5), __ldg(src + 6), __ldg(src + 7), __ldg(src + 8));
            d = __half2float(__ushort_as_half(static_cast<unsigned short>(ds & 0xFFFFu)));
            sm = __dp4a(static_cast<int>(q0.x), 0x01010101, sm);
            sm = __dp4a(static_cast<int>(q0.y), 0x01010101, sm);
            sm = __dp4a(static_cast<int>(q0.z), 0x01010101, sm);
            sm = __dp4a(static_cast<int>(q0.w), 0x01010101, sm);
            sm = __dp4a(static_cast<int>(q1.x), 0x01010101, sm);
            sm = __dp4a(static_cast<int>(q1.y), 0x01010101, sm);
            sm = __dp4a(static_cast<int>(q1.z), 0x01010101, sm);
            sm = __dp4a(static_cast<int>(q1.w), 0x01010101, sm);
        }
        qa[(static_cast<size_t>(g) * nb + b) * 2] = q0;
        qa[(static_cast<size_t>(g) * nb + b) * 2 + 1] = q1;
        aux[static_cast<size_t>(g) * nb + b] = make_float2(d, __int_as_float(8 * sm));
    }
    __syncthreads();

    const int64_t erow0 = static_cast<int64_t>(e) * a.nrows;   // first weight row of the expert
    if (static_cast<int32_t>(warp) == n_compute) {
        // ------------------------------------------------------------ producer
        // boxes in order: row block g, box ks -> stage index g * n_ks + ks
        const int64_t n_it = my_groups * n_ks;
        int64_t grp = blockIdx.y;
        int32_t ks = 0;
        for (int64_t it = 0; it < n_it; ++it) {
            const int32_t s = static_cast<int32_t>(it % NS);
            if (!mbar_wait_warp(&empty[s], static_cast<uint32_t>(((it / NS) & 1) ^ 1), a.err)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                tma_load_2d(ring + static_cast<size_t>(s) * stage_bytes, &wmap, ks * BOX_ROW,
                            static_cast<int32_t>(erow0 + grp * 32 * RW), &full[s]);
            }
            __syncwarp();
            if (++ks == n_ks) {
                ks = 0;
                grp += gridDim.y;
            }
        }
        return;
    }

    // ----------------------------------------------------------------- compute
    const int32_t r = static_cast<int32_t>(warp) % RW, kk = static_cast<int32_t>(warp) / RW;
    float acc[G];
    bool ok = true;
    for (int64_t gi = 0; gi < my_groups && ok; ++gi) {
        const int64_t grp = blockIdx.y + gi * gridDim.y;
        const int64_t row = grp * 32 * RW + r * 32 + lane;     // row within the expert
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = 0.0f;
        for (int32_t ks = kk; ks < n_ks; ks += KS) {
            const int64_t it = gi * n_ks + ks;
            const int32_t s = static_cast<int32_t>(it % NS);
            if (!mbar_wait_warp(&full[s], static_cast<uint32_t>((it / NS) & 1), a.err)) { ok = false; break; }
            const uint4* rowp = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(s) * stage_bytes +
                                                               (r * 32 + lane) * BOX_ROW);
            uint32_t wv[36];
#pragma unroll
            for (int c = 0; c < 9; ++c) {
                const uint4 v = rowp[c];
                wv[4 * c] = v.x;
                wv[4 * c + 1] = v.y;
                wv[4 * c + 2] = v.z;
                wv[4 * c + 3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                // block j of the box starts at byte 18 j: word 9j/2 (j even, d in its
                // low half) or the high half of word (18j - 2)/4 (j odd)
                uint32_t q[4], dbits;
                if ((j & 1) == 0) {
                    const int w0 = 9 * j / 2;
                    dbits = wv[w0] & 0xFFFFu;
#pragma unroll
                    for (int i = 0; i < 4; ++i) q[i] = __byte_perm(wv[w0 + i], wv[w0 + i + 1], 0x5432u);
                } else {
                    const int w0 = (18 * j - 2) / 4;
                    dbits = wv[w0] >> 16;
#pragma unroll
                    for (int i = 0; i < 4; ++i) q[i] = wv[w0 + 1 + i];
                }
                const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
                int lo[4], hi[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    lo[i] = static_cast<int>(q[i] & 0x0F0F0F0Fu);          // values 4i .. 4i+3
                    hi[i] = static_cast<int>((q[i] >> 4) & 0x0F0F0F0Fu);   // values 16+4i .. 16+4i+3
                }
                const int32_t b = ks * KB + j;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint4 A0 = qa[(static_cast<size_t>(g) * nb + b) * 2];
                    const uint4 A1 = qa[(static_cast<size_t>(g) * nb + b) * 2 + 1];
                    const float2 x = aux[static_cast<size_t>(g) * nb + b];
                    int dot = -__float_as_int(x.y);
                    dot = __dp4a(lo[0], static_cast<int>(A0.x), dot);
                    dot = __dp4a(lo[1], static_cast<int>(A0.y), dot);
                    dot = __dp4a(lo[2], static_cast<int>(A0.z), dot);
                    dot = __dp4a(lo[3], static_cast<int>(A0.w), dot);
                    dot = __dp4a(hi[0], static_cast<int>(A1.x), dot);
                    dot = __dp4a(hi[1], static_cast<int>(A1.y), dot);
                    dot = __dp4a(hi[2], static_cast<int>(A1.z), dot);
                    dot = __dp4a(hi[3], static_cast<int>(A1.w), dot);
                    if constexpr (DUMP) {
                        if (g < ng && row < a.nrows)
                            a.dots[(static_cast<int64_t>(slot[g]) * a.nrows + row) * nb + b] = dot;
                    } else {
                        acc[g] = fmaf(small_int_to_float(dot), dw * x.x, acc[g]);
                    }
                }
            }
            // release the box only after its values have been used: an arrival
            // right after the shared loads can reach the producer while the
            // loaded values are still on their way to registers, and its next
            // TMA write then overtakes them
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (!ok) break;
        if constexpr (!DUMP) {
            if (KS > 1) {
                // hand the partial sums to warp (r, 0); buffer gi & 1 is free again
                // once warp (r, 0) has read what it held two row blocks ago
                const uint32_t pb = static_cast<uint32_t>(gi & 1), ph = static_cast<uint32_t>((gi >> 1) & 1);
                float* rb = red + static_cast<size_t>(pb) * (KS - 1) * RW * 32 * G;
                if (kk > 0) {
                    if (!mbar_wait_warp(&red_empty[pb], ph ^ 1u, a.err)) break;
#pragma unroll
                    for (int g = 0; g < G; ++g) rb[((static_cast<size_t>(kk - 1) * RW + r) * 32 + lane) * G + g] = acc[g];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&red_full[pb]);
                    continue;
                }
                if (!mbar_wait_warp(&red_full[pb], ph, a.err)) break;
                for (int32_t k2 = 1; k2 < KS; ++k2)
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] += rb[((static_cast<size_t>(k2 - 1) * RW + r) * 32 + lane) * G + g];
                __syncwarp();
                if (lane == 0) mbar_arrive(&red_empty[pb]);
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
                if (g < ng && row < a.nrows) a.out[static_cast<int64_t>(slot[g]) * a.nrows + row] = acc[g];
        }
    }
}

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

GemvPlan plan_gemv(int64_t n_slots, int32_t n_experts, int64_t nrows, int64_t ncols, double mean, int wtype) {
    // row bytes per 32 weights (144 / 8, 176 / 8 for Q4_K, Q5_K; Q6_K's 210 / 8
    // rounded up, enough for sizing the ring)
    const int block_bytes = (weight_block_bytes(wtype) * 32 + weight_block_values(wtype) - 1) / weight_block_values(wtype);
    GemvPlan p{};
    const int64_t nb = ncols / QK;
    p.group = mean <= 1.0 ? 1 : mean <= 2.0 ? 2 : mean <= 4.0 ? 4 : 8;
    if (ncols % 256 == 0 && wtype == FT_TYPE_Q4_0) {
        // row-per-lane kernel (Q4_0 only).  KS warps per row group so that the batch
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
        const size_t stage = static_cast<size_t>(144) * 32 * rw;
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
static int resident_ctas(const void* kernel, int threads, size_t smem) {
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

template <int G, bool DUMP>
static int launch_gemv_rows(const GemvPlan& plan, const CUtensorMap& wmap, const GemvArgs& a, cudaStream_t s) {
    const void* kernel = reinterpret_cast<const void*>(moe_gemv_rows_kernel<G, DUMP>);
    if (int st = set_smem_limit(kernel, static_cast<int>(plan.smem))) return st;
    const int threads = 32 * (plan.row_warps * plan.ksplit + 1);
    // grid.y: row blocks per slot tile, few enough that every CTA is resident
    // at once (each then loops over the same number of row blocks)
    const int64_t ng = plan.rows_per_cta;
    const int64_t slots = static_cast<int64_t>(sm_count()) * resident_ctas(kernel, threads, plan.smem);
    const int64_t tiles = plan.min_tiles > 0 ? plan.min_tiles : 1;   // grid.x is only an upper bound
    const int64_t per_cta = (ng * tiles + slots - 1) / slots;
    int64_t y = (ng + per_cta - 1) / per_cta;
    y = y < 1 ? 1 : y > 65535 ? 65535 : y;
    const dim3 grid(static_cast<unsigned>(plan.grid_x), static_cast<unsigned>(y));
    const dim3 block(threads);
    moe_gemv_rows_kernel<G, DUMP><<<grid, block, plan.smem, s>>>(wmap, a);
    return check_launch(DUMP ? "moe_gemv_rows_kernel<dump>" : "moe_gemv_rows_kernel", grid, block, plan.smem);
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
    if (wtype != FT_TYPE_Q4_0) {
        if (dump || plan.row_warps > 0) return fail(FT_ERR_ARG, "weight type %d: block dots and row tiles are Q4_0 only", wtype);
        return launch_gemv_gguf(wtype, plan, a, s);
    }
    if (plan.row_warps > 0) {
        CUtensorMap wmap;
        if (int st = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, weights, a.nb * Q4_0_BYTES,
                               static_cast<uint64_t>(n_experts) * nrows, a.nb * Q4_0_BYTES, 144, 32 * plan.row_warps,
                               CU_TENSOR_MAP_SWIZZLE_NONE, "weights"))
            return st;
        switch (plan.group) {
            case 1: return dump ? launch_gemv_rows<1, true>(plan, wmap, a, s) : launch_gemv_rows<1, false>(plan, wmap, a, s);
            case 2: return dump ? launch_gemv_rows<2, true>(plan, wmap, a, s) : launch_gemv_rows<2, false>(plan, wmap, a, s);
            case 4: return dump ? launch_gemv_rows<4, true>(plan, wmap, a, s) : launch_gemv_rows<4, false>(plan, wmap, a, s);
            default: return dump ? launch_gemv_rows<8, true>(plan, wmap, a, s) : launch_gemv_rows<8, false>(plan, wmap, a, s);
        }
    }
    switch (plan.group) {
        case 1: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 1, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 1, false>(plan, a, s);
        case 2: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 2, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 2, false>(plan, a, s);
        case 4: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 4, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 4, false>(plan, a, s);
        default: return dump ? launch_gemv_rw<FT_TYPE_Q4_0, 8, true>(plan, a, s) : launch_gemv_rw<FT_TYPE_Q4_0, 8, false>(plan, a, s);
    }
}

}  // namespace ft
