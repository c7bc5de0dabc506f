// Row-per-lane GEMV kernel of the routed expert matmul (moe_vec_q4_0_q8_1
// and the other per-type launchers of moe_vec.cuh on FreeToken PR #185,
// "Problem" and "Notes"), templated on the weight type, for rows that are a
// whole number of 256-weight runs (ncols % 256 == 0).  moe_gemv.cu
// instantiates it for Q4_0 (with the block-dot dump), moe_decode.cu its
// one-launch decode form, moe_gemv_rows_gguf.cu the Q4_1, Q5_0, Q5_1, Q8_0,
// Q4_K and Q5_K forms.  (Tiles with more than 4 slots per expert of Q4_0,
// Q4_1, Q8_0 and Q4_K run on moe_gemv_mma.cu instead, unless the dp4a
// kernels are forced.)
//
// grid.x: slot tiles (G slots of one expert); grid.y: blocks of 32 RW weight
// rows of that expert (looping past 65535).  Lane l of a compute warp owns one
// row, so the lane keeps the G partial sums of its row in registers: no
// cross-lane reduction, and a warp's output store is 32 consecutive floats.
// The weights stream through a ring of TMA boxes of 256 weights (8 blocks of
// 32, or one K-quant super-block) x 32 RW rows, refilled by a producer warp.
// In shared memory a box row is PITCH bytes, an odd number of 16-byte chunks
// (the box reads 16 bytes past a row's 256 weights where their bytes are an
// even number of chunks: Q4_1, Q5_1), so the 32 lanes' 16-byte loads of their
// own rows never collide on a bank.  The G slots' activations are staged once
// per CTA and every read of them is the same address for the whole warp (a
// broadcast).
//
// When the batch has few tiles (one token), KS warps share each row group:
// warp (r, k) takes boxes k, k + KS, ... of row group r, so a CTA streams with
// KS times as many warps; warps k > 0 hand their partial sums to warp k = 0
// through shared memory (two mbarriers per parity, bounded waits), which adds
// them in order k = 0, 1, ..., KS-1, so the result does not depend on timing.
//
// Arithmetic per 32-weight block and slot: the integer dot of the stored
// levels with the activation codes (dp4a; minus level0 * sum(q_a) for Q4_0 and
// Q5_0, exact), scaled by d_w d_a in fp32, plus the offset term m d_a sum(q_a)
// for the types with an offset (the m of Q4_1 / Q5_1, minus d_min m_j for the
// K-quants), with the exact code sum.
#pragma once

#include <type_traits>

#include <cuda_fp16.h>

#include "gemv_blocks.cuh"
#include "q8_1_math.cuh"

namespace ft {

constexpr int kMaxRowStages = 16;

// Box geometry of a weight type on the row-per-lane kernel: BYTES of a row's
// 256 weights, the PITCH they take in shared memory (odd in 16-byte chunks),
// and the parts a lane decodes the box row in (a part's 16-byte chunks held
// in registers at once: at most 11).
template <int WT>
struct RowBox {
    static constexpr int WB = WBlock<WT>::bytes;
    static constexpr bool KQ = WBlock<WT>::per == 8;
    static constexpr int BYTES = KQ ? WB : 8 * WB;
    static constexpr int PITCH = (BYTES / 16) % 2 ? BYTES : BYTES + 16;
    static constexpr int NPART = BYTES > 176 ? 2 : 1;
    static_assert(BYTES % 16 == 0, "a box row must be whole 16-byte chunks");
};

// Part P of a box row: blocks (sub-blocks) [J0, J1) from chunks [C0, C1).
template <int WT, int P>
struct RowPart {
    using B = RowBox<WT>;
    static constexpr int J0 = P * 8 / B::NPART, J1 = (P + 1) * 8 / B::NPART;
    static constexpr int C0 = B::KQ ? 0 : J0 * B::WB / 16;
    static constexpr int C1 = B::KQ ? B::BYTES / 16 : (J1 * B::WB + 15) / 16;
    static constexpr int NW = 4 * (C1 - C0);
};

// Shared memory: mbarriers full/empty [kMaxRowStages] and red_full/red_empty
// [2] | slot ids int32[G] | 4 words (the one-launch routing's result) | qa
// [G][nb][32] | aux float2 [G][nb] | partial sums [2][ksplit-1][row
// warps][32][G] fp32 | ring of boxes (128-byte aligned, PITCH x 32 * row
// warps bytes each).
__host__ __device__ inline size_t gemv_rows_qa_offset(int G) {
    return (8 * (2 * kMaxRowStages + 4) + static_cast<size_t>(G) * 4 + 16 + 15) / 16 * 16;
}
__host__ __device__ inline size_t gemv_rows_red_offset(int G, int nb) {
    return gemv_rows_qa_offset(G) + static_cast<size_t>(G) * nb * 40;
}
__host__ __device__ inline size_t gemv_rows_ring_offset(int G, int nb, int row_warps, int ksplit) {
    const size_t red = static_cast<size_t>(2) * (ksplit - 1) * row_warps * 32 * G * 4;
    return (gemv_rows_red_offset(G, nb) + red + 127) / 128 * 128;
}

// 32-bit word / fp16 at even byte offset o of a register window (o is a
// constant once the loops around the call are unrolled)
template <int NW>
__device__ __forceinline__ uint32_t win_word(const uint32_t (&w)[NW], int o) {
    return (o & 2) ? __byte_perm(w[o >> 2], w[(o >> 2) + 1], 0x5432u) : w[o >> 2];
}
template <int NW>
__device__ __forceinline__ float win_half(const uint32_t (&w)[NW], int o) {
    const uint32_t v = (o & 2) ? (w[o >> 2] >> 16) : (w[o >> 2] & 0xFFFFu);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v)));
}

// The block at byte o of the window (sub-block j of the super-block the
// window holds, for the K-quants): fp32 d and offset m (d_min m_j for the
// K-quants) and its 32 levels as int8 lanes, weights 0..15 in lo[0..3] and
// 16..31 in hi[0..3].  The byte layouts are those decode_block reads.
template <int WT, int NW>
__device__ __forceinline__ void decode_win(const uint32_t (&w)[NW], int o, int j, float& d, float& m, int (&lo)[4],
                                           int (&hi)[4]) {
    m = 0.0f;
    if constexpr (WT == FT_TYPE_Q4_0 || WT == FT_TYPE_Q4_1) {
        constexpr int Q0 = WT == FT_TYPE_Q4_0 ? 2 : 4;
        d = win_half(w, o);
        if constexpr (WT == FT_TYPE_Q4_1) m = win_half(w, o + 2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t q = win_word(w, o + Q0 + 4 * i);
            lo[i] = static_cast<int>(q & 0x0F0F0F0Fu);
            hi[i] = static_cast<int>((q >> 4) & 0x0F0F0F0Fu);
        }
    } else if constexpr (WT == FT_TYPE_Q5_0 || WT == FT_TYPE_Q5_1) {
        constexpr int H0 = WT == FT_TYPE_Q5_0 ? 2 : 4;
        d = win_half(w, o);
        if constexpr (WT == FT_TYPE_Q5_1) m = win_half(w, o + 2);
        const uint32_t qh = win_word(w, o + H0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t q = win_word(w, o + H0 + 4 + 4 * i);
            lo[i] = static_cast<int>((q & 0x0F0F0F0Fu) | spread4(qh >> (4 * i)));
            hi[i] = static_cast<int>(((q >> 4) & 0x0F0F0F0Fu) | spread4(qh >> (16 + 4 * i)));
        }
    } else if constexpr (WT == FT_TYPE_Q8_0) {
        d = win_half(w, o);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = static_cast<int>(win_word(w, o + 2 + 4 * i));
            hi[i] = static_cast<int>(win_word(w, o + 18 + 4 * i));
        }
    } else {
        static_assert(WT == FT_TYPE_Q4_K || WT == FT_TYPE_Q5_K, "weight type of the row-per-lane kernel");
        constexpr int Q0 = WT == FT_TYPE_Q5_K ? 48 : 16;   // nibbles (Q5_K: after 32 bytes of 5th bits)
        const uint32_t sc12[3] = {w[1], w[2], w[3]};
        int sc, mn;
        kquant_scale_min(sc12, j, sc, mn);
        d = win_half(w, 0) * static_cast<float>(sc);
        m = win_half(w, 2) * static_cast<float>(mn);
        const int sh = 4 * (j & 1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t l = (w[(Q0 + 32 * (j >> 1)) / 4 + i] >> sh) & 0x0F0F0F0Fu;
            uint32_t h = (w[(Q0 + 32 * (j >> 1)) / 4 + 4 + i] >> sh) & 0x0F0F0F0Fu;
            if constexpr (WT == FT_TYPE_Q5_K) {   // bit j of each qh byte -> bit 4 of the level byte
                l |= ((w[4 + i] >> j) & 0x01010101u) << 4;
                h |= ((w[8 + i] >> j) & 0x01010101u) << 4;
            }
            lo[i] = static_cast<int>(l);
            hi[i] = static_cast<int>(h);
        }
    }
}

// Limits of the one-launch decode step (FUSED): its routing scratch, ids
// [n_slots] | counts [E], lives in the weight ring before the first box
// arrives.
constexpr int kFuseMaxSlots = 512;
constexpr int kFuseMaxExperts = 1024;
__host__ __device__ inline size_t gemv_fused_scratch_bytes(int64_t n_slots, int32_t n_experts) {
    return 4 * (static_cast<size_t>(n_slots) + n_experts);
}

// The routing of the one-launch decode step, done by each CTA for itself:
// the stable counting sort of the router restricted to what slot tile t
// needs.  All threads load the ids and count them per expert (ids outside
// [0, E) are left out; the CTAs of slot-tile column 0 zero their output rows
// over the row groups they own, and one raises the device error flag); warp 0
// scans ceil(count / G) over the experts to find the expert e owning tile t
// (tiles in expert order, searchsorted(right=True) as with the router's
// prefix), then lists that expert's slots of ranks [r0, r0 + G) in ascending
// slot order.  Returns false where t is past the last tile (uniform).
template <int G>
__device__ __forceinline__ bool fused_route(const GemvArgs& a, int32_t t, int32_t* scratch, int32_t* slot,
                                            int64_t my_groups, int32_t rows_per_group, int32_t& e, int32_t& ng) {
    const int32_t S = static_cast<int32_t>(a.n_slots), E = a.n_experts;
    int32_t* ids = scratch;
    int32_t* cnt = scratch + S;
    int32_t* info = slot + G;                             // outside the ring the weights arrive in
    for (int32_t i = threadIdx.x; i < S; i += blockDim.x) ids[i] = __ldg(a.ids + i);
    for (int32_t i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    bool bad = false;
    for (int32_t i = threadIdx.x; i < S; i += blockDim.x) {
        const int32_t id = ids[i];
        if (id >= 0 && id < E) atomicAdd(&cnt[id], 1);
        else bad = true;
    }
    bad = __syncthreads_or(bad);
    if (bad && blockIdx.x == 0) {
        if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(a.err, FT_DEVERR_BAD_EXPERT_ID);
        for (int32_t s = 0; s < S; ++s) {
            const int32_t id = ids[s];
            if (id >= 0 && id < E) continue;
            for (int64_t gi = 0; gi < my_groups; ++gi) {
                const int64_t r0 = (blockIdx.y + gi * gridDim.y) * rows_per_group;
                for (int32_t r = threadIdx.x; r < rows_per_group; r += blockDim.x)
                    if (r0 + r < a.nrows) a.out[static_cast<int64_t>(s) * a.nrows + r0 + r] = 0.0f;
            }
        }
    }
    if (threadIdx.x < 32) {
        const uint32_t lane = threadIdx.x;
        int32_t base = 0, fe = -1, fr0 = 0;
        for (int32_t c0 = 0; c0 < E; c0 += 32) {
            const int32_t ee = c0 + static_cast<int32_t>(lane);
            const int32_t n = ee < E ? (cnt[ee] + G - 1) / G : 0;
            int32_t inc = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (static_cast<int>(lane) >= o) inc += y;
            }
            const int32_t excl = base + inc - n;
            if (n > 0 && t >= excl && t < excl + n) {
                fe = ee;
                fr0 = (t - excl) * G;
            }
            base += __shfl_sync(0xFFFFFFFFu, inc, 31);
        }
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, fe >= 0);
        if (m) {
            const int src = __ffs(m) - 1;
            fe = __shfl_sync(0xFFFFFFFFu, fe, src);
            fr0 = __shfl_sync(0xFFFFFFFFu, fr0, src);
            if (lane < G) slot[lane] = 0;
            __syncwarp();
            int32_t rank0 = 0;
            for (int32_t c0 = 0; c0 < S; c0 += 32) {
                const int32_t s = c0 + static_cast<int32_t>(lane);
                const bool hit = s < S && ids[s] == fe;
                const uint32_t bm = __ballot_sync(0xFFFFFFFFu, hit);
                const int32_t rank = rank0 + __popc(bm & ((1u << lane) - 1u));
                if (hit && rank >= fr0 && rank < fr0 + G) slot[rank - fr0] = s;
                rank0 += __popc(bm);
            }
        }
        if (lane == 0) {
            info[0] = m ? fe : -1;
            info[1] = m ? min(G, cnt[fe] - fr0) : 0;
        }
    }
    __syncthreads();
    e = info[0];
    ng = info[1];
    return e >= 0;
}

template <int WT, int G, bool DUMP, bool FUSED>
__global__ void __launch_bounds__(288, G >= 8 ? 1 : 2) moe_gemv_rows_kernel(const __grid_constant__ CUtensorMap wmap,
                                                             const GemvArgs a) {
    using BX = RowBox<WT>;
    constexpr int PITCH = BX::PITCH;
    constexpr int LEVEL0 = WBlock<WT>::level0;
    constexpr bool OFFSET = WBlock<WT>::has_m || WBlock<WT>::has_min;   // an m d_a sum(q_a) term
    constexpr float MSIGN = WBlock<WT>::has_min ? -1.0f : 1.0f;       // K-quant mins are subtracted
    static_assert(!DUMP || WT == FT_TYPE_Q4_0, "block dots are a Q4_0 diagnostic");
    const int32_t RW = a.row_warps, KS = a.ksplit;
    const int32_t n_compute = RW * KS;
    static_assert(!(DUMP && FUSED), "block dots come from the routed form");
    const int64_t t = blockIdx.x;
    const int32_t E = a.n_experts;
    int32_t e = 0, ng = 0;
    int64_t p0 = 0;
    if constexpr (!FUSED) {
        if (t >= a.tiles[E]) return;
        e = find_expert(a.tiles, E, t);
        p0 = static_cast<int64_t>(a.offsets[e]) + (t - a.tiles[e]) * G;
        ng = static_cast<int32_t>(min(static_cast<int64_t>(G), a.offsets[e + 1] - p0));
    }
    const int32_t nb = a.nb;
    const int32_t n_ks = nb / 8;                          // boxes per row
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
    float2* aux = reinterpret_cast<float2*>(qa + static_cast<size_t>(G) * nb * 2);  // [G][nb]
    float* red = reinterpret_cast<float*>(smem_rows + gemv_rows_red_offset(G, nb));   // [2][KS-1][RW][32][G]
    uint8_t* ring = smem_rows + gemv_rows_ring_offset(G, nb, RW, KS);
    const uint32_t stage_bytes = static_cast<uint32_t>(PITCH * 32 * RW);
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
    if constexpr (FUSED) {
        // the routing's barriers also publish the mbarriers; the producer then
        // starts streaming at once while the compute warps quantize
        if (!fused_route<G>(a, static_cast<int32_t>(t), reinterpret_cast<int32_t*>(ring), slot, my_groups, 32 * RW,
                            e, ng))
            return;
    } else {
        if (threadIdx.x < G) slot[threadIdx.x] = threadIdx.x < ng ? a.perm[p0 + threadIdx.x] : 0;
        __syncthreads();
    }

    // stage the G activation rows once: 32 int8 as two 16-byte chunks and
    // aux = {d_a, level0 * sum q (int bits: the dot starts from its negative)}
    // for Q4_0 / Q5_0, {d_a, d_a * sum q} for the types with an offset term
    if constexpr (FUSED) {
        // the one-launch decode step quantizes the slots' fp16 rows itself with
        // the quantizer's arithmetic and lane layout (eight lanes per block,
        // four values each), so the same codes; d rounded to fp16 as stored
        const uint32_t sub = lane & 7u, gmask = 0xFFu << (lane & 24u);
        const int32_t n_items = G * nb;
        // each warp takes 4 blocks at a time (one per 8 lanes), FU of them in a
        // batch whose loads are all issued before any is used
        constexpr int FU = 4;
        for (int32_t base = static_cast<int32_t>(warp) * 4 * FU;
             base < n_items && static_cast<int32_t>(warp) < n_compute; base += n_compute * 4 * FU) {
            uint2 raw[FU];
#pragma unroll
            for (int u = 0; u < FU; ++u) {
                const int32_t i = base + 4 * u + static_cast<int32_t>(lane >> 3);
                const int32_t g = i / nb, b = i - g * nb;
                raw[u] = make_uint2(0, 0);
                if (i < n_items && g < ng) {
                    const int64_t tok = slot[g] / a.top_k;
                    raw[u] = __ldg(reinterpret_cast<const uint2*>(a.x + (tok * nb + b) * QK) + sub);
                }
            }
#pragma unroll
            for (int u = 0; u < FU; ++u) {
                const int32_t i = base + 4 * u + static_cast<int32_t>(lane >> 3);
                const int32_t g = i / nb, b = i - g * nb;
                const bool live = i < n_items && g < ng;
                const __half2 h01 = *reinterpret_cast<const __half2*>(&raw[u].x);
                const __half2 h23 = *reinterpret_cast<const __half2*>(&raw[u].y);
                const float v[4] = {__low2float(h01), __high2float(h01), __low2float(h23), __high2float(h23)};
                float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, o));
                const float d32 = __fdiv_rn(amax, 127.0f);
                int q[4];
                q8_codes<4>(v, amax, d32, q);
                uint32_t packed = 0;
                int sm = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sm += q[j];
                    packed |= (static_cast<uint32_t>(q[j]) & 0xFFu) << (8 * j);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) sm += __shfl_xor_sync(gmask, sm, o);
                if (i < n_items) {
                    reinterpret_cast<uint32_t*>(qa)[(static_cast<size_t>(g) * nb + b) * 8 + sub] = packed;
                    if (sub == 0) {
                        const float d = live ? __half2float(__float2half_rn(d32)) : 0.0f;
                        const float y = OFFSET ? d * small_int_to_float(sm) : __int_as_float(LEVEL0 * sm);
                        aux[static_cast<size_t>(g) * nb + b] = make_float2(d, y);
                    }
                }
            }
        }
    }
    for (int32_t i = threadIdx.x; i < G * nb && !FUSED; i += blockDim.x) {
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
        const float y = OFFSET ? d * small_int_to_float(sm) : __int_as_float(LEVEL0 * sm);
        aux[static_cast<size_t>(g) * nb + b] = make_float2(d, y);
    }
    if constexpr (FUSED) {
        if (static_cast<int32_t>(warp) < n_compute) named_bar_sync(1, static_cast<uint32_t>(n_compute) * 32u);
    } else {
        __syncthreads();
    }

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
                // 16-bit elements: x counts 2-byte units
                tma_load_2d(ring + static_cast<size_t>(s) * stage_bytes, &wmap, ks * (BX::BYTES / 2),
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
                                                               (r * 32 + lane) * PITCH);
            auto part = [&](auto P) {
                using PT = RowPart<WT, decltype(P)::value>;
                uint32_t wv[PT::NW];
#pragma unroll
                for (int c = 0; c < PT::C1 - PT::C0; ++c) {
                    const uint4 v = rowp[PT::C0 + c];
                    wv[4 * c] = v.x;
                    wv[4 * c + 1] = v.y;
                    wv[4 * c + 2] = v.z;
                    wv[4 * c + 3] = v.w;
                }
#pragma unroll
                for (int j = PT::J0; j < PT::J1; ++j) {
                    float dw, mw;
                    int lo[4], hi[4];
                    decode_win<WT>(wv, BX::KQ ? 0 : j * BX::WB - 16 * PT::C0, j, dw, mw, lo, hi);
                    const int32_t b = ks * 8 + j;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const uint4 A0 = qa[(static_cast<size_t>(g) * nb + b) * 2];
                        const uint4 A1 = qa[(static_cast<size_t>(g) * nb + b) * 2 + 1];
                        const float2 x = aux[static_cast<size_t>(g) * nb + b];
                        int dot = LEVEL0 ? -__float_as_int(x.y) : 0;
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
                            if constexpr (OFFSET) acc[g] = fmaf(MSIGN * mw, x.y, acc[g]);
                        }
                    }
                }
            };
            part(std::integral_constant<int, 0>{});
            if constexpr (BX::NPART > 1) part(std::integral_constant<int, 1>{});
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

// CTAs of a kernel that fit on one SM at once (cached; moe_gemv.cu).
int resident_ctas(const void* kernel, int threads, size_t smem);

template <int WT, int G, bool DUMP, bool FUSED = false>
static int launch_gemv_rows(const GemvPlan& plan, const CUtensorMap& wmap, const GemvArgs& a, cudaStream_t s) {
    const void* kernel = reinterpret_cast<const void*>(moe_gemv_rows_kernel<WT, G, DUMP, FUSED>);
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
    moe_gemv_rows_kernel<WT, G, DUMP, FUSED><<<grid, block, plan.smem, s>>>(wmap, a);
    return check_launch(DUMP ? "moe_gemv_rows_kernel<dump>" : FUSED ? "moe_gemv_rows_kernel<fused>" : "moe_gemv_rows_kernel",
                        grid, block, plan.smem);
}

template <int WT>
static int launch_gemv_rows_type(const GemvPlan& plan, const CUtensorMap& wmap, const GemvArgs& a, cudaStream_t s) {
    switch (plan.group) {
        case 1: return launch_gemv_rows<WT, 1, false>(plan, wmap, a, s);
        case 2: return launch_gemv_rows<WT, 2, false>(plan, wmap, a, s);
        case 4: return launch_gemv_rows<WT, 4, false>(plan, wmap, a, s);
        default: return launch_gemv_rows<WT, 8, false>(plan, wmap, a, s);
    }
}

// The row-per-lane kernel for a weight type other than Q4_0 (moe_gemv_gguf.cu).
int launch_gemv_rows_gguf(int wtype, const GemvPlan& plan, const CUtensorMap& wmap, const GemvArgs& a,
                          cudaStream_t s);

// Q4_0 and Q4_K tiles of nt groups of 8 slots on mma.sync (moe_gemv_mma.cu): shared
// memory of a CTA of row_warps warps of 16 rows with a ring of `stages` boxes,
// and the launch (dump: block dots); wmap's box is 16 * row_warps rows high,
// wmap16's 16 rows (for the short row blocks at the ends of a CTA's range).
size_t gemv_mma_smem(int nb, int nt, int row_warps, int stages, int wtype);
int launch_gemv_mma(const GemvPlan& plan, const CUtensorMap& wmap, const CUtensorMap& wmap16, const GemvArgs& a,
                    bool dump, int wtype, cudaStream_t s);

}  // namespace ft
