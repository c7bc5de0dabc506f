// Expert-grouped GEMM path of the routed Q4_0 x Q8_1 expert matmul on the
// sm_103a tensor cores (tcgen05 MMA into TMEM).
//
// The grouped form follows the expert_offsets layout of nvfp4-megamoe-kernel
// CURRENT_BUG.md (Bug 4: offsets with a leading 0; Bug 2: position -> expert
// by searchsorted(right=True)), but without the fixed-layout padding of
// "Key Architecture: Fixed-Layout Padding": tiles are cut from the router's
// padding-free permutation, so no expert is padded to a fixed row count.
//
// gather_act_kernel writes, in router order, each routed slot's Q8_1
// activation row as an fp16 row (exact: q in [-127, 127]) plus its fp16 block
// scales, so that the GEMM's activation operand is a plain 2-D array the TMA
// can load straight into the MMA's swizzled layout.
//
// moe_gemm_tc_kernel: tile = (expert e, up to BN routed slots of e, 128
// weight rows of e).  A persistent grid (one CTA per SM) walks the tile list,
// whose length is read on the device from the router's tile prefix; empty
// experts own no tile.  Per CTA, warp-specialized:
//   producer: per stage of 8 Q4_0 blocks (K = 256) a 2-D TMA load of the
//            128 x 144-byte weight box and of the BN x 8 activation-scale
//            box; per pair of blocks a 2-D TMA load of the BN x 64 fp16
//            activation box with 128-byte swizzle (the MMA's B layout);
//   unpack (4 warps): Q4_0 nibbles -> fp16 (q - 8), exact, into the K-major
//            128-byte-swizzled A layout (each thread one weight row, 16-byte
//            shared loads that are bank-conflict free because a 144-byte row
//            is an odd number of 16-byte chunks), plus the fp32 block scales
//            d_w (per row) and d_a (per slot) for the drain;
//   MMA:     per 32-value block, two tcgen05.mma kind::f16 (K = 16)
//            M = 128, N = BN into its own TMEM accumulator (4 buffers);
//   drain:   each warp owns 16 TMEM lanes x min(BN, 64) columns and loads
//            them with the 16x256b shape, so a thread holds 2 rows x 16
//            columns and one shared load of scales serves four different
//            column pairs of the warp; the block's exact integer dot (fp32
//            holds it exactly: |dot| <= 32512) is scaled as
//            acc += d_w * (dot * d_a) with one packed fp32x2 multiply and one
//            packed fp32x2 FMA per column pair; at the end of the tile the
//            outputs go to out[slot][row].
//
// Why fp16 operands: every operand value is a small integer (q_w - 8 in
// [-8, 7], q_a in [-127, 127]), exact in fp16, and a 32-term block dot is
// exact in the fp32 accumulator, so the per-block integer dot is bit-exact
// while running at the fp16 tensor rate.  The scales change every 32 values
// along K, so each block needs its own accumulator and a drain; the drain's
// two fp32 operations per (row, slot, block) set this kernel's ceiling.
#include "gemm_common.cuh"
#include "gemv_blocks.cuh"   // kquant_scale_min
#include "q8_1_math.cuh"

namespace ft {

// Compile-time configuration for a slot-tile width BN (32 for decode-sized
// batches, 128 for prefill) and the weight type: Q4_0 (KQ_ false) or Q4_K
// (KQ_ true: a raw stage is one 144-byte super-block per row, the same box as
// eight Q4_0 blocks; each block also carries a min d_min m_j per row and the
// activation block's d_a sum(q_a) per slot, one more fp32 term in the drain).
template <int BN_, bool KQ_ = false>
struct Gemm {
    static constexpr bool KQ = KQ_;
    static constexpr int BN = BN_;                      // slots per tile
    static constexpr int BM = kGemmBM;                  // weight rows per tile
    static constexpr int KB = 8;                        // Q4_0 blocks per raw stage (K = 256)
    static constexpr int RAW_STAGES = 2;
    static constexpr int OP_SLOTS = 4;                  // operand slots of 2 blocks (K = 64, one 128-B swizzle atom)
    static constexpr int NACC = 4;                      // TMEM accumulators, BN columns each
    // Narrow tiles hand accumulators between the MMA thread and the drain per
    // 2-block unit (a pair of accumulators, one commit, one release), which
    // halves the hand-offs when the drain's work per block is small; wide
    // tiles hand them off per block, which keeps the drain fed more evenly.
    static constexpr bool PAIRED = BN_ <= 32;
    static constexpr int NBAR_ACC = PAIRED ? NACC / 2 : NACC;   // accumulator barriers
    static constexpr int NSC = 8;                       // scale ring depth (blocks)
    static constexpr int W_RAW_BYTES = BM * KB * Q4_0_BYTES;   // 18432
    static constexpr int DA_RAW_BYTES = BN * KB * 2;           // [slot][8] fp16 activation scales
    static constexpr int SA_RAW_BYTES = KQ ? BN * KB * 4 : 0;   // [slot][8] fp32 d_a sum(q_a) (Q4_K)
    static constexpr int RAW_STAGE_BYTES = W_RAW_BYTES + DA_RAW_BYTES + SA_RAW_BYTES;
    static constexpr int OPA_BYTES = BM * 128;
    static constexpr int OPB_BYTES = BN * 128;
    static constexpr int OP_SLOT_BYTES = OPA_BYTES + OPB_BYTES;
    // drain: each warp owns 16 TMEM lanes x CW columns (CW / 32 loads of 16 registers)
    static constexpr int CW = BN < 64 ? BN : 64;
    static constexpr int N_DRAIN_WARPS = 8 * (BN / CW);
    // Scales of one block, fp32: d_w[BM], then d_a in the drain's read order:
    // for each CW-column group and column-pair index q (0..3) a group of CW/4
    // floats {d_a[CW g + 8 i + 2 q + e] : i < CW/8, e < 2} at a pitch of
    // CW/4 + 4 floats, so that the four 16-byte groups a warp's quads load at
    // once fall in four different bank groups.
    static constexpr int DA_QPITCH = CW / 4 + 4;
    static constexpr int DA_FLOATS = (BN / CW) * 4 * DA_QPITCH;
    // Q4_K adds the mins d_min m_j [BM] and the slots' d_a sum(q_a) (d_a's layout)
    static constexpr int SC_BYTES = (BM * 4 + DA_FLOATS * 4) * (KQ ? 2 : 1);
    static constexpr int N_UNPACK_WARPS = 4;
    static constexpr int UNPACK_THREADS = N_UNPACK_WARPS * 32;  // one weight row per thread
    static constexpr int WARP_PRODUCER = N_DRAIN_WARPS + N_UNPACK_WARPS, WARP_MMA = WARP_PRODUCER + 1;
    static constexpr int THREADS = (WARP_MMA + 1) * 32;
    static constexpr int N_EPI_WARPS = 2;                        // fused layer 1: quantizing warps after the MMA warp
    static constexpr int THREADS_FUSED = THREADS + N_EPI_WARPS * 32;
    static constexpr uint32_t TMEM_COLS = NACC * BN;
    // smem offsets from a 1024-aligned base
    static constexpr int OFF_OP = 0;
    static constexpr int OFF_RAW = OFF_OP + OP_SLOTS * OP_SLOT_BYTES;
    static constexpr int OFF_SC = OFF_RAW + RAW_STAGES * RAW_STAGE_BYTES;
    // Fused layer-1 epilogue: the up rows' sums as float2 [64 rows][BN / 2 + 4]
    // (the 4 extra float2 per row keep a warp's float2 stores conflict-free),
    // then, in the same bytes, act(gate) * up as float [BN slots][64 + 4]
    // (rows 16-byte aligned, one 128-byte run per quarter-warp read)
    static constexpr int EPI_P2 = BN / 2 + 4;
    static constexpr int EPI_AP = 64 + 4;
    static constexpr int EPI_BYTES = KQ ? 0 : 64 * EPI_P2 * 8 > BN * EPI_AP * 4 ? 64 * EPI_P2 * 8 : BN * EPI_AP * 4;
    static constexpr int OFF_EPI = OFF_SC + NSC * SC_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int N_BARS = 2 * RAW_STAGES + 2 * OP_SLOTS + 2 * NBAR_ACC + NSC + 4;
    static constexpr int OFF_TMEM = OFF_BAR + N_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM + 16 + 1024;    // + alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(OP_SLOT_BYTES % 1024 == 0 && OPA_BYTES % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
    static_assert(BN % 32 == 0 && BN <= 256, "tile width");
};

// Byte offset of 16-byte chunk c of row r in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) {
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

// Four int8 bytes -> two fp16x2 words holding the same integers.
__device__ __forceinline__ void i8x4_to_h2(uint32_t v, uint32_t& lo, uint32_t& hi) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    const uint32_t u = v ^ 0x80808080u;
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

// Fused layer-1 epilogue.  A tile's 128 rows are 64 gate rows i0 .. i0+63
// (TMEM lanes 0..63) and the matching up rows (lanes 64..127), so gate row m
// and up row m sit in the same thread position of drain warps w and w + 2.
// At the end of a tile (tc counts the CTA's earlier tiles: the phase of the
// epilogue barriers) the drain warps
//   1. (up warps) store their sums, float2 [row][slot];
//   2. (gate warps) read the up value of each of their sums and replace the
//      sum g by act(g) * up; once every gate warp has read, they store those
//      values slot-major ([slot][row]) in the same bytes;
// and go on with the next tile, while two epilogue warps
//   3. quantize (slot, 32-row block) units, eight lanes per unit with four
//      values each - the lane layout and arithmetic of the separate
//      activation/requantize step - and write the Q8_1 block of columns
//      i0 + 32 j .. +31 of the slot's act_mid row.
// The up warps wait before step 1 until step 3 of the previous tile is done
// with the bytes.  Every wait is bounded; false: one gave up.
template <int BN>
__device__ __forceinline__ bool fused_act_drain(float2 (&acc)[2][Gemm<BN>::CW / 8], const GemmArgs& a,
                                                uint8_t* epi, uint64_t* ebar, uint32_t tc, uint32_t warp,
                                                uint32_t lane) {
    using C = Gemm<BN>;
    constexpr int CW = C::CW, P2 = C::EPI_P2, AP = C::EPI_AP;
    uint64_t* up_ready = ebar;        // step 1 done (up warps)
    uint64_t* up_read = ebar + 1;     // up values read (gate warps)
    uint64_t* a_ready = ebar + 2;     // step 2 done (gate warps)
    uint64_t* a_done = ebar + 3;      // step 3 done (epilogue warps)
    const uint32_t ph = tc & 1u;
    const uint32_t lane0 = (warp & 3u) * 32u + ((warp >> 2) & 1u) * 16u;
    const uint32_t col0 = (warp >> 3) * static_cast<uint32_t>(CW);
    const uint32_t q = lane & 3u, r0 = lane0 + (lane >> 2);
    float2* ub = reinterpret_cast<float2*>(epi);
    float* ab = reinterpret_cast<float*>(epi);
    if ((warp & 3u) >= 2u) {
        if (!mbar_wait_warp(a_done, ph ^ 1u, a.err)) return false;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
#pragma unroll
            for (int i = 0; i < CW / 8; ++i) ub[(r0 - 64 + 8 * hr) * P2 + (col0 >> 1) + 4 * i + q] = acc[hr][i];
        __syncwarp();
        if (lane == 0) mbar_arrive(up_ready);
        return true;
    }
    if (!mbar_wait_warp(up_ready, ph, a.err)) return false;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int i = 0; i < CW / 8; ++i) {
            const float2 u = ub[(r0 + 8 * hr) * P2 + (col0 >> 1) + 4 * i + q];
            acc[hr][i].x = act_mul(acc[hr][i].x, u.x, a.act_kind);
            acc[hr][i].y = act_mul(acc[hr][i].y, u.y, a.act_kind);
        }
    __syncwarp();
    if (lane == 0) mbar_arrive(up_read);
    if (!mbar_wait_warp(up_read, ph, a.err)) return false;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int i = 0; i < CW / 8; ++i) {
            const uint32_t n = col0 + 8 * i + 2 * q;
            ab[n * AP + r0 + 8 * hr] = acc[hr][i].x;
            ab[(n + 1) * AP + r0 + 8 * hr] = acc[hr][i].y;
        }
    __syncwarp();
    if (lane == 0) mbar_arrive(a_ready);
    return true;
}

// Step 3 for one tile, by epilogue warp ew (0 or 1).
template <int BN>
__device__ __forceinline__ bool fused_act_quantize(const GemmArgs& a, const TileInfo& ti, const uint8_t* epi,
                                                   uint64_t* ebar, uint32_t tc, uint32_t ew, uint32_t lane) {
    using C = Gemm<BN>;
    constexpr int AP = C::EPI_AP;
    const float* ab = reinterpret_cast<const float*>(epi);
    if (!mbar_wait_warp(ebar + 2, tc & 1u, a.err)) return false;
    const uint32_t grp = lane >> 3, sub = lane & 7u;
    const uint32_t gmask = 0xFFu << (lane & 24u);
    const int64_t i0 = ti.m0 / 2, nbi = a.n_inter / QK;
#pragma unroll 1
    for (int it = 0; it < 2 * BN / (4 * C::N_EPI_WARPS); ++it) {
        const uint32_t u = (static_cast<uint32_t>(it) * C::N_EPI_WARPS + ew) * 4u + grp;
        const uint32_t n = u >> 1, j = u & 1u;
        const float4 x = *reinterpret_cast<const float4*>(ab + n * AP + 32 * j + 4 * sub);
        const float v[4] = {x.x, x.y, x.z, x.w};
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, o));
        const float d = __fdiv_rn(amax, 127.0f);
        int qv[4];
        q8_codes<4>(v, amax, d, qv);
        uint32_t packed = 0;
        int sum = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sum += qv[k];
            packed |= (static_cast<uint32_t>(qv[k]) & 0xFFu) << (8 * k);
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(gmask, sum, o);
        if (static_cast<int32_t>(n) < ti.nvalid && i0 + 32 * static_cast<int64_t>(j) < a.n_inter) {
            const int64_t slot = a.perm[ti.p0 + n];
            uint8_t* ob = a.act_mid + (slot * nbi + i0 / QK + j) * Q8_1_BYTES;
            *reinterpret_cast<uint32_t*>(ob + 4 + 4 * sub) = packed;
            if (sub == 0) *reinterpret_cast<uint32_t*>(ob) = q8_header(d, sum);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(ebar + 3);
    return true;
}

template <int BN, bool DUMP, bool FUSE, bool KQ>
__global__ void __launch_bounds__(FUSE ? Gemm<BN>::THREADS_FUSED : Gemm<BN>::THREADS, 1)
    moe_gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                       const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap amap,
                       const GemmArgs a) {
    using C = Gemm<BN, KQ>;
    static_assert(!(KQ && (DUMP || FUSE)), "Q4_K takes the plain matmul only");
    constexpr int SA_RAW_BYTES = C::SA_RAW_BYTES, DA_FLOATS = C::DA_FLOATS;
    constexpr int BM = C::BM, KB = C::KB, RAW_STAGES = C::RAW_STAGES, OP_SLOTS = C::OP_SLOTS, NACC = C::NACC;
    constexpr int NBAR_ACC = C::NBAR_ACC;
    constexpr bool PAIRED = C::PAIRED;
    constexpr int NSC = C::NSC, W_RAW_BYTES = C::W_RAW_BYTES, DA_RAW_BYTES = C::DA_RAW_BYTES;
    constexpr int RAW_STAGE_BYTES = C::RAW_STAGE_BYTES, OPA_BYTES = C::OPA_BYTES, OPB_BYTES = C::OPB_BYTES;
    constexpr int OP_SLOT_BYTES = C::OP_SLOT_BYTES, CW = C::CW, N_DRAIN_WARPS = C::N_DRAIN_WARPS;
    constexpr int DA_QPITCH = C::DA_QPITCH, SC_BYTES = C::SC_BYTES, N_UNPACK_WARPS = C::N_UNPACK_WARPS;
    constexpr int UNPACK_THREADS = C::UNPACK_THREADS, WARP_PRODUCER = C::WARP_PRODUCER, WARP_MMA = C::WARP_MMA;
    constexpr uint32_t TMEM_COLS = C::TMEM_COLS;
    constexpr int OFF_OP = C::OFF_OP, OFF_RAW = C::OFF_RAW, OFF_SC = C::OFF_SC, OFF_BAR = C::OFF_BAR;
    constexpr int OFF_TMEM = C::OFF_TMEM;
    static_assert(!(DUMP && FUSE), "block dots come from the plain matmul");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + RAW_STAGES;
    uint64_t* op_full = raw_empty + RAW_STAGES;
    uint64_t* op_empty = op_full + OP_SLOTS;
    uint64_t* acc_full = op_empty + OP_SLOTS;
    uint64_t* acc_empty = acc_full + NBAR_ACC;
    uint64_t* sc_empty = acc_empty + NBAR_ACC;
    uint64_t* epi_bar = sc_empty + NSC;          // fused epilogue: up_ready, up_read, a_ready, a_done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);

    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const int32_t nb = a.nb;
    const int32_t n_stages = nb / KB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RAW_STAGES; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], UNPACK_THREADS);
        }
        for (int i = 0; i < OP_SLOTS; ++i) {
            mbar_init(&op_full[i], UNPACK_THREADS + 1);   // unpack threads + the producer's TMA
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < NBAR_ACC; ++i) {
            // an accumulator (pair) is ready once its MMAs completed (the commit)
            // and the MMA thread has arrived after issuing them.  That second,
            // explicit arrival releases what the MMA thread acquired from the
            // operand barrier - the unpack threads' scale writes for the blocks -
            // and, being made only after acc_empty was observed, can never fall
            // into an earlier phase of the barrier.
            mbar_init(&acc_full[i], 2);
            mbar_init(&acc_empty[i], N_DRAIN_WARPS);
        }
        for (int i = 0; i < NSC; ++i) mbar_init(&sc_empty[i], N_DRAIN_WARPS);
        for (int i = 0; i < 3; ++i) mbar_init(&epi_bar[i], N_DRAIN_WARPS / 2);
        mbar_init(&epi_bar[3], C::N_EPI_WARPS);
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == WARP_PRODUCER && lane == 0) {
        prefetch_tmap(&wmap);
        prefetch_tmap(&xmap);
        prefetch_tmap(&smap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int64_t total = static_cast<int64_t>(a.tiles[a.n_experts]) * a.row_tiles;

    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ producer
        uint32_t it = 0, ou = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
            const TileInfo ti = decode_tile<BN>(a, w);
            // fused layer 1: gate rows i0 .. i0+63 and up rows n_inter + i0 .. (i0 = m0 / 2)
            const int64_t row0 = static_cast<int64_t>(ti.e) * a.nrows + (FUSE ? ti.m0 / 2 : ti.m0);
            const int32_t wy = static_cast<int32_t>(row0);
            const int32_t wy_up = static_cast<int32_t>(FUSE ? row0 + a.n_inter : 0);
            const int32_t py = static_cast<int32_t>(ti.p0);
            for (int32_t ks = 0; ks < n_stages && ok; ++ks, ++it) {
                const uint32_t s = it % RAW_STAGES;
                if (!mbar_wait_warp(&raw_empty[s], ((it / RAW_STAGES) & 1u) ^ 1u, a.err)) { ok = false; break; }
                uint8_t* wraw = smem + OFF_RAW + s * RAW_STAGE_BYTES;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&raw_full[s], W_RAW_BYTES + DA_RAW_BYTES + SA_RAW_BYTES);
                    tma_load_2d(wraw, &wmap, ks * KB * Q4_0_BYTES, wy, &raw_full[s]);
                    if constexpr (KQ)   // the slots' d_a sum(q_a) of the stage's 8 blocks
                        tma_load_2d(wraw + W_RAW_BYTES + DA_RAW_BYTES, &amap, ks * KB, py, &raw_full[s]);
                    if constexpr (FUSE)
                        tma_load_2d(wraw + (BM / 2) * KB * Q4_0_BYTES, &wmap, ks * KB * Q4_0_BYTES, wy_up,
                                    &raw_full[s]);
                    tma_load_2d(wraw + W_RAW_BYTES, &smap, ks * KB, py, &raw_full[s]);
                }
                for (int j = 0; j < KB / 2; ++j, ++ou) {
                    const uint32_t os = ou % OP_SLOTS;
                    if (!mbar_wait_warp(&op_empty[os], ((ou / OP_SLOTS) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    if (lane == 0) {
                        uint8_t* opb = smem + OFF_OP + os * OP_SLOT_BYTES + OPA_BYTES;
                        mbar_arrive_expect_tx(&op_full[os], OPB_BYTES);
                        tma_load_2d(opb, &xmap, (ks * (KB / 2) + j) * 64, py, &op_full[os]);
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp >= N_DRAIN_WARPS && warp < N_DRAIN_WARPS + N_UNPACK_WARPS) {
        // -------------------------------------------------------------- unpack
        constexpr int RPT = BM / UNPACK_THREADS;                  // rows (and slots) per thread
        const uint32_t u0 = threadIdx.x - N_DRAIN_WARPS * 32;     // rows u0, u0 + UNPACK_THREADS, ...
        uint32_t it = 0, ou = 0, bc = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
            for (int32_t ks = 0; ks < n_stages && ok; ++ks, ++it) {
                const uint32_t s = it % RAW_STAGES;
                if (!mbar_wait(&raw_full[s], (it / RAW_STAGES) & 1u, a.err)) { ok = false; break; }
                const uint8_t* wraw = smem + OFF_RAW + s * RAW_STAGE_BYTES;
                // each slot's 8 activation scales of the stage (rows past the
                // tile's routed slots hold the next expert's or zero-filled data
                // and only reach output columns that are never stored)
                uint32_t dav[RPT][4];                                     // 8 fp16 scales, packed in pairs
#pragma unroll
                for (int rr = 0; rr < RPT; ++rr) {
                    const uint32_t us = u0 + rr * UNPACK_THREADS;
                    uint4 x = make_uint4(0, 0, 0, 0);
                    if (us < static_cast<uint32_t>(BN))
                        x = *reinterpret_cast<const uint4*>(wraw + W_RAW_BYTES + us * (KB * 2));
                    dav[rr][0] = x.x;
                    dav[rr][1] = x.y;
                    dav[rr][2] = x.z;
                    dav[rr][3] = x.w;
                }
#pragma unroll
                for (int j = 0; j < KB / 2; ++j, ++ou) {
                    const uint32_t os = ou % OP_SLOTS;
                    if (!mbar_wait(&op_empty[os], ((ou / OP_SLOTS) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    uint8_t* opa = smem + OFF_OP + os * OP_SLOT_BYTES;
                    if constexpr (KQ) {
                        // Q4_K: the row's stage is one super-block: chunk 0 = fp16 d, fp16
                        // d_min, 12 bytes of 6-bit scale/min pairs; sub-blocks 2j and 2j+1 are
                        // the low and high nibbles of the 32 bytes in chunks 1 + 2j, 2 + 2j
                        // (levels 0..15, no offset); per block d sc_j, d_min m_j per row and
                        // d_a, d_a sum(q_a) per slot go to the scale ring
#pragma unroll
                        for (int h = 0; h < 2; ++h, ++bc) {
                            const uint32_t sc = bc % NSC;
                            if (!mbar_wait(&sc_empty[sc], ((bc / NSC) & 1u) ^ 1u, a.err)) { ok = false; break; }
                            float* dws = reinterpret_cast<float*>(smem + OFF_SC + sc * SC_BYTES);
                            float* das = dws + BM;
                            float* mws = das + DA_FLOATS;
                            float* sas = mws + BM;
#pragma unroll
                            for (int rr = 0; rr < RPT; ++rr) {
                                const uint32_t u = u0 + rr * UNPACK_THREADS;
                                const uint4* wrow = reinterpret_cast<const uint4*>(wraw + u * (KB * Q4_0_BYTES));
                                const uint4 hd = wrow[0], qc0 = wrow[1 + 2 * j], qc1 = wrow[2 + 2 * j];
                                const uint32_t sc12[3] = {hd.y, hd.z, hd.w};
                                int scv, mnv;
                                kquant_scale_min(sc12, 2 * j + h, scv, mnv);
                                dws[u] = __half2float(__ushort_as_half(static_cast<unsigned short>(hd.x & 0xFFFFu))) *
                                         static_cast<float>(scv);
                                mws[u] = __half2float(__ushort_as_half(static_cast<unsigned short>(hd.x >> 16))) *
                                         static_cast<float>(mnv);
                                if (u < static_cast<uint32_t>(BN)) {
                                    const uint32_t pair = dav[rr][j];         // d_a of blocks 2j, 2j+1
                                    const unsigned short hb =
                                        static_cast<unsigned short>(h ? (pair >> 16) : (pair & 0xFFFFu));
                                    das[da_index<CW>(u)] = __half2float(__ushort_as_half(hb));
                                    sas[da_index<CW>(u)] = *reinterpret_cast<const float*>(
                                        wraw + W_RAW_BYTES + DA_RAW_BYTES + u * (KB * 4) + (2 * j + h) * 4);
                                }
                                const uint32_t w8[8] = {qc0.x, qc0.y, qc0.z, qc0.w, qc1.x, qc1.y, qc1.z, qc1.w};
                                // 16-byte chunk c of the block holds values 8c..8c+7: bytes 8c..8c+7
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    uint32_t h0, h1, h2, h3;
                                    nib4_to_h2<0>((w8[2 * c] >> (4 * h)) & 0x0F0F0F0Fu, h0, h1);
                                    nib4_to_h2<0>((w8[2 * c + 1] >> (4 * h)) & 0x0F0F0F0Fu, h2, h3);
                                    *reinterpret_cast<uint4*>(opa + sw128_off(u, 4 * h + c)) = make_uint4(h0, h1, h2, h3);
                                }
                            }
                        }
                        if (!ok) break;
                        fence_proxy_async_smem();
                        mbar_arrive(&op_full[os]);
                        continue;
                    }
                    // the unit's 36 bytes of a row start at byte 36j = 16 * (2j) + 4j: words
                    // j .. j+8 of a 3-chunk window starting at chunk 2j (9 chunks per row, so
                    // 8 consecutive rows hit 8 different 16-byte bank groups)
                    uint32_t wv[RPT][12];
#pragma unroll
                    for (int rr = 0; rr < RPT; ++rr) {
                        const uint4* wrow =
                            reinterpret_cast<const uint4*>(wraw + (u0 + rr * UNPACK_THREADS) * (KB * Q4_0_BYTES));
#pragma unroll
                        for (int c = 0; c < 3; ++c) {
                            const uint4 q = wrow[2 * j + c];
                            wv[rr][4 * c + 0] = q.x;
                            wv[rr][4 * c + 1] = q.y;
                            wv[rr][4 * c + 2] = q.z;
                            wv[rr][4 * c + 3] = q.w;
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h, ++bc) {
                        const uint32_t sc = bc % NSC;
                        if (!mbar_wait(&sc_empty[sc], ((bc / NSC) & 1u) ^ 1u, a.err)) { ok = false; break; }
                        float* dws = reinterpret_cast<float*>(smem + OFF_SC + sc * SC_BYTES);
                        float* das = dws + BM;
#pragma unroll
                        for (int rr = 0; rr < RPT; ++rr) {
                            const uint32_t u = u0 + rr * UNPACK_THREADS;
                            uint32_t q[4], dbits;
                            if (h == 0) {   // bytes 4j .. 4j+17 of the window: 2-byte aligned nibbles
                                dbits = wv[rr][j] & 0xFFFFu;
#pragma unroll
                                for (int i = 0; i < 4; ++i) q[i] = __byte_perm(wv[rr][j + i], wv[rr][j + i + 1], 0x5432u);
                            } else {        // bytes 4j+18 .. 4j+35: word-aligned nibbles
                                dbits = wv[rr][j + 4] >> 16;
#pragma unroll
                                for (int i = 0; i < 4; ++i) q[i] = wv[rr][j + 5 + i];
                            }
                            dws[u] = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
                            {
                                const uint32_t pair = dav[rr][j];             // scales of blocks 2j, 2j+1
                                const unsigned short hb = static_cast<unsigned short>(h ? (pair >> 16) : (pair & 0xFFFFu));
                                if (u < static_cast<uint32_t>(BN)) das[da_index<CW>(u)] = __half2float(__ushort_as_half(hb));
                            }
                            // 16-byte chunk c holds values 8c..8c+7: the low nibbles of q[0..3] are
                            // values 0..15, the high nibbles values 16..31
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t qa = q[2 * (c & 1)], qb = q[2 * (c & 1) + 1];
                                const uint32_t sh = (c >> 1) * 4u;
                                uint32_t h0, h1, h2, h3;
                                nib4_to_h2((qa >> sh) & 0x0F0F0F0Fu, h0, h1);
                                nib4_to_h2((qb >> sh) & 0x0F0F0F0Fu, h2, h3);
                                *reinterpret_cast<uint4*>(opa + sw128_off(u, 4 * h + c)) = make_uint4(h0, h1, h2, h3);
                            }
                        }
                    }
                    if (!ok) break;
                    fence_proxy_async_smem();
                    mbar_arrive(&op_full[os]);
                }
                if (!ok) break;
                mbar_arrive(&raw_empty[s]);
            }
        }
    } else if (warp == WARP_MMA) {
        // ----------------------------------------------------------------- MMA
        if (PAIRED && lane == 0) {
            // one accumulator pair per 2-block unit
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            uint32_t ou = 0;
            bool ok = true;
            for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
                for (int32_t ks = 0; ks < n_stages && ok; ++ks) {
                    for (int j = 0; j < KB / 2; ++j, ++ou) {
                        const uint32_t os = ou % OP_SLOTS;
                        if (!mbar_wait(&op_full[os], (ou / OP_SLOTS) & 1u, a.err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t abase = smem_u32(smem + OFF_OP + os * OP_SLOT_BYTES);
                        const uint32_t bbase = abase + OPA_BYTES;
                        const uint32_t pa = ou % NBAR_ACC;
                        if (!mbar_wait(&acc_empty[pa], ((ou / NBAR_ACC) & 1u) ^ 1u, a.err)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t d_tmem = tmem_base + (2 * pa + h) * BN;
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const uint32_t koff = h * 64 + k * 32;
                                tc_mma_f16(d_tmem, smem_desc_sw128(abase + koff), smem_desc_sw128(bbase + koff), idesc,
                                           k);
                            }
                        }
                        tc_commit(&acc_full[pa]);
                        mbar_arrive(&acc_full[pa]);
                        tc_commit(&op_empty[os]);
                    }
                }
            }
        }
        if (!PAIRED && lane == 0) {
            // one accumulator per block
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            uint32_t ou = 0, bc = 0;
            bool ok = true;
            for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
                for (int32_t ks = 0; ks < n_stages && ok; ++ks) {
                    for (int j = 0; j < KB / 2; ++j, ++ou) {
                        const uint32_t os = ou % OP_SLOTS;
                        if (!mbar_wait(&op_full[os], (ou / OP_SLOTS) & 1u, a.err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t abase = smem_u32(smem + OFF_OP + os * OP_SLOT_BYTES);
                        const uint32_t bbase = abase + OPA_BYTES;
                        for (int h = 0; h < 2; ++h, ++bc) {
                            const uint32_t ab = bc % NACC;
                            if (!mbar_wait(&acc_empty[ab], ((bc / NACC) & 1u) ^ 1u, a.err)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t d_tmem = tmem_base + ab * BN;
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const uint32_t koff = h * 64 + k * 32;
                                tc_mma_f16(d_tmem, smem_desc_sw128(abase + koff), smem_desc_sw128(bbase + koff), idesc,
                                           k);
                            }
                            tc_commit(&acc_full[ab]);
                            mbar_arrive(&acc_full[ab]);
                        }
                        tc_commit(&op_empty[os]);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp > WARP_MMA) {
        // ---------------------------------------- fused layer 1: quantizing warps
        if constexpr (FUSE) {
            uint32_t tc = 0;
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x, ++tc) {
                const TileInfo ti = decode_tile<BN>(a, w);
                if (!fused_act_quantize<BN>(a, ti, smem + C::OFF_EPI, epi_bar, tc, warp - WARP_MMA - 1, lane)) break;
            }
        }
    } else {
        // --------------------------------------------------------------- drain
        // warp w: TMEM lanes 32 (w % 4) + 16 ((w / 4) % 2) .. +15, columns CW (w / 8) .. +CW-1,
        // loaded as CW/32 halves of 16 registers (the drain's register budget)
        constexpr int NH = CW / 32;
        const uint32_t lane0 = (warp & 3u) * 32u + ((warp >> 2) & 1u) * 16u;
        const uint32_t col0 = (warp >> 3) * static_cast<uint32_t>(CW);
        const uint32_t q = lane & 3u;                      // column pair 2q, 2q+1 of each group of 8
        const uint32_t r0 = lane0 + (lane >> 2);           // rows r0 and r0 + 8 of the tile
        const uint32_t tlane = tmem_base + (lane0 << 16) + col0;
        float2 acc[2][CW / 8];                             // [row][column group]
        uint32_t tc = 0;                                   // tiles drained
#pragma unroll
        for (int i = 0; i < CW / 8; ++i) acc[0][i] = acc[1][i] = make_float2(0.0f, 0.0f);
        if constexpr (PAIRED) {
            uint32_t bc = 0, uc = 0;                           // blocks and 2-block units drained
            bool ok = true;
            for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x, ++tc) {
                const TileInfo ti = decode_tile<BN>(a, w);
                for (int32_t b = 0; b < nb; ++b, ++bc) {
                    const uint32_t h = static_cast<uint32_t>(b) & 1u;   // block within its unit (nb is even)
                    // the unit's accumulator pair, its phase, and the block's accumulator
                    const uint32_t bi = uc % NBAR_ACC, ph = (uc / NBAR_ACC) & 1u;
                    const uint32_t ab = 2 * bi + h, sc = bc % NSC;
                    if (h == 0) {
                        if (!mbar_wait_warp(&acc_full[bi], ph, a.err)) { ok = false; break; }
                        tc_fence_after();
                    }
                    const float* dws = reinterpret_cast<const float*>(smem + OFF_SC + sc * SC_BYTES);
                    const float4* dap =
                        reinterpret_cast<const float4*>(dws + BM + (col0 / CW) * (4 * DA_QPITCH) + q * DA_QPITCH);
                    const float dw0 = dws[r0], dw1 = dws[r0 + 8];
                    const float2 dw0x2 = make_float2(dw0, dw0), dw1x2 = make_float2(dw1, dw1);
                    // Q4_K: - d_min m_j per row, and d_a sum(q_a) in d_a's layout
                    const float* mws = dws + BM + DA_FLOATS;
                    const float4* sap =
                        reinterpret_cast<const float4*>(mws + BM + (col0 / CW) * (4 * DA_QPITCH) + q * DA_QPITCH);
                    const float2 nm0x2 = KQ ? make_float2(-mws[r0], -mws[r0]) : make_float2(0.0f, 0.0f);
                    const float2 nm1x2 = KQ ? make_float2(-mws[r0 + 8], -mws[r0 + 8]) : make_float2(0.0f, 0.0f);
    #pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        uint32_t d[16];
                        tmem_ld_16x256b_x4(tlane + ab * BN + 32 * hh, d);
                        tmem_wait_ld();
                        if (h == 1 && hh == NH - 1) {            // the unit's accumulator pair fully read
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&acc_empty[bi]);
                        }
                        if constexpr (DUMP) {
    #pragma unroll
                            for (int ig = 0; ig < 4; ++ig)
    #pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int64_t row = ti.m0 + r0 + (e >> 1) * 8;
                                    const int n = col0 + 8 * (4 * hh + ig) + 2 * static_cast<int>(q) + (e & 1);
                                    if (row < a.nrows && n < ti.nvalid) {
                                        const int64_t s = a.perm[ti.p0 + n];
                                        a.dots[(s * a.nrows + row) * nb + b] =
                                            static_cast<int32_t>(__uint_as_float(d[4 * ig + e]));
                                    }
                                }
                        } else {
                            // acc += d_w * (dot * d_a): one packed multiply and one packed FMA per column pair
    #pragma unroll
                            for (int k2 = 0; k2 < 2; ++k2) {
                                const float4 v = dap[2 * hh + k2];   // d_a of columns 8i+2q+{0,1}, i = 4hh+2k2, +1
    #pragma unroll
                                for (int ii = 0; ii < 2; ++ii) {
                                    const int ig = 2 * k2 + ii, i = 4 * hh + ig;
                                    const float2 da2 = ii ? make_float2(v.z, v.w) : make_float2(v.x, v.y);
                                    const float2 t0 =
                                        __fmul2_rn(make_float2(__uint_as_float(d[4 * ig]), __uint_as_float(d[4 * ig + 1])), da2);
                                    const float2 t1 = __fmul2_rn(
                                        make_float2(__uint_as_float(d[4 * ig + 2]), __uint_as_float(d[4 * ig + 3])), da2);
                                    acc[0][i] = __ffma2_rn(t0, dw0x2, acc[0][i]);
                                    acc[1][i] = __ffma2_rn(t1, dw1x2, acc[1][i]);
                                    if constexpr (KQ) {
                                        const float4 sv = sap[2 * hh + k2];
                                        const float2 sa2 = ii ? make_float2(sv.z, sv.w) : make_float2(sv.x, sv.y);
                                        acc[0][i] = __ffma2_rn(sa2, nm0x2, acc[0][i]);
                                        acc[1][i] = __ffma2_rn(sa2, nm1x2, acc[1][i]);
                                    }
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sc_empty[sc]);   // scale slot sc free again
                    uc += h;
                }
                if (!ok) break;
                if constexpr (FUSE) {
                    if (!fused_act_drain<BN>(acc, a, smem + C::OFF_EPI, epi_bar, tc, warp, lane)) break;
    #pragma unroll
                    for (int i = 0; i < CW / 8; ++i) acc[0][i] = acc[1][i] = make_float2(0.0f, 0.0f);
                } else if constexpr (!DUMP) {
    #pragma unroll
                    for (int i = 0; i < CW / 8; ++i) {
    #pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int n = col0 + 8 * i + 2 * static_cast<int>(q) + e;
                            if (n < ti.nvalid) {
                                const int64_t s = a.perm[ti.p0 + n];
                                float* o = a.out + s * a.nrows + ti.m0 + r0;
                                if (ti.m0 + r0 < a.nrows) o[0] = e ? acc[0][i].y : acc[0][i].x;
                                if (ti.m0 + r0 + 8 < a.nrows) o[8] = e ? acc[1][i].y : acc[1][i].x;
                            }
                        }
                        acc[0][i] = acc[1][i] = make_float2(0.0f, 0.0f);
                    }
                }
            }
        } else {
            uint32_t bc = 0;
            bool ok = true;
            for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x, ++tc) {
                const TileInfo ti = decode_tile<BN>(a, w);
                for (int32_t b = 0; b < nb; ++b, ++bc) {
                    const uint32_t ab = bc % NACC, sc = bc % NSC;
                    if (!mbar_wait_warp(&acc_full[ab], (bc / NACC) & 1u, a.err)) { ok = false; break; }
                    tc_fence_after();
                    const float* dws = reinterpret_cast<const float*>(smem + OFF_SC + sc * SC_BYTES);
                    const float4* dap =
                        reinterpret_cast<const float4*>(dws + BM + (col0 / CW) * (4 * DA_QPITCH) + q * DA_QPITCH);
                    const float dw0 = dws[r0], dw1 = dws[r0 + 8];
                    const float2 dw0x2 = make_float2(dw0, dw0), dw1x2 = make_float2(dw1, dw1);
                    // Q4_K: - d_min m_j per row, and d_a sum(q_a) in d_a's layout
                    const float* mws = dws + BM + DA_FLOATS;
                    const float4* sap =
                        reinterpret_cast<const float4*>(mws + BM + (col0 / CW) * (4 * DA_QPITCH) + q * DA_QPITCH);
                    const float2 nm0x2 = KQ ? make_float2(-mws[r0], -mws[r0]) : make_float2(0.0f, 0.0f);
                    const float2 nm1x2 = KQ ? make_float2(-mws[r0 + 8], -mws[r0 + 8]) : make_float2(0.0f, 0.0f);
    #pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        uint32_t d[16];
                        tmem_ld_16x256b_x4(tlane + ab * BN + 32 * hh, d);
                        tmem_wait_ld();
                        if (hh == NH - 1) {                      // TMEM buffer ab fully read
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&acc_empty[ab]);
                        }
                        if constexpr (DUMP) {
    #pragma unroll
                            for (int ig = 0; ig < 4; ++ig)
    #pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int64_t row = ti.m0 + r0 + (e >> 1) * 8;
                                    const int n = col0 + 8 * (4 * hh + ig) + 2 * static_cast<int>(q) + (e & 1);
                                    if (row < a.nrows && n < ti.nvalid) {
                                        const int64_t s = a.perm[ti.p0 + n];
                                        a.dots[(s * a.nrows + row) * nb + b] =
                                            static_cast<int32_t>(__uint_as_float(d[4 * ig + e]));
                                    }
                                }
                        } else {
                            // acc += d_w * (dot * d_a): one packed multiply and one packed FMA per column pair
    #pragma unroll
                            for (int k2 = 0; k2 < 2; ++k2) {
                                const float4 v = dap[2 * hh + k2];   // d_a of columns 8i+2q+{0,1}, i = 4hh+2k2, +1
    #pragma unroll
                                for (int ii = 0; ii < 2; ++ii) {
                                    const int ig = 2 * k2 + ii, i = 4 * hh + ig;
                                    const float2 da2 = ii ? make_float2(v.z, v.w) : make_float2(v.x, v.y);
                                    const float2 t0 =
                                        __fmul2_rn(make_float2(__uint_as_float(d[4 * ig]), __uint_as_float(d[4 * ig + 1])), da2);
                                    const float2 t1 = __fmul2_rn(
                                        make_float2(__uint_as_float(d[4 * ig + 2]), __uint_as_float(d[4 * ig + 3])), da2);
                                    acc[0][i] = __ffma2_rn(t0, dw0x2, acc[0][i]);
                                    acc[1][i] = __ffma2_rn(t1, dw1x2, acc[1][i]);
                                    if constexpr (KQ) {
                                        const float4 sv = sap[2 * hh + k2];
                                        const float2 sa2 = ii ? make_float2(sv.z, sv.w) : make_float2(sv.x, sv.y);
                                        acc[0][i] = __ffma2_rn(sa2, nm0x2, acc[0][i]);
                                        acc[1][i] = __ffma2_rn(sa2, nm1x2, acc[1][i]);
                                    }
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sc_empty[sc]);   // scale slot sc free again
                }
                if (!ok) break;
                if constexpr (FUSE) {
                    if (!fused_act_drain<BN>(acc, a, smem + C::OFF_EPI, epi_bar, tc, warp, lane)) break;
    #pragma unroll
                    for (int i = 0; i < CW / 8; ++i) acc[0][i] = acc[1][i] = make_float2(0.0f, 0.0f);
                } else if constexpr (!DUMP) {
    #pragma unroll
                    for (int i = 0; i < CW / 8; ++i) {
    #pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int n = col0 + 8 * i + 2 * static_cast<int>(q) + e;
                            if (n < ti.nvalid) {
                                const int64_t s = a.perm[ti.p0 + n];
                                float* o = a.out + s * a.nrows + ti.m0 + r0;
                                if (ti.m0 + r0 < a.nrows) o[0] = e ? acc[0][i].y : acc[0][i].x;
                                if (ti.m0 + r0 + 8 < a.nrows) o[8] = e ? acc[1][i].y : acc[1][i].x;
                            }
                        }
                        acc[0][i] = acc[1][i] = make_float2(0.0f, 0.0f);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// --------------------------------------------------------------- gather
// One warp per router position p: slot s = perm[p] of token t = s / k.  Four
// lanes per Q8_1 block, eight blocks per step: lane 4i + q of block b loads
// the block's code words 1 + 2q and 2 + 2q (the warp reads 8 whole blocks,
// 288 contiguous bytes) and stores their 8 codes as fp16 (exact integers) in
// one 16-byte store at xh[p][32b + 8q] (the warp writes 512 contiguous
// bytes); lane q = 0 also copies the block's fp16 d to da[p][b].  Positions
// past the routed slots (bad ids, and the padding up to a multiple of 128
// rows) are written as zeros.
__global__ void __launch_bounds__(256)
    gather_act_kernel(const uint8_t* __restrict__ act, const int32_t* __restrict__ perm,
                      const int32_t* __restrict__ offsets, int32_t n_experts, int32_t top_k, int32_t nb,
                      int64_t n_rows, uint4* __restrict__ xh, uint16_t* __restrict__ da) {
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t n_valid = offsets[n_experts];
    const uint32_t lane = lane_id(), q = lane & 3u;
    const int32_t b0 = static_cast<int32_t>(lane >> 2);
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); p < n_rows;
         p += warps) {
        uint4* xrow = xh + p * nb * 4;      // 4 x 16 bytes per block
        uint16_t* drow = da + p * nb;
        if (p < n_valid) {
            const int64_t t = perm[p] / top_k;
            const uint8_t* src = act + t * nb * Q8_1_BYTES;
#pragma unroll 2
            for (int32_t b = b0; b < nb; b += 8) {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(src + static_cast<int64_t>(b) * Q8_1_BYTES);
                const uint32_t v0 = __ldg(w + 1 + 2 * q), v1 = __ldg(w + 2 + 2 * q);
                uint4 o;
                i8x4_to_h2(v0, o.x, o.y);
                i8x4_to_h2(v1, o.z, o.w);
                xrow[b * 4 + q] = o;
                if (q == 0) drow[b] = static_cast<uint16_t>(__ldg(w) & 0xFFFFu);
            }
        } else {
            for (int32_t j = static_cast<int32_t>(lane); j < nb * 4; j += 32) xrow[j] = make_uint4(0, 0, 0, 0);
            for (int32_t b = static_cast<int32_t>(lane); b < nb; b += 32) drow[b] = 0;
        }
    }
}

// The gather for Q4_K weights: the same fp16 rows and fp16 scales, plus the
// exact d_a * sum(q_a) of every block as fp32 (|sum| <= 4064 and d_a an fp16,
// so the product is exact), the activation factor of the K-quant min term.
// One warp per router position; lane l takes blocks l, l + 32, ... whole.
__global__ void __launch_bounds__(256)
    gather_act_sums_kernel(const uint8_t* __restrict__ act, const int32_t* __restrict__ perm,
                           const int32_t* __restrict__ offsets, int32_t n_experts, int32_t top_k, int32_t nb,
                           int64_t n_rows, uint2* __restrict__ xh, uint16_t* __restrict__ da, float* __restrict__ sa) {
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t n_valid = offsets[n_experts];
    const uint32_t lane = lane_id();
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); p < n_rows;
         p += warps) {
        uint2* xrow = xh + p * nb * 8;      // 8 x 8 bytes per block
        for (int32_t b = lane; b < nb; b += 32) {
            uint32_t w[9];
            if (p < n_valid) {
                const int64_t t = perm[p] / top_k;
                const uint32_t* src = reinterpret_cast<const uint32_t*>(act + (t * nb + b) * Q8_1_BYTES);
#pragma unroll
                for (int i = 0; i < 9; ++i) w[i] = __ldg(src + i);
            } else {
#pragma unroll
                for (int i = 0; i < 9; ++i) w[i] = 0;
            }
            int sum = 0;
#pragma unroll
            for (int i = 1; i < 9; ++i) {
                sum = __dp4a(static_cast<int>(w[i]), 0x01010101, sum);
                uint32_t lo, hi;
                i8x4_to_h2(w[i], lo, hi);
                xrow[b * 8 + (i - 1)] = make_uint2(lo, hi);
            }
            const unsigned short dbits = static_cast<unsigned short>(w[0] & 0xFFFFu);
            da[p * nb + b] = dbits;
            sa[p * nb + b] = __half2float(__ushort_as_half(dbits)) * static_cast<float>(sum);
        }
    }
}

// ------------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz,
                     const char* what) {
    auto encode = get_encode_fn();
    if (!encode) return fail(FT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t gdim[2] = {inner, outer};
    const cuuint64_t gstride[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult cr = encode(map, dt, 2, const_cast<void*>(base), gdim, gstride, box, estride,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(FT_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed (%d)", what, static_cast<int>(cr));
    return FT_OK;
}

int launch_gather(const uint8_t* act, const int32_t* perm, const int32_t* offsets, int32_t n_experts, int32_t top_k,
                  int64_t nb, int64_t n_slots, uint16_t* xh, uint16_t* da, cudaStream_t s, float* sa) {
    const int64_t rows = gemm_rows(n_slots);
    const int64_t want = (rows + 7) / 8;   // one warp per row, all rows at once
    const int64_t cap = 0x7FFFFFFF;
    const dim3 grid(static_cast<unsigned>(want < cap ? want : cap));
    if (sa) {
        gather_act_sums_kernel<<<grid, 256, 0, s>>>(act, perm, offsets, n_experts, top_k, static_cast<int32_t>(nb),
                                                    rows, reinterpret_cast<uint2*>(xh), da, sa);
        return check_launch("gather_act_sums_kernel", grid, dim3(256), 0);
    }
    gather_act_kernel<<<grid, 256, 0, s>>>(act, perm, offsets, n_experts, top_k, static_cast<int32_t>(nb), rows,
                                           reinterpret_cast<uint4*>(xh), da);
    return check_launch("gather_act_kernel", grid, dim3(256), 0);
}

template <int BN, bool DUMP, bool FUSE, bool KQ = false>
static int launch_gemm_kernel(const CUtensorMap& wmap, const CUtensorMap& xmap, const CUtensorMap& smap,
                              const CUtensorMap& amap, const GemmArgs& ga, dim3 grid, cudaStream_t s,
                              const char* name) {
    using C = Gemm<BN, KQ>;
    const void* k = reinterpret_cast<const void*>(moe_gemm_tc_kernel<BN, DUMP, FUSE, KQ>);
    if (int st = set_smem_limit(k, C::SMEM_BYTES)) return st;
    constexpr int threads = FUSE ? C::THREADS_FUSED : C::THREADS;
    moe_gemm_tc_kernel<BN, DUMP, FUSE, KQ><<<grid, threads, C::SMEM_BYTES, s>>>(wmap, xmap, smap, amap, ga);
    return check_launch(name, grid, dim3(threads), C::SMEM_BYTES);
}

template <int BN>
static int launch_gemm_bn(const uint8_t* weights, const int32_t* perm, const int32_t* offsets, const int32_t* tiles,
                          float* out, int32_t* dots, uint32_t* err, int64_t n_slots, int32_t top_k, int32_t n_experts,
                          int64_t nrows, int64_t ncols, const uint16_t* xh, const uint16_t* da, const ActFuse* af,
                          cudaStream_t s, const float* sa) {
    using C = Gemm<BN>;
    const int64_t nb = ncols / QK;
    const int sms = sm_count();
    const int64_t rows = gemm_rows(n_slots);
    // the fused layer 1 loads its 128 rows as two boxes of 64 (gate, up)
    const uint32_t box_rows = af ? C::BM / 2 : C::BM;
    CUtensorMap wmap, xmap, smap;
    if (int st = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, weights, nb * Q4_0_BYTES, n_experts * nrows,
                           nb * Q4_0_BYTES, C::KB * Q4_0_BYTES, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE, "weights"))
        return st;
    if (int st = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, ncols, rows, ncols * 2, 64, BN,
                           CU_TENSOR_MAP_SWIZZLE_128B, "activations"))
        return st;
    if (int st = encode_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, da, nb, rows, nb * 2, C::KB, BN,
                           CU_TENSOR_MAP_SWIZZLE_NONE, "activation scales"))
        return st;
    CUtensorMap amap = smap;   // Q4_K: the slots' d_a sum(q_a), [rows][nb] fp32
    if (sa)
        if (int st = encode_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sa, nb, rows, nb * 4, C::KB, BN,
                               CU_TENSOR_MAP_SWIZZLE_NONE, "activation sums"))
            return st;

    GemmArgs ga{};
    ga.perm = perm;
    ga.offsets = offsets;
    ga.tiles = tiles;
    ga.out = out;
    ga.dots = dots;
    ga.err = err;
    ga.nrows = nrows;
    ga.nb = static_cast<int32_t>(nb);
    ga.top_k = top_k;
    ga.n_experts = n_experts;
    ga.row_tiles = static_cast<int32_t>(af ? (af->n_inter + C::BM / 2 - 1) / (C::BM / 2)
                                           : (nrows + C::BM - 1) / C::BM);
    if (af) {
        ga.act_mid = af->act_mid;
        ga.n_inter = af->n_inter;
        ga.act_kind = af->kind;
    }

    const int64_t slot_tiles_ub = (n_slots + BN - 1) / BN + (n_experts < n_slots ? n_experts : n_slots);
    const int64_t tiles_ub = slot_tiles_ub * ga.row_tiles;
    const dim3 grid(static_cast<unsigned>(tiles_ub < sms ? tiles_ub : sms));
    if (sa) return launch_gemm_kernel<BN, false, false, true>(wmap, xmap, smap, amap, ga, grid, s, "moe_gemm_tc_kernel<q4_k>");
    if (dots) return launch_gemm_kernel<BN, true, false>(wmap, xmap, smap, amap, ga, grid, s, "moe_gemm_tc_kernel<dump>");
    if (af) return launch_gemm_kernel<BN, false, true>(wmap, xmap, smap, amap, ga, grid, s, "moe_gemm_tc_kernel<act>");
    return launch_gemm_kernel<BN, false, false>(wmap, xmap, smap, amap, ga, grid, s, "moe_gemm_tc_kernel");
}

int gemm_tile_width(double mean_slots_per_expert) {
    // narrow slot tiles while experts see few slots each (the drain then scales
    // 32 instead of 128 columns per block); measured crossover between 32 and
    // 64 slots per expert
    return mean_slots_per_expert < 48.0 ? 32 : kGemmBN;
}

int launch_gemm(const uint8_t* weights, const uint8_t* act, const int32_t* perm, const int32_t* offsets,
                const int32_t* tiles, float* out, int32_t* dots, uint32_t* err, int64_t n_slots, int32_t top_k,
                int32_t n_experts, int64_t nrows, int64_t ncols, uint16_t* xh, uint16_t* da, int tile_width,
                cudaStream_t s, const ActFuse* af, const float* sa) {
    (void)act;   // read by launch_gather, which the caller runs first
    if (n_slots == 0) return FT_OK;
    if (af && (dots || af->n_inter * 2 != nrows))
        return fail(FT_ERR_ARG, "the fused activation needs nrows = 2 n_inter and no block dots");
    if (sa && (dots || af)) return fail(FT_ERR_ARG, "Q4_K weights take the plain matmul only");
    if (tile_width == 32)
        return launch_gemm_bn<32>(weights, perm, offsets, tiles, out, dots, err, n_slots, top_k, n_experts, nrows,
                                  ncols, xh, da, af, s, sa);
    return launch_gemm_bn<kGemmBN>(weights, perm, offsets, tiles, out, dots, err, n_slots, top_k, n_experts, nrows,
                                   ncols, xh, da, af, s, sa);
}

}  // namespace ft
