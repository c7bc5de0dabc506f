// The block-per-lane GEMV kernel of the routed expert matmul, templated on the
// weight block type (GGUF Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q2_K..Q6_K: the
// per-type launchers of moe_vec.cuh on FreeToken PR #185, "Notes"), with its shared
// arguments and launch helpers.  moe_gemv.cu instantiates it for Q4_0 next to
// the row-per-lane kernel; moe_gemv_gguf.cu for the other types.
#pragma once

#include <cuda_fp16.h>

#include "gemm_common.cuh"

namespace ft {


struct GemvArgs {
    const uint8_t* weights;
    const uint8_t* act;
    const int32_t* perm;
    const int32_t* offsets;
    const int32_t* tiles;
    float* out;
    int32_t* dots;
    uint32_t* err;
    int64_t nrows;
    int32_t nb;          // blocks per row
    int32_t top_k;
    int32_t n_experts;
    int32_t stages;      // depth of the weight ring (1..kMaxStages)
    int64_t rows_per_cta;
    int32_t bulk;        // weight rows 16-byte aligned -> bulk copies
    int32_t row_warps;   // row-per-lane kernel: row groups of 32 per CTA
    int32_t ksplit;      // row-per-lane kernel: warps sharing a row group, each on every ksplit-th box
    // decode step in one launch (row-per-lane kernel, FUSED): the kernel routes
    // the n_slots ids itself and quantizes the fp16 rows x [tokens][nb * 32]
    const uint16_t* x;
    const int32_t* ids;
    int64_t n_slots;
};

constexpr int kMaxStages = 4;

// Shared-memory carve-up (bytes), in this order:
//   mbarriers [kMaxStages] (32) | slot ids int32[G] (pad 16) | qa [G][nb][32] |
//   da f32 [G][nb] | suma i32 [G][nb] | weight ring [stages][R rows][row bytes] (+16 pad each)
__host__ __device__ inline size_t gemv_act_bytes(int G, int nb) {
    return (32 + ((static_cast<size_t>(G) * 4 + 15) / 16) * 16 + static_cast<size_t>(G) * nb * 40 + 15) / 16 * 16;
}
__host__ __device__ inline size_t gemv_stage_bytes(int R, int nb, int block_bytes = Q4_0_BYTES) {
    return (static_cast<size_t>(R) * nb * block_bytes + 16 + 15) / 16 * 16;
}

__device__ __forceinline__ int32_t find_expert(const int32_t* tiles, int32_t n_experts, int64_t t) {
    // largest e in [0, E) with tiles[e] <= t  (tiles[E] > t is guaranteed by the caller)
    int32_t lo = 0, hi = n_experts - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (tiles[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// One 18-byte Q4_0 block at a 2-byte aligned shared-memory offset: fp32 d and
// the 16 nibble bytes as four words (qs[4i..4i+3] in word i).
__device__ __forceinline__ void load_q4_block(const uint8_t* base, uint32_t off, float& d, uint32_t (&q)[4]) {
    const uint32_t sh = off & 2u;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(base + (off - sh));
    const uint32_t W0 = w[0], W1 = w[1], W2 = w[2], W3 = w[3], W4 = w[4];
    const uint32_t sel = sh ? 0x7654u : 0x5432u;
    q[0] = __byte_perm(W0, W1, sel);
    q[1] = __byte_perm(W1, W2, sel);
    q[2] = __byte_perm(W2, W3, sel);
    q[3] = __byte_perm(W3, W4, sel);
    d = __half2float(__ushort_as_half(static_cast<unsigned short>((W0 >> (sh * 8)) & 0xFFFFu)));
}

// NW words starting at a 2-byte aligned shared-memory offset (reads one word
// past them: every ring stage carries 16 bytes of padding)
template <int NW>
__device__ __forceinline__ void load_words(const uint8_t* base, uint32_t off, uint32_t (&w)[NW]) {
    const uint32_t sh = off & 2u;
    const uint32_t* p = reinterpret_cast<const uint32_t*>(base + (off - sh));
    uint32_t raw[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) raw[i] = p[i];
    const uint32_t sel = sh ? 0x5432u : 0x3210u;
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __byte_perm(raw[i], raw[i + 1], sel);
}

__device__ __forceinline__ float half_at(const uint8_t* base, uint32_t off) {
    return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(base + off)));
}

// bits 0..3 of x -> bit 4 of bytes 0..3
__device__ __forceinline__ uint32_t spread4(uint32_t x) {
    return ((x & 1u) << 4) | ((x & 2u) << 11) | ((x & 4u) << 18) | ((x & 8u) << 25);
}

// Weight block types of the block-per-lane kernel (GGUF): per type its bytes
// per stored block, the 32-weight sub-blocks a stored block holds (8 for the
// K-quant super-blocks), the level offset subtracted from the stored level
// (Q4_0: 8, Q5_0: 16), whether the block stores an fp16 m (c = m, Q4_1 / Q5_1:
// the offset term is m s_a) and whether a sub-block carries a min
// (K-quants: - dmin m_j d_a sum(q_a), with the exact sum of the codes), and
// whether the block's two 16-weight halves carry their own scales (Q6_K,
// Q3_K, Q2_K: d sc_lo and d sc_hi come back in d and m) and their own mins
// (Q2_K: dmin min_lo and dmin min_hi, from decode_mins).
template <int WT>
struct WBlock;
template <> struct WBlock<FT_TYPE_Q4_0> { static constexpr int bytes = 18, per = 1, level0 = 8; static constexpr bool has_m = false, has_min = false, split = false, split_min = false; };
template <> struct WBlock<FT_TYPE_Q4_1> { static constexpr int bytes = 20, per = 1, level0 = 0; static constexpr bool has_m = true, has_min = false, split = false, split_min = false; };
template <> struct WBlock<FT_TYPE_Q5_0> { static constexpr int bytes = 22, per = 1, level0 = 16; static constexpr bool has_m = false, has_min = false, split = false, split_min = false; };
template <> struct WBlock<FT_TYPE_Q5_1> { static constexpr int bytes = 24, per = 1, level0 = 0; static constexpr bool has_m = true, has_min = false, split = false, split_min = false; };
template <> struct WBlock<FT_TYPE_Q8_0> { static constexpr int bytes = 34, per = 1, level0 = 0; static constexpr bool has_m = false, has_min = false, split = false, split_min = false; };
template <> struct WBlock<FT_TYPE_Q4_K> { static constexpr int bytes = 144, per = 8, level0 = 0; static constexpr bool has_m = false, has_min = true, split = false, split_min = false; };
template <> struct WBlock<FT_TYPE_Q5_K> { static constexpr int bytes = 176, per = 8, level0 = 0; static constexpr bool has_m = false, has_min = true, split = false, split_min = false; };
template <> struct WBlock<FT_TYPE_Q6_K> { static constexpr int bytes = 210, per = 8, level0 = 0; static constexpr bool has_m = false, has_min = false, split = true, split_min = false; };
template <> struct WBlock<FT_TYPE_Q2_K> { static constexpr int bytes = 84, per = 8, level0 = 0; static constexpr bool has_m = false, has_min = false, split = true, split_min = true; };
template <> struct WBlock<FT_TYPE_Q3_K> { static constexpr int bytes = 110, per = 8, level0 = 0; static constexpr bool has_m = false, has_min = false, split = true, split_min = false; };

// 6-bit scale and min of sub-block j of a K-quant super-block from its 12
// packed bytes (w[0..2] = bytes 0..11): j < 4 the low 6 bits of bytes j and
// j + 4; j >= 4 the low / high nibble of byte j + 4 with the top two bits of
// byte j - 4 / j above it.
__device__ __forceinline__ void kquant_scale_min(const uint32_t (&w)[3], int j, int& sc, int& mn) {
    auto byte = [&](int i) { return static_cast<int>((w[i >> 2] >> (8 * (i & 3))) & 0xFFu); };
    if (j < 4) {
        sc = byte(j) & 63;
        mn = byte(j + 4) & 63;
    } else {
        sc = (byte(j + 4) & 15) | ((byte(j - 4) >> 6) << 4);
        mn = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
    }
}

// One 32-weight block (sub-block j of the stored block at a 2-byte aligned
// shared-memory offset): fp32 d and m (the K-quants: d sc_j and dmin m_j),
// and its 32 stored levels as int8 lanes of eight words, weights 0..15 in
// lo[0..3] and 16..31 in hi[0..3] (the order of the Q8_1 codes they meet).
template <int WT>
__device__ __forceinline__ void decode_block(const uint8_t* base, uint32_t off, int j, float& d, float& m,
                                             int (&lo)[4], int (&hi)[4]) {
    m = 0.0f;
    if constexpr (WT == FT_TYPE_Q4_0) {
        uint32_t q[4];
        load_q4_block(base, off, d, q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = static_cast<int>(q[i] & 0x0F0F0F0Fu);
            hi[i] = static_cast<int>((q[i] >> 4) & 0x0F0F0F0Fu);
        }
    } else if constexpr (WT == FT_TYPE_Q4_1) {
        uint32_t w[5];
        load_words<5>(base, off, w);
        d = __half2float(__ushort_as_half(static_cast<unsigned short>(w[0] & 0xFFFFu)));
        m = __half2float(__ushort_as_half(static_cast<unsigned short>(w[0] >> 16)));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = static_cast<int>(w[1 + i] & 0x0F0F0F0Fu);
            hi[i] = static_cast<int>((w[1 + i] >> 4) & 0x0F0F0F0Fu);
        }
    } else if constexpr (WT == FT_TYPE_Q5_0 || WT == FT_TYPE_Q5_1) {
        constexpr uint32_t H0 = WT == FT_TYPE_Q5_0 ? 2 : 4;   // offset of the 5th-bit word
        d = half_at(base, off);
        if constexpr (WT == FT_TYPE_Q5_1) m = half_at(base, off + 2);
        uint32_t qh[1], qs[4];
        load_words<1>(base, off + H0, qh);
        load_words<4>(base, off + H0 + 4, qs);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = static_cast<int>((qs[i] & 0x0F0F0F0Fu) | spread4(qh[0] >> (4 * i)));
            hi[i] = static_cast<int>(((qs[i] >> 4) & 0x0F0F0F0Fu) | spread4(qh[0] >> (16 + 4 * i)));
        }
    } else if constexpr (WT == FT_TYPE_Q4_K || WT == FT_TYPE_Q5_K) {
        constexpr uint32_t Q0 = WT == FT_TYPE_Q5_K ? 48 : 16;   // offset of the nibbles
        uint32_t hd[1], sc12[3], qs[8];
        load_words<1>(base, off, hd);
        load_words<3>(base, off + 4, sc12);
        load_words<8>(base, off + Q0 + 32 * (j >> 1), qs);
        int sc, mn;
        kquant_scale_min(sc12, j, sc, mn);
        d = __half2float(__ushort_as_half(static_cast<unsigned short>(hd[0] & 0xFFFFu))) * static_cast<float>(sc);
        m = __half2float(__ushort_as_half(static_cast<unsigned short>(hd[0] >> 16))) * static_cast<float>(mn);
        const int sh = 4 * (j & 1);
        uint32_t qh[8];
        if constexpr (WT == FT_TYPE_Q5_K) load_words<8>(base, off + 16, qh);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t l = (qs[i] >> sh) & 0x0F0F0F0Fu, h = (qs[4 + i] >> sh) & 0x0F0F0F0Fu;
            if constexpr (WT == FT_TYPE_Q5_K) {   // bit j of each qh byte -> bit 4 of the level byte
                l |= ((qh[i] >> j) & 0x01010101u) << 4;
                h |= ((qh[4 + i] >> j) & 0x01010101u) << 4;
            }
            lo[i] = static_cast<int>(l);
            hi[i] = static_cast<int>(h);
        }
    } else if constexpr (WT == FT_TYPE_Q6_K) {
        // sub-block j = 4 h + k: low nibbles from byte 64 h + 32 (k % 2) + l
        // (high nibble for k >= 2), 2-bit high parts from bits 2k of byte
        // 128 + 32 h + l, level - 32; int8 scales 8 h + 2k (weights < 16) and
        // 8 h + 2k + 1; fp16 d last
        const int h = j >> 2, k = j & 3;
        uint32_t ql[8], qh[8];
        load_words<8>(base, off + 64 * h + 32 * (k & 1), ql);
        load_words<8>(base, off + 128 + 32 * h, qh);
        const unsigned short scw = *reinterpret_cast<const unsigned short*>(base + off + 192 + 8 * h + 2 * k);
        const float d6 = half_at(base, off + 208);
        d = d6 * static_cast<float>(static_cast<int8_t>(scw & 0xFFu));
        m = d6 * static_cast<float>(static_cast<int8_t>(scw >> 8));
        const int sh = 4 * (k >> 1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t l = ((ql[i] >> sh) & 0x0F0F0F0Fu) | (((qh[i] >> (2 * k)) & 0x03030303u) << 4);
            const uint32_t hh = ((ql[4 + i] >> sh) & 0x0F0F0F0Fu) | (((qh[4 + i] >> (2 * k)) & 0x03030303u) << 4);
            lo[i] = static_cast<int>(__vsub4(l, 0x20202020u));   // per byte: level - 32 as int8
            hi[i] = static_cast<int>(__vsub4(hh, 0x20202020u));
        }
    } else if constexpr (WT == FT_TYPE_Q2_K || WT == FT_TYPE_Q3_K) {
        // sub-block j = 4 h + k: bits 2k of code byte 32 h + l; groups 2j (weights
        // < 16) and 2j + 1.  Q2_K: scale bytes 0..15 (scale | min << 4), codes at
        // 16, fp16 d at 80.  Q3_K: hmask at 0 (bit j = third bit), codes at 32,
        // twelve bytes of 6-bit scales at 96 (minus 32), fp16 d at 108; level =
        // (code | third bit << 2) - 4.
        const int h = j >> 2, k = j & 3;
        constexpr uint32_t C0 = WT == FT_TYPE_Q2_K ? 16 : 32;
        uint32_t c[8];
        load_words<8>(base, off + C0 + 32 * h, c);
        uint32_t hm[8];
        if constexpr (WT == FT_TYPE_Q3_K) load_words<8>(base, off, hm);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t l = (c[i] >> (2 * k)) & 0x03030303u, hh = (c[4 + i] >> (2 * k)) & 0x03030303u;
            if constexpr (WT == FT_TYPE_Q3_K) {
                l = __vsub4(l | (((hm[i] >> j) & 0x01010101u) << 2), 0x04040404u);
                hh = __vsub4(hh | (((hm[4 + i] >> j) & 0x01010101u) << 2), 0x04040404u);
            }
            lo[i] = static_cast<int>(l);
            hi[i] = static_cast<int>(hh);
        }
        if constexpr (WT == FT_TYPE_Q2_K) {
            const unsigned short scw = *reinterpret_cast<const unsigned short*>(base + off + 2 * j);
            const float d2 = half_at(base, off + 80);
            d = d2 * static_cast<float>(scw & 0x0Fu);
            m = d2 * static_cast<float>((scw >> 8) & 0x0Fu);
        } else {
            uint32_t sw[3];
            load_words<3>(base, off + 96, sw);
            auto byte = [&](int i) { return static_cast<int>((sw[i >> 2] >> (8 * (i & 3))) & 0xFFu); };
            int v[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int g = 2 * j + t;
                const int low4 = g < 8 ? (byte(g & 7) & 15) : (byte(g & 7) >> 4);
                const int top2 = (byte(8 + (g & 3)) >> (2 * (g >> 2))) & 3;
                v[t] = (low4 | (top2 << 4)) - 32;
            }
            const float d3 = half_at(base, off + 108);
            d = d3 * static_cast<float>(v[0]);
            m = d3 * static_cast<float>(v[1]);
        }
    } else {
        static_assert(WT == FT_TYPE_Q8_0, "weight type");
        d = half_at(base, off);
        uint32_t q[8];
        load_words<8>(base, off + 2, q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = static_cast<int>(q[i]);
            hi[i] = static_cast<int>(q[4 + i]);
        }
    }
}

// Q2_K's two group mins of sub-block j: dmin * (scale byte >> 4).
__device__ __forceinline__ void decode_mins_q2k(const uint8_t* base, uint32_t off, int j, float& mn_lo, float& mn_hi) {
    const unsigned short scw = *reinterpret_cast<const unsigned short*>(base + off + 2 * j);
    const float dmin = half_at(base, off + 82);
    mn_lo = dmin * static_cast<float>((scw >> 4) & 0x0Fu);
    mn_hi = dmin * static_cast<float>(scw >> 12);
}

// int32 -> fp32 for |v| < 2^22 with an integer add and a float subtract
__device__ __forceinline__ float small_int_to_float(int v) {
    return __int_as_float(v + 0x4B400000) - 12582912.0f;
}

// grid.x: slot tiles (G slots of one expert); grid.y: a contiguous range of that
// expert's rows, streamed through a ring of `stages` bulk copies of R = 8 * RW
// rows.  Warp w handles rows w*RW .. w*RW+RW-1 of each stage, lane l the blocks
// b = l, l + 32, ... of those rows, and every activation block it loads from
// shared memory serves RW rows.  WT is the weight block type: per block
//   d_w d_a (sum_i q_i q_a[i] - level0 * sum_i q_a[i])  +  m d_a sum_i q_a[i]
// with q_i the stored level, the m term only for the types that store m, and
// the exact sum of the activation codes (never the Q8_1 block's rounded s).
template <int WT, int G, int RW, bool DUMP>
__global__ void __launch_bounds__(256) moe_gemv_kernel(const GemvArgs a) {
    constexpr int R = 8 * RW;
    constexpr int WB = WBlock<WT>::bytes;
    constexpr int PER = WBlock<WT>::per;
    constexpr bool HAS_M = WBlock<WT>::has_m;
    constexpr bool HAS_MIN = WBlock<WT>::has_min;
    constexpr bool SPLIT = WBlock<WT>::split;
    constexpr bool SPLIT_MIN = WBlock<WT>::split_min;
    static_assert(!(SPLIT && DUMP), "block dots are a Q4_0 diagnostic");
    extern __shared__ __align__(16) uint8_t smem[];
    const int64_t t = blockIdx.x;
    const int32_t E = a.n_experts;
    if (t >= a.tiles[E]) return;
    const int64_t r_begin = static_cast<int64_t>(blockIdx.y) * a.rows_per_cta;
    if (r_begin >= a.nrows) return;
    const int64_t r_end = min(a.nrows, r_begin + a.rows_per_cta);
    const int32_t n_st = static_cast<int32_t>((r_end - r_begin + R - 1) / R);
    const int32_t e = find_expert(a.tiles, E, t);
    const int64_t p0 = static_cast<int64_t>(a.offsets[e]) + (t - a.tiles[e]) * G;
    const int32_t ng = static_cast<int32_t>(min(static_cast<int64_t>(G), a.offsets[e + 1] - p0));
    const int32_t nb = a.nb;
    const int NS = a.stages;

    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* slot = reinterpret_cast<int32_t*>(smem + 32);
    size_t o = 32 + ((static_cast<size_t>(G) * 4 + 15) / 16) * 16;
    uint8_t* qa = smem + o;
    o += static_cast<size_t>(G) * nb * 32;
    float* da = reinterpret_cast<float*>(smem + o);
    o += static_cast<size_t>(G) * nb * 4;
    int32_t* suma = reinterpret_cast<int32_t*>(smem + o);
    uint8_t* ring = smem + gemv_act_bytes(G, nb);
    const int64_t row_bytes = static_cast<int64_t>(nb / PER) * WB;
    // R rows + 16 bytes of padding, 16-byte granular (Q6_K's 210-byte blocks
    // make a row no whole number of bytes per 32 weights)
    const size_t stage_bytes = (static_cast<size_t>(R) * row_bytes + 16 + 15) / 16 * 16;
    const uint8_t* wexp = a.weights + static_cast<int64_t>(e) * a.nrows * row_bytes;
    auto stage_rows = [&](int32_t st) { return static_cast<int32_t>(min(static_cast<int64_t>(R), r_end - (r_begin + st * R))); };
    auto issue = [&](int32_t st) {   // one thread: bulk copy of stage st into its ring slot
        const int32_t buf = st % NS;
        const uint32_t bytes = static_cast<uint32_t>(stage_rows(st) * row_bytes);
        mbar_arrive_expect_tx(&bar[buf], bytes);
        bulk_g2s(ring + buf * stage_bytes, wexp + (r_begin + static_cast<int64_t>(st) * R) * row_bytes, bytes, &bar[buf]);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    if (threadIdx.x < G) slot[threadIdx.x] = threadIdx.x < ng ? a.perm[p0 + threadIdx.x] : 0;
    __syncthreads();
    if (a.bulk && threadIdx.x == 0)
        for (int32_t st = 0; st < min(NS, n_st); ++st) issue(st);

    // stage the G activation rows once: int8 block, fp32 d, exact sum of q
    for (int32_t i = threadIdx.x; i < ng * nb; i += blockDim.x) {
        const int32_t g = i / nb, b = i - g * nb;
        const int64_t tok = slot[g] / a.top_k;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.act + (tok * nb + b) * Q8_1_BYTES);
        const uint32_t ds = __ldg(src);
        const uint4 q0 = make_uint4(__ldg(src + 1), __ldg(src + 2), __ldg(src + 3), __ldg(src + 4));
        const uint4 q1 = make_uint4(__ldg(src + 5), __ldg(src + 6), __ldg(src + 7), __ldg(src + 8));
        uint4* dst = reinterpret_cast<uint4*>(qa + (static_cast<size_t>(g) * nb + b) * 32);
        dst[0] = q0;
        dst[1] = q1;
        da[g * nb + b] = __half2float(__ushort_as_half(static_cast<unsigned short>(ds & 0xFFFFu)));
        int sm = 0;
        sm = __dp4a(static_cast<int>(q0.x), 0x01010101, sm);
        sm = __dp4a(static_cast<int>(q0.y), 0x01010101, sm);
        sm = __dp4a(static_cast<int>(q0.z), 0x01010101, sm);
        sm = __dp4a(static_cast<int>(q0.w), 0x01010101, sm);
        const int sm_lo = sm;
        sm = __dp4a(static_cast<int>(q1.x), 0x01010101, sm);
        sm = __dp4a(static_cast<int>(q1.y), 0x01010101, sm);
        sm = __dp4a(static_cast<int>(q1.z), 0x01010101, sm);
        sm = __dp4a(static_cast<int>(q1.w), 0x01010101, sm);
        // split-min types keep the two 16-code sums (|sum| <= 2032) in one word
        suma[g * nb + b] = SPLIT_MIN ? static_cast<int>((static_cast<uint32_t>(sm_lo) & 0xFFFFu) |
                                                        (static_cast<uint32_t>(sm - sm_lo) << 16))
                                     : sm;
    }
    __syncthreads();

    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    for (int32_t st = 0; st < n_st; ++st) {
        const int32_t buf = st % NS;
        const int32_t nr = stage_rows(st);
        const int64_t r0 = r_begin + static_cast<int64_t>(st) * R;
        uint8_t* wt = ring + buf * stage_bytes;
        if (a.bulk) {
            if (!mbar_wait(&bar[buf], static_cast<uint32_t>((st / NS) & 1), a.err)) break;
        } else {
            // rows not 16-byte aligned: 2-byte loads (blocks are 2-byte aligned)
            const uint16_t* s16 = reinterpret_cast<const uint16_t*>(wexp + r0 * row_bytes);
            uint16_t* d16 = reinterpret_cast<uint16_t*>(wt);
            const uint32_t n16 = static_cast<uint32_t>(nr * row_bytes / 2);
            for (uint32_t i = threadIdx.x; i < n16; i += blockDim.x) d16[i] = __ldg(s16 + i);
            __syncthreads();
        }

        const int32_t rl0 = static_cast<int32_t>(warp) * RW;   // this warp's first row in the stage
        float acc[RW][G];
#pragma unroll
        for (int j = 0; j < RW; ++j)
#pragma unroll
            for (int g = 0; g < G; ++g) acc[j][g] = 0.0f;
        if (rl0 < nr) {
            for (int b = static_cast<int>(lane); b < nb; b += 32) {
                int lo[RW][4], hi[RW][4];
                float dw[RW], mw[RW], mn_lo[RW], mn_hi[RW];
#pragma unroll
                for (int j = 0; j < RW; ++j) {
                    const int rl = min(rl0 + j, nr - 1);       // rows past the stage repeat the last one
                    if constexpr (SPLIT_MIN)
                        decode_mins_q2k(wt, static_cast<uint32_t>(rl * row_bytes + (b / PER) * WB), b % PER, mn_lo[j],
                                        mn_hi[j]);
                    else
                        mn_lo[j] = mn_hi[j] = 0.0f;
                    decode_block<WT>(wt, static_cast<uint32_t>(rl * row_bytes + (b / PER) * WB), b % PER, dw[j], mw[j],
                                     lo[j], hi[j]);
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (g < ng) {
                        const uint4* av = reinterpret_cast<const uint4*>(qa + (static_cast<size_t>(g) * nb + b) * 32);
                        const uint4 A0 = av[0], A1 = av[1];
                        const float dag = da[g * nb + b];
                        const int sa0 = WBlock<WT>::level0 * suma[g * nb + b];
                        // offset term's activation factor, with the exact code sum:
                        // d_a sum(q_a) (Q4_1, Q5_1) or -d_a sum(q_a) (K-quant mins)
                        const float sag = HAS_M     ? dag * small_int_to_float(suma[g * nb + b])
                                          : HAS_MIN ? -dag * small_int_to_float(suma[g * nb + b])
                                                    : 0.0f;
#pragma unroll
                        for (int j = 0; j < RW; ++j) {
                            if constexpr (SPLIT) {   // two scale groups of 16 weights
                                int dl = __dp4a(lo[j][0], static_cast<int>(A0.x), 0);
                                dl = __dp4a(lo[j][1], static_cast<int>(A0.y), dl);
                                dl = __dp4a(lo[j][2], static_cast<int>(A0.z), dl);
                                dl = __dp4a(lo[j][3], static_cast<int>(A0.w), dl);
                                int dh = __dp4a(hi[j][0], static_cast<int>(A1.x), 0);
                                dh = __dp4a(hi[j][1], static_cast<int>(A1.y), dh);
                                dh = __dp4a(hi[j][2], static_cast<int>(A1.z), dh);
                                dh = __dp4a(hi[j][3], static_cast<int>(A1.w), dh);
                                acc[j][g] = fmaf(small_int_to_float(dl), dw[j] * dag, acc[j][g]);
                                acc[j][g] = fmaf(small_int_to_float(dh), mw[j] * dag, acc[j][g]);
                                if constexpr (SPLIT_MIN) {   // - min_g d_a sum_g(q_a), both groups
                                    const int sw = suma[g * nb + b];
                                    const float s_lo = small_int_to_float(static_cast<int16_t>(sw & 0xFFFF));
                                    const float s_hi = small_int_to_float(sw >> 16);
                                    acc[j][g] = fmaf(-mn_lo[j] * dag, s_lo, acc[j][g]);
                                    acc[j][g] = fmaf(-mn_hi[j] * dag, s_hi, acc[j][g]);
                                }
                                continue;
                            }
                            int dot = -sa0;
                            dot = __dp4a(lo[j][0], static_cast<int>(A0.x), dot);
                            dot = __dp4a(lo[j][1], static_cast<int>(A0.y), dot);
                            dot = __dp4a(lo[j][2], static_cast<int>(A0.z), dot);
                            dot = __dp4a(lo[j][3], static_cast<int>(A0.w), dot);
                            dot = __dp4a(hi[j][0], static_cast<int>(A1.x), dot);
                            dot = __dp4a(hi[j][1], static_cast<int>(A1.y), dot);
                            dot = __dp4a(hi[j][2], static_cast<int>(A1.z), dot);
                            dot = __dp4a(hi[j][3], static_cast<int>(A1.w), dot);
                            if constexpr (DUMP) {
                                if (rl0 + j < nr)
                                    a.dots[(static_cast<int64_t>(slot[g]) * a.nrows + r0 + rl0 + j) * nb + b] = dot;
                            } else {
                                acc[j][g] = fmaf(small_int_to_float(dot), dw[j] * dag, acc[j][g]);
                                if constexpr (HAS_M || HAS_MIN) acc[j][g] = fmaf(mw[j], sag, acc[j][g]);
                            }
                        }
                    }
                }
            }
        }
        if constexpr (!DUMP) {
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v = acc[j][g];
#pragma unroll
                    for (int o2 = 16; o2 > 0; o2 >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o2);
                    acc[j][g] = v;
                }
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < RW; ++j)
                    if (rl0 + j < nr) {
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            if (g < ng) a.out[static_cast<int64_t>(slot[g]) * a.nrows + r0 + rl0 + j] = acc[j][g];
                    }
            }
        }
        __syncthreads();   // ring slot consumed
        if (a.bulk && threadIdx.x == 0 && st + NS < n_st) issue(st + NS);
    }
}


template <int WT, int G, int RW, bool DUMP>
static int launch_gemv_t(const GemvPlan& plan, const GemvArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(plan.grid_x), static_cast<unsigned>(plan.row_tiles));
    const dim3 block(256);
    if (int st = set_smem_limit(reinterpret_cast<const void*>(moe_gemv_kernel<WT, G, RW, DUMP>),
                                static_cast<int>(plan.smem)))
        return st;
    moe_gemv_kernel<WT, G, RW, DUMP><<<grid, block, plan.smem, s>>>(a);
    return check_launch(DUMP ? "moe_gemv_kernel<dump>" : "moe_gemv_kernel", grid, block, plan.smem);
}

template <int WT, int G, bool DUMP>
static int launch_gemv_rw(const GemvPlan& plan, const GemvArgs& a, cudaStream_t s) {
    switch (plan.lanes_per_row) {
        case 4: return launch_gemv_t<WT, G, 4, DUMP>(plan, a, s);
        case 2: return launch_gemv_t<WT, G, 2, DUMP>(plan, a, s);
        default: return launch_gemv_t<WT, G, 1, DUMP>(plan, a, s);
    }
}


// The block-per-lane kernel for a weight type other than Q4_0 (moe_gemv_gguf.cu).
int launch_gemv_gguf(int wtype, const GemvPlan& plan, const GemvArgs& a, cudaStream_t s);

}  // namespace ft
