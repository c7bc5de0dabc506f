// GEMV tiles of 8 or 16 slots of the routed Q4_0 x Q8_1 expert matmul
// (moe_vec_q4_0_q8_1 on FreeToken PR #185, "Problem" and "Notes"), and of its
// Q4_1, Q8_0 and Q4_K forms (the per-type launchers of moe_vec.cuh there), on
// the warp-level tensor-core instruction mma.sync.m16n8k16 (fp16 operands,
// fp32 accumulation), for decode batches with more than 4 slots per expert.
// The notes below describe Q4_0; the other types differ only in how a lane's
// weight words are found and widened, in the accumulator's start and in the
// offset term after the dot (at the weight-type branches below).
//
// Why: with 8 slots per tile the row-per-lane kernel (gemv_rows.cuh) spends
// 8 dp4a, three shared loads and two float ops per weight block and slot, and
// is bound by instruction issue well below the memory roofline.  Here one
// m16n8k16 pair forms 16 rows x 8 slots x 32 weights of block dots at once;
// the per-block scales stay in the epilogue of every block (the accumulator
// is in registers, so reading it back costs nothing, where tcgen05 would need
// a tensor-memory round trip per 32-weight block).  A tile of NT = 2 slot
// groups (16 slots) shares the weight fragments between two MMA pairs, so an
// expert with up to 16 slots streams its weights once.
//
// Exactness.  Both operands hold small integers exactly: A = 1024 + q (low
// nibbles) and 1024 + 16 q (high nibbles), formed by OR-ing the nibble into the
// fp16 pattern of 1024; B = the activation codes, divided by 16 for the high
// nibbles (a power of two: exact).  Every product is an integer and every
// partial sum stays below 2^23, so the fp32 accumulation is exact whatever its
// order.  The accumulator starts at -(1032 S_lo + 72 S_hi) with S_lo, S_hi the
// sums of the block's first and last 16 codes, which removes the 1024 offsets
// and the Q4_0 level 8; the result is the integer block dot
// sum_i (q_i - 8) q_a[i], the same integer the dp4a kernels form.  It is then
// scaled as there, acc = fma(dot, d_w * d_a, acc), blocks in order, so the
// outputs equal the row-per-lane kernel's bit for bit wherever that kernel
// does not split K.
//
// Fragment layout (m16n8k16, A row-major 16 x 16, B 16 x 8, per the PTX ISA):
// lane = 4 g + t holds A rows g, g + 8 at k = 2t, 2t+1 (regs 0, 1) and
// 2t+8, 2t+9 (regs 2, 3); B column (slot) g at k = 2t, 2t+1 and 2t+8, 2t+9;
// C rows g, g + 8 at columns (slots) 2t, 2t+1.  Which of a block's 32 weights
// sits at which k is free as long as A and B agree: lane t takes the four
// nibble bytes P_t of the block (an aligned 32-bit word of the shared box:
// bytes 4t..4t+3 for odd blocks, whose nibbles start 4-byte aligned; for even
// blocks 4t-2..4t+1, and 0, 1, 14, 15 for t = 0, joined from two words with a
// byte permute), the low nibbles of bytes 0, 2 / 1, 3 of that word at k = 2t,
// 2t+1 / 2t+8, 2t+9 of the first MMA, the high nibbles likewise in the second.
// The activation side is staged in that order as the lane's 8 codes (biased
// to unsigned bytes), 8 bytes per lane, block and slot group (one
// conflict-free 8-byte load), and turned into fp16 pairs with a byte permute
// and one fp16 op per pair: half the shared memory of staged fp16 pairs,
// which leaves room for 15 row warps and a 3-box ring.
//
// Work split.  The grid is one CTA per SM.  A work unit is (slot tile, group
// of 16 rows), numbered tile-major; there are tiles x ceil(rows / 16) of them
// (the tile count is read on the device).  Each CTA takes one contiguous
// range, cut by weight: a unit whose tile uses its second slot group counts
// 3, any other 2 (about their costs), so the SMs finish together whatever
// the routing; where the tiles are few, each tile gets its share of the CTAs
// so that no CTA stages two tiles.  The CTA walks its range in row blocks of
// RW groups (one TMA box high), cut short at the end of a tile and of the range (the
// warps without a group there skip that block), and restages the activations
// only where the range enters a new tile (units handed out one by one from a
// global counter balance as well but restage at nearly every block, which
// measured slower).  Weights stream as in the row-per-lane kernel: TMA boxes
// of 256 weights (8 blocks; 144 bytes per row for Q4_0) x 16 RW rows through an
// mbarrier ring filled by one producer warp, which runs ahead of the staging.
// Warp r owns rows 16 r .. 16 r + 15 of each box (one m16 tile), so a CTA
// keeps up to 15 row warps busy on one staged activation tile.
#include <type_traits>

#include <cuda_fp16.h>

#include "gemv_rows.cuh"

namespace ft {

// Shared memory: mbarriers full/empty [kMaxRowStages] | work range int64[2] |
// qb [nb][NT][32 lanes] uint2 (codes + 128 at P_t: first / last 16) | xc
// [nb][NT][4] float4 (the accumulator's start for lane t: minus the offset
// sums of slots 2t, 2t+1, twice, as the MMA's C quad) | xd [nb][NT][4] float2
// (d_a of slots 2t, 2t+1; for the types with an offset term float4, then d_a
// sum(q_a) of those slots) | ring (128-byte aligned)
__host__ __device__ inline size_t gemv_mma_qb_offset() { return 8 * 2 * kMaxRowStages + 16; }
__host__ __device__ inline size_t gemv_mma_ring_offset(int nb, int nt, bool offset) {
    return (gemv_mma_qb_offset() + static_cast<size_t>(nb) * nt * (256 + 64 + (offset ? 64 : 32)) + 127) / 128 * 128;
}

// The weight types of this kernel: box row bytes and pitch of 256 weights
// (RowBox), whether a block has an offset term (m, or minus d_min m_j) and
// whether the nibble / code words of lane t are the block's bytes 4t..4t+3
// for every block (Q4_1's and Q4_K's data start 4-byte aligned; Q4_0's and
// Q8_0's every other block 2 bytes off a word).
template <int WT>
struct MmaType {
    static constexpr int PITCH = RowBox<WT>::PITCH;
    static constexpr int BYTES = RowBox<WT>::BYTES;
    static constexpr bool KQ = WT == FT_TYPE_Q4_K;
    static constexpr bool OFFSET = WT == FT_TYPE_Q4_K || WT == FT_TYPE_Q4_1;
    static constexpr bool ALIGNED = WT == FT_TYPE_Q4_K || WT == FT_TYPE_Q4_1;
    static_assert(WT == FT_TYPE_Q4_0 || WT == FT_TYPE_Q4_1 || WT == FT_TYPE_Q8_0 || KQ,
                  "weight type of the mma.sync kernel");
};

size_t gemv_mma_smem(int nb, int nt, int row_warps, int stages, int wtype) {
    const bool offset = wtype == FT_TYPE_Q4_K || wtype == FT_TYPE_Q4_1;
    const int pitch = wtype == FT_TYPE_Q4_1 ? MmaType<FT_TYPE_Q4_1>::PITCH
                      : wtype == FT_TYPE_Q8_0 ? MmaType<FT_TYPE_Q8_0>::PITCH
                                              : MmaType<FT_TYPE_Q4_0>::PITCH;
    return gemv_mma_ring_offset(nb, nt, offset) + static_cast<size_t>(stages) * pitch * 16 * row_warps;
}

// D = A B + C on m16n8k16, fp16 operands, fp32 accumulators (not volatile: a
// pure function of its operands, which the compiler may schedule freely, so
// independent MMAs overlap their latencies)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, float c0,
                                          float c1, float c2, float c3) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// The nibble word P_t of block j (compile-time) of a box row.
template <int J>
__device__ __forceinline__ uint32_t nibble_word(const uint8_t* row, uint32_t t) {
    if constexpr (J & 1) {
        return lds32(row + 18 * J + 2 + 4 * t);
    } else {
        const uint32_t x = lds32(row + 18 * J + 4 * t);
        const uint32_t y = lds32(row + 18 * J + (t ? 4 * t : 16));
        return __byte_perm(x, y, t ? 0x3210u : 0x5432u);
    }
}

// The word of bytes P_t of 16 bytes that start 2 bytes after `base` (the
// first or second half of a Q8_0 block's codes; base 4-byte aligned when the
// block index is even, 2 bytes off when odd): aligned load when ODD, two loads
// and a byte permute (for t = 0) when not, as in nibble_word.
template <bool ODD>
__device__ __forceinline__ uint32_t word_at(const uint8_t* base, uint32_t t) {
    if constexpr (ODD) {
        return lds32(base + 2 + 4 * t);
    } else {
        const uint32_t x = lds32(base + 4 * t);
        const uint32_t y = lds32(base + (t ? 4 * t : 16));
        return __byte_perm(x, y, t ? 0x3210u : 0x5432u);
    }
}

// Four int8 bytes of a word as fp16 pairs under the pattern of 1024: bytes 0, 2
// and 1, 3 -> 1152 + q each (q + 128 is the byte's unsigned value)
__device__ __forceinline__ void int8_to_a(uint32_t w, uint32_t& a02, uint32_t& a13) {
    const uint32_t u = w ^ 0x80808080u;
    a02 = __byte_perm(u, 0x64646464u, 0x4240u);
    a13 = __byte_perm(u, 0x64646464u, 0x4341u);
}

// Activation codes of the staging item (slot, block b, lane t): the 4 bytes
// at positions P_t of the block's first 16 codes (hi: of its last 16).
__device__ __forceinline__ uint32_t code_word(const uint8_t* codes, int32_t b, uint32_t t) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(codes);
    if (b & 1) return __ldg(w + t);
    if (t == 0) return __byte_perm(__ldg(w), __ldg(w + 3), 0x7610u);
    return __byte_perm(__ldg(w + t - 1), __ldg(w + t), 0x5432u);
}

// B fragments from four codes biased by 128 (bytes u = q + 128): bytes 0, 2
// (k = 2t, 2t+1) and 1, 3 (k = 2t+8, 2t+9) as fp16 pairs.  A byte under the
// fp16 pattern of 1024 is 1024 + u exactly; minus 1152 it is q (lo), times
// 1/16 minus 72 it is q / 16 (hi); both exact in fp16.
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }
__device__ __forceinline__ void codes_lo(uint32_t u, uint32_t& b0, uint32_t& b1) {
    const __half2 k = __float2half2_rn(1152.0f);
    b0 = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4240u)), k));
    b1 = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4341u)), k));
}
__device__ __forceinline__ void codes_hi(uint32_t u, uint32_t& b0, uint32_t& b1) {
    const __half2 s = __float2half2_rn(0.0625f), k = __float2half2_rn(-72.0f);
    b0 = h2_bits(__hfma2(bits_h2(__byte_perm(u, 0x64646464u, 0x4240u)), s, k));
    b1 = h2_bits(__hfma2(bits_h2(__byte_perm(u, 0x64646464u, 0x4341u)), s, k));
}


// Enter slot tile `tile` (compute warps, n_threads of them): stage its
// activations as B fragments and offset sums, and return its slot count and
// the slot ids of this thread's output columns (-1: none).
template <int NT, int WT, typename XD>
__device__ __forceinline__ void mma_stage_tile(const GemvArgs& a, int64_t tile, uint2* qb, float4* xc, XD* xd,
                                               int32_t n_threads, int32_t& ng, int32_t (&sid)[NT][2]) {
    using T = MmaType<WT>;
    constexpr bool KQ = T::KQ;
    constexpr int G = 8 * NT;
    const int32_t nb = a.nb;
    const int32_t e = find_expert(a.tiles, a.n_experts, tile);
    const int64_t p0 = static_cast<int64_t>(a.offsets[e]) + (tile - a.tiles[e]) * G;
    ng = static_cast<int32_t>(min(static_cast<int64_t>(G), a.offsets[e + 1] - p0));
    const uint32_t lane = lane_id(), g = lane >> 2, tq = lane & 3u;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int32_t n = nt * 8 + static_cast<int32_t>(2 * tq) + c;
            sid[nt][c] = n < ng ? __ldg(a.perm + p0 + n) : -1;
        }
    // item i = ((b NT + group) 32 + lane), lane = 4 g + t: slot (group, g)'s
    // codes at P_t of block b; the four lanes of a slot add up the block's
    // code sums with two shuffles
    for (int32_t i = static_cast<int32_t>(threadIdx.x); i < nb * NT * 32; i += n_threads) {
        const int32_t bn = i >> 5, b = bn / NT, n = (bn - b * NT) * 8 + static_cast<int32_t>(g);
        uint32_t wl = 0, wh = 0;
        float d = 0.0f;
        if (n < ng) {
            const int64_t tok = __ldg(a.perm + p0 + n) / a.top_k;
            const uint8_t* blk = a.act + (tok * nb + b) * Q8_1_BYTES;
            d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(blk))));
            if constexpr (T::ALIGNED) {                      // P_t = 4t..4t+3 for every block
                wl = __ldg(reinterpret_cast<const uint32_t*>(blk + 4) + tq);
                wh = __ldg(reinterpret_cast<const uint32_t*>(blk + 20) + tq);
            } else {
                wl = code_word(blk + 4, b, tq);
                wh = code_word(blk + 20, b, tq);
            }
        }
        qb[i] = make_uint2(wl ^ 0x80808080u, wh ^ 0x80808080u);
        int sl = __dp4a(static_cast<int>(wl), 0x01010101, 0), sh = __dp4a(static_cast<int>(wh), 0x01010101, 0);
        sl += __shfl_xor_sync(0xFFFFFFFFu, sl, 1);
        sh += __shfl_xor_sync(0xFFFFFFFFu, sh, 1);
        sl += __shfl_xor_sync(0xFFFFFFFFu, sl, 2);
        sh += __shfl_xor_sync(0xFFFFFFFFu, sh, 2);
        if (tq == 0) {
            float* c = reinterpret_cast<float*>(xc + static_cast<size_t>(bn) * 4 + (g >> 1));
            // Q4_0: A = 1024 + q (first 16) and 1024 + 16 q with B / 16 (last 16),
            // level 8; Q4_1 the same with levels 0..15; Q4_K (levels 0..15,
            // sub-block j = b mod 8 = the low nibbles for even j, the high ones
            // as 1024 + 16 q with B / 16 for odd); Q8_0: A = 1152 + q
            const float c0 = KQ                     ? -static_cast<float>(((b & 1) ? 64 : 1024) * (sl + sh))
                             : WT == FT_TYPE_Q4_1 ? -static_cast<float>(1024 * sl + 64 * sh)
                             : WT == FT_TYPE_Q8_0 ? -static_cast<float>(1152 * (sl + sh))
                                                  : -static_cast<float>(1032 * sl + 72 * sh);
            c[g & 1] = c0;
            c[2 + (g & 1)] = c0;
            float* x = reinterpret_cast<float*>(xd + static_cast<size_t>(bn) * 4 + (g >> 1));
            x[g & 1] = d;
            if constexpr (T::OFFSET) x[2 + (g & 1)] = d * small_int_to_float(sl + sh);   // the offset term's d_a sum(q_a)
        }
    }
}

// Unit weights of the work split: a row group of a tile whose second slot
// group holds slots counts 3, one of a tile with 8 slots or fewer 2 (their
// costs, roughly: the second group's MMAs and scaling are most of a unit).
constexpr int64_t kMmaW1 = 2, kMmaW2 = 3;

// The CTA's contiguous range [w0, w1) of the work units (tile-major (tile,
// 16-row group), n_u units per tile), written to range[0..1].  A unit weighs
// W1 or W2 by its tile's slot groups, W in all.  Where every tile's share of
// the grid, grid * (tile weight) / W, is at least one CTA, each tile gets
// that share rounded (cumulatively, so the counts add up to the grid) and
// its units are cut evenly among them: no CTA stages two tiles.  Otherwise
// (many small tiles) CTA c takes the units whose weight interval starts in
// [c W / grid, (c + 1) W / grid).  One warp scans the experts' slot counts
// (tiles of expert e: ceil(count / G), all full but the last).
template <int NT>
__device__ void mma_work_range(const GemvArgs& a, int64_t n_u, int64_t* range) {
    constexpr int G = 8 * NT;
    constexpr int64_t W1 = NT > 1 ? kMmaW1 : 1, W2 = NT > 1 ? kMmaW2 : 1;
    const int32_t E = a.n_experts;
    const uint32_t lane = lane_id();
    const int64_t grid = gridDim.x, c = blockIdx.x;
    auto expert = [&](int32_t e, int64_t& tl, int64_t& wt, int64_t& ulast) {
        const int64_t n = e < E ? static_cast<int64_t>(a.offsets[e + 1] - a.offsets[e]) : 0;
        tl = (n + G - 1) / G;
        ulast = n - G * (tl - 1) > 8 ? W2 : W1;
        wt = tl > 0 ? (tl - 1) * W2 + ulast : 0;
    };
    int64_t tot = 0;
    bool light = false;                            // some tile weighs W1 per unit
    for (int32_t e0 = 0; e0 < E; e0 += 32) {
        int64_t tl, wt, ul;
        expert(e0 + static_cast<int32_t>(lane), tl, wt, ul);
        tot += wt;
        light |= tl > 0 && ul == W1;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
    light = __any_sync(0xFFFFFFFFu, light);
    const int64_t W = tot * n_u;
    const bool per_tile = W > 0 && grid * n_u * (light ? W1 : W2) >= W;
    // CTAs before weight x, per tile mode: round(grid x / W)
    auto ctas_before = [&](int64_t x) { return (2 * grid * x + W) / (2 * W); };
    const int64_t P[2] = {W * c / grid, W * (c + 1) / grid};
    int64_t wbase = 0, ibase = 0;                  // weight and units before the chunk
    if (lane < 2) range[lane] = static_cast<int64_t>(a.tiles[E]) * n_u;   // past the last unit
    __syncwarp();
    for (int32_t e0 = 0; e0 < E; e0 += 32) {
        int64_t tl, wt, ul;
        expert(e0 + static_cast<int32_t>(lane), tl, wt, ul);
        int64_t wi = wt * n_u, ii = tl * n_u;    // inclusive prefix over the chunk
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xFFFFFFFFu, wi, o), z = __shfl_up_sync(0xFFFFFFFFu, ii, o);
            if (static_cast<int>(lane) >= o) {
                wi += y;
                ii += z;
            }
        }
        const int64_t ws = wbase + wi - wt * n_u, is = ibase + ii - tl * n_u;   // this expert's start
        if (per_tile) {
            if (wt > 0 && c >= ctas_before(ws) && c < ctas_before(ws + wt * n_u)) {
                for (int64_t j = 0; j < tl; ++j) {
                    const int64_t c0 = ctas_before(ws + j * W2 * n_u);
                    const int64_t c1 = j + 1 < tl ? ctas_before(ws + (j + 1) * W2 * n_u) : ctas_before(ws + wt * n_u);
                    if (c >= c0 && c < c1) {
                        const int64_t k = c1 - c0, cc = c - c0;
                        range[0] = is + j * n_u + n_u * cc / k;
                        range[1] = is + j * n_u + n_u * (cc + 1) / k;
                    }
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (wt > 0 && P[k] >= ws && P[k] < ws + wt * n_u) {
                    const int64_t q = P[k] - ws, full = (tl - 1) * W2 * n_u;
                    int64_t unit;
                    if (q < full) {
                        const int64_t t = q / (W2 * n_u), q2 = q - t * W2 * n_u;
                        unit = is + t * n_u + (q2 + W2 - 1) / W2;
                    } else {
                        unit = is + (tl - 1) * n_u + (q - full + ul - 1) / ul;
                    }
                    range[k] = unit;
                }
            }
        }
        wbase += __shfl_sync(0xFFFFFFFFu, wi, 31);
        ibase += __shfl_sync(0xFFFFFFFFu, ii, 31);
    }
}

template <int NT, int WT, bool DUMP>
__global__ void __launch_bounds__(512, 1) moe_gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ CUtensorMap wmap16,
                                                              const GemvArgs a) {
    using T = MmaType<WT>;
    constexpr int PITCH = T::PITCH;                       // a box row: 8 blocks, or one Q4_K super-block
    constexpr bool KQ = T::KQ;
    static_assert(!DUMP || WT == FT_TYPE_Q4_0, "block dots are a Q4_0 diagnostic");
    using XD = std::conditional_t<T::OFFSET, float4, float2>;
    const int32_t RW = a.row_warps;                       // warps of 16 rows
    const int32_t E = a.n_experts;
    const int32_t nb = a.nb;
    const int32_t n_ks = nb / 8;                          // boxes per row
    const int NS = a.stages;
    const int64_t n_g = (a.nrows + 15) / 16;              // 16-row groups of a tile

    extern __shared__ __align__(128) uint8_t smem_mma[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_mma);
    uint64_t* empty = full + kMaxRowStages;
    int64_t* range = reinterpret_cast<int64_t*>(empty + kMaxRowStages);
    uint2* qb = reinterpret_cast<uint2*>(smem_mma + gemv_mma_qb_offset());          // [nb][NT][32]
    float4* xc = reinterpret_cast<float4*>(qb + static_cast<size_t>(nb) * NT * 32);  // [nb][NT][4]
    XD* xd = reinterpret_cast<XD*>(xc + static_cast<size_t>(nb) * NT * 4);             // [nb][NT][4]
    uint8_t* ring = smem_mma + gemv_mma_ring_offset(nb, NT, T::OFFSET);
    const uint32_t stage_bytes = static_cast<uint32_t>(PITCH * 16 * RW);
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], RW);
        }
        fence_mbar_init();
    }
    if (warp == 0) mma_work_range<NT>(a, n_g, range);
    __syncthreads();
    const int64_t w0 = range[0], w1 = range[1];
    if (w0 >= w1) return;

    if (static_cast<int32_t>(warp) == RW) {
        // ------------------------------------------------------------ producer
        // the boxes of each row block in K order; a row block is the next RW
        // groups of the range, cut at the end of its tile and of the range
        int64_t it = 0, tile = -1, erow0 = 0;
        for (int64_t u = w0; u < w1;) {
            const int64_t tl = u / n_g, g0 = u - tl * n_g;
            const int64_t cnt = min(static_cast<int64_t>(RW), min(n_g - g0, w1 - u));
            if (tl != tile) {
                tile = tl;
                erow0 = static_cast<int64_t>(find_expert(a.tiles, E, tl)) * a.nrows;
            }
            for (int32_t ks = 0; ks < n_ks; ++ks, ++it) {
                const int32_t s = static_cast<int32_t>(it % NS);
                if (!mbar_wait_warp(&empty[s], static_cast<uint32_t>(((it / NS) & 1) ^ 1), a.err)) return;
                if (lane == 0) {
                    uint8_t* dst = ring + static_cast<size_t>(s) * stage_bytes;
                    if (cnt == RW) {
                        mbar_arrive_expect_tx(&full[s], stage_bytes);
                        tma_load_2d(dst, &wmap, ks * (T::BYTES / 2), static_cast<int32_t>(erow0 + g0 * 16), &full[s]);
                    } else {
                        // a short block: only its groups, 16 rows per copy,
                        // so that no row outside the range leaves memory
                        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(cnt) * 16 * PITCH);
                        for (int64_t i = 0; i < cnt; ++i)
                            tma_load_2d(dst + i * 16 * PITCH, &wmap16, ks * (T::BYTES / 2),
                                        static_cast<int32_t>(erow0 + (g0 + i) * 16), &full[s]);
                    }
                }
                __syncwarp();
            }
            u += cnt;
        }
        return;
    }

    // ----------------------------------------------------------------- compute
    // A warp whose bounded wait gave up stops waiting and computing but still
    // takes every tile change's barriers, so no other warp waits on it.
    const int32_t r = static_cast<int32_t>(warp);
    const uint32_t g = lane >> 2, tq = lane & 3u;
    const uint32_t n_threads = static_cast<uint32_t>(RW) * 32u;
    int64_t cur = -1, it = 0;
    int32_t ng = 0, sid[NT][2];
    bool ok = true;
    for (int64_t u = w0; u < w1;) {
        const int64_t tile = u / n_g, g0 = u - tile * n_g;
        const int64_t cnt = min(static_cast<int64_t>(RW), min(n_g - g0, w1 - u));
        u += cnt;
        if (tile != cur) {
            if (cur >= 0) named_bar_sync(1, n_threads);  // every warp is done with the previous tile
            mma_stage_tile<NT, WT>(a, tile, qb, xc, xd, static_cast<int32_t>(n_threads), ng, sid);
            named_bar_sync(1, n_threads);
            cur = tile;
        }
        if (!ok) continue;
        const bool mine = r < cnt;                         // the block has a group for this warp
        const int64_t row0 = (g0 + r) * 16;                // first row of the warp within the expert
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[nt][c] = 0.0f;
        // one box: 8 blocks x rows g, g + 8 of the warp's 16, against the
        // first (USE = 1) or both (USE = 2) slot groups
        auto box_pass = [&](const uint8_t* ra, int32_t ks, auto USE_) {
            constexpr int USE = decltype(USE_)::value;
            const uint8_t* rb8 = ra + 8 * PITCH;
            auto block = [&](auto J) {
                constexpr int j = decltype(J)::value;
                const int32_t b = ks * 8 + j;
                uint32_t alo[4], ahi[4];                    // A of weights 0..15 and 16..31
                float dwa, dwb, mwa = 0.0f, mwb = 0.0f;
                if constexpr (KQ) {
                    // sub-block j: the low (even j) or high (odd j) nibbles of
                    // qs[32 (j / 2) ..] (the super-block's bytes 16 + ..): weights
                    // 4t..4t+3 and 16+4t.. of it in two aligned words per row
                    constexpr int Q = 16 + 32 * (j >> 1);
                    constexpr uint32_t MASK = (j & 1) ? 0x00F000F0u : 0x000F000Fu;
                    const uint32_t wa0 = lds32(ra + Q + 4 * tq), wa1 = lds32(ra + Q + 16 + 4 * tq);
                    const uint32_t wb0 = lds32(rb8 + Q + 4 * tq), wb1 = lds32(rb8 + Q + 16 + 4 * tq);
                    alo[0] = (wa0 & MASK) | 0x64006400u;
                    alo[1] = (wb0 & MASK) | 0x64006400u;
                    alo[2] = ((wa0 >> 8) & MASK) | 0x64006400u;
                    alo[3] = ((wb0 >> 8) & MASK) | 0x64006400u;
                    ahi[0] = (wa1 & MASK) | 0x64006400u;
                    ahi[1] = (wb1 & MASK) | 0x64006400u;
                    ahi[2] = ((wa1 >> 8) & MASK) | 0x64006400u;
                    ahi[3] = ((wb1 >> 8) & MASK) | 0x64006400u;
                    // d sc_j and d_min m_j of each row, as the dp4a kernels form them
                    const uint4 ha = *reinterpret_cast<const uint4*>(ra), hb = *reinterpret_cast<const uint4*>(rb8);
                    const uint32_t sa[3] = {ha.y, ha.z, ha.w}, sb[3] = {hb.y, hb.z, hb.w};
                    int sca, mna, scb, mnb;
                    kquant_scale_min(sa, j, sca, mna);
                    kquant_scale_min(sb, j, scb, mnb);
                    dwa = __half2float(__ushort_as_half(static_cast<unsigned short>(ha.x & 0xFFFFu))) * static_cast<float>(sca);
                    dwb = __half2float(__ushort_as_half(static_cast<unsigned short>(hb.x & 0xFFFFu))) * static_cast<float>(scb);
                    mwa = __half2float(__ushort_as_half(static_cast<unsigned short>(ha.x >> 16))) * static_cast<float>(mna);
                    mwb = __half2float(__ushort_as_half(static_cast<unsigned short>(hb.x >> 16))) * static_cast<float>(mnb);
                } else if constexpr (WT == FT_TYPE_Q4_1) {
                    // d, m, then the 16 nibble bytes, 4-byte aligned in every block
                    constexpr int O = 20 * j;
                    const uint32_t wa = lds32(ra + O + 4 + 4 * tq), wb = lds32(rb8 + O + 4 + 4 * tq);
                    dwa = __half2float(*reinterpret_cast<const __half*>(ra + O));
                    dwb = __half2float(*reinterpret_cast<const __half*>(rb8 + O));
                    mwa = __half2float(*reinterpret_cast<const __half*>(ra + O + 2));
                    mwb = __half2float(*reinterpret_cast<const __half*>(rb8 + O + 2));
                    const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
                    alo[0] = (wa & 0x000F000Fu) | 0x64006400u;
                    alo[1] = (wb & 0x000F000Fu) | 0x64006400u;
                    alo[2] = (wa8 & 0x000F000Fu) | 0x64006400u;
                    alo[3] = (wb8 & 0x000F000Fu) | 0x64006400u;
                    ahi[0] = (wa & 0x00F000F0u) | 0x64006400u;
                    ahi[1] = (wb & 0x00F000F0u) | 0x64006400u;
                    ahi[2] = (wa8 & 0x00F000F0u) | 0x64006400u;
                    ahi[3] = (wb8 & 0x00F000F0u) | 0x64006400u;
                } else if constexpr (WT == FT_TYPE_Q8_0) {
                    // d, then 32 int8 levels: P_t of the first and of the last 16
                    (void)mwa;
                    (void)mwb;
                    constexpr int O = 34 * j;
                    const uint32_t w0a = word_at<(j & 1) != 0>(ra + O, tq), w1a = word_at<(j & 1) != 0>(ra + O + 16, tq);
                    const uint32_t w0b = word_at<(j & 1) != 0>(rb8 + O, tq), w1b = word_at<(j & 1) != 0>(rb8 + O + 16, tq);
                    dwa = __half2float(*reinterpret_cast<const __half*>(ra + O));
                    dwb = __half2float(*reinterpret_cast<const __half*>(rb8 + O));
                    int8_to_a(w0a, alo[0], alo[2]);
                    int8_to_a(w0b, alo[1], alo[3]);
                    int8_to_a(w1a, ahi[0], ahi[2]);
                    int8_to_a(w1b, ahi[1], ahi[3]);
                } else {
                    (void)mwa;
                    (void)mwb;
                    const uint32_t wa = nibble_word<j>(ra, tq), wb = nibble_word<j>(rb8, tq);
                    dwa = __half2float(*reinterpret_cast<const __half*>(ra + 18 * j));
                    dwb = __half2float(*reinterpret_cast<const __half*>(rb8 + 18 * j));
                    const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
                    alo[0] = (wa & 0x000F000Fu) | 0x64006400u;
                    alo[1] = (wb & 0x000F000Fu) | 0x64006400u;
                    alo[2] = (wa8 & 0x000F000Fu) | 0x64006400u;
                    alo[3] = (wb8 & 0x000F000Fu) | 0x64006400u;
                    ahi[0] = (wa & 0x00F000F0u) | 0x64006400u;
                    ahi[1] = (wb & 0x00F000F0u) | 0x64006400u;
                    ahi[2] = (wa8 & 0x00F000F0u) | 0x64006400u;
                    ahi[3] = (wb8 & 0x00F000F0u) | 0x64006400u;
                }
#pragma unroll
                for (int nt = 0; nt < USE; ++nt) {
                    const size_t bn = static_cast<size_t>(b) * NT + nt;
                    const uint2 Q = qb[bn * 32 + lane];
                    const float4 C = xc[bn * 4 + tq];
                    const XD D = xd[bn * 4 + tq];
                    uint32_t bl0, bl1, bh0, bh1;
                    if constexpr (WT == FT_TYPE_Q8_0 || (KQ && (j & 1) == 0)) {
                        codes_lo(Q.x, bl0, bl1);            // both halves as q
                        codes_lo(Q.y, bh0, bh1);
                    } else if constexpr (KQ) {              // Q4_K, high nibbles: both halves as q / 16
                        codes_hi(Q.x, bl0, bl1);
                        codes_hi(Q.y, bh0, bh1);
                    } else {                                // Q4_0, Q4_1: the high nibbles' codes as q / 16
                        codes_lo(Q.x, bl0, bl1);
                        codes_hi(Q.y, bh0, bh1);
                    }
                    float d0[4], d1[4];
                    mma_16816(d0, alo, bl0, bl1, C.x, C.y, C.z, C.w);
                    mma_16816(d1, ahi, bh0, bh1, d0[0], d0[1], d0[2], d0[3]);
                    if constexpr (DUMP) {
                        (void)D;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int32_t sl = sid[nt][c & 1];
                            const int64_t row = row0 + g + (c < 2 ? 0 : 8);
                            if (sl >= 0 && row < a.nrows)
                                a.dots[(static_cast<int64_t>(sl) * a.nrows + row) * nb + b] = __float2int_rn(d1[c]);
                        }
                    } else {
                        acc[nt][0] = fmaf(d1[0], dwa * D.x, acc[nt][0]);
                        acc[nt][1] = fmaf(d1[1], dwa * D.y, acc[nt][1]);
                        acc[nt][2] = fmaf(d1[2], dwb * D.x, acc[nt][2]);
                        acc[nt][3] = fmaf(d1[3], dwb * D.y, acc[nt][3]);
                        if constexpr (T::OFFSET) {          // + m d_a sum(q_a); Q4_K: minus d_min m_j d_a sum(q_a)
                            constexpr float SG = KQ ? -1.0f : 1.0f;
                            acc[nt][0] = fmaf(SG * mwa, D.z, acc[nt][0]);
                            acc[nt][1] = fmaf(SG * mwa, D.w, acc[nt][1]);
                            acc[nt][2] = fmaf(SG * mwb, D.z, acc[nt][2]);
                            acc[nt][3] = fmaf(SG * mwb, D.w, acc[nt][3]);
                        }
                    }
                }
            };
            block(std::integral_constant<int, 0>{});
            block(std::integral_constant<int, 1>{});
            block(std::integral_constant<int, 2>{});
            block(std::integral_constant<int, 3>{});
            block(std::integral_constant<int, 4>{});
            block(std::integral_constant<int, 5>{});
            block(std::integral_constant<int, 6>{});
            block(std::integral_constant<int, 7>{});
        };
        const bool two = NT > 1 && ng > 8;                // the second slot group holds slots
        for (int32_t ks = 0; ks < n_ks; ++ks, ++it) {
            const int32_t s = static_cast<int32_t>(it % NS);
            if (!mbar_wait_warp(&full[s], static_cast<uint32_t>((it / NS) & 1), a.err)) {
                ok = false;
                break;
            }
            const uint8_t* ra = ring + static_cast<size_t>(s) * stage_bytes + static_cast<size_t>(r * 16 + g) * PITCH;
            if (mine) {
                if (two)
                    box_pass(ra, ks, std::integral_constant<int, NT>{});
                else
                    box_pass(ra, ks, std::integral_constant<int, 1>{});
            }
            // release the box once its values are in registers and used (as in
            // the row-per-lane kernel: the next TMA write must not overtake them)
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (!ok || DUMP || !mine) continue;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int32_t sl = sid[nt][c & 1];
                const int64_t row = row0 + g + (c < 2 ? 0 : 8);
                if (sl >= 0 && row < a.nrows) a.out[static_cast<int64_t>(sl) * a.nrows + row] = acc[nt][c];
            }
    }
}

template <int NT, int WT, bool DUMP>
static int launch_gemv_mma_nt(const GemvPlan& plan, const CUtensorMap& wmap, const CUtensorMap& wmap16, const GemvArgs& a,
                              cudaStream_t s) {
    const void* kernel = reinterpret_cast<const void*>(moe_gemv_mma_kernel<NT, WT, DUMP>);
    if (int st = set_smem_limit(kernel, static_cast<int>(plan.smem))) return st;
    const int threads = 32 * (plan.row_warps + 1);
    // one CTA per SM (or as many as fit); each takes an equal share of the work
    const dim3 grid(static_cast<unsigned>(sm_count() * resident_ctas(kernel, threads, plan.smem)));
    const dim3 block(threads);
    moe_gemv_mma_kernel<NT, WT, DUMP><<<grid, block, plan.smem, s>>>(wmap, wmap16, a);
    return check_launch(DUMP ? "moe_gemv_mma_kernel<dump>" : "moe_gemv_mma_kernel", grid, block, plan.smem);
}

int launch_gemv_mma(const GemvPlan& plan, const CUtensorMap& wmap, const CUtensorMap& wmap16, const GemvArgs& a,
                    bool dump, int wtype, cudaStream_t s) {
    if (wtype != FT_TYPE_Q4_0 && dump) return fail(FT_ERR_ARG, "block dots are Q4_0 only");
    if (wtype == FT_TYPE_Q4_K)
        return plan.mma == 2 ? launch_gemv_mma_nt<2, FT_TYPE_Q4_K, false>(plan, wmap, wmap16, a, s)
                             : launch_gemv_mma_nt<1, FT_TYPE_Q4_K, false>(plan, wmap, wmap16, a, s);
    if (wtype == FT_TYPE_Q4_1)
        return plan.mma == 2 ? launch_gemv_mma_nt<2, FT_TYPE_Q4_1, false>(plan, wmap, wmap16, a, s)
                             : launch_gemv_mma_nt<1, FT_TYPE_Q4_1, false>(plan, wmap, wmap16, a, s);
    if (wtype == FT_TYPE_Q8_0)
        return plan.mma == 2 ? launch_gemv_mma_nt<2, FT_TYPE_Q8_0, false>(plan, wmap, wmap16, a, s)
                             : launch_gemv_mma_nt<1, FT_TYPE_Q8_0, false>(plan, wmap, wmap16, a, s);
    if (plan.mma == 2)
        return dump ? launch_gemv_mma_nt<2, FT_TYPE_Q4_0, true>(plan, wmap, wmap16, a, s)
                    : launch_gemv_mma_nt<2, FT_TYPE_Q4_0, false>(plan, wmap, wmap16, a, s);
    return dump ? launch_gemv_mma_nt<1, FT_TYPE_Q4_0, true>(plan, wmap, wmap16, a, s)
                : launch_gemv_mma_nt<1, FT_TYPE_Q4_0, false>(plan, wmap, wmap16, a, s);
}

}  // namespace ft
