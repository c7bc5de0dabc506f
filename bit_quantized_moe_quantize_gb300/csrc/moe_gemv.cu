// GEMV path of the routed Q4_0 x Q8_1 expert matmul (moe_vec_q4_0_q8_1 on
// FreeToken PR #185), for batches with few slots per expert (decode).
//
// Launch geometry.  grid.x enumerates slot tiles: each is up to G slots of
// one expert taken from the router's permutation, so grid.x is bounded by
// ceil(S / G) + min(E, S) and can reach 2^31 - 1 (FreeToken PR #185, "Fix":
// the flat (token, top-k) index belongs on grid.x, never on grid.z).  The
// tile -> expert map is a binary search over the router's tile prefix, i.e.
// searchsorted(right=True) (nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 2), so
// empty experts own no tile.  grid.y walks weight-row tiles (kept <= 65535;
// a CTA loops when there are more).  Extra CTAs of the upper bound exit.
//
// Per CTA: one bulk copy (cp.async.bulk, mbarrier-tracked) stages the row
// tile's Q4_0 bytes, which are contiguous because an expert's rows are; the
// G activation rows are unpacked into shared memory as 16-byte aligned int8
// blocks plus fp32 scales and exact block sums.  Each weight block is read
// once from shared memory and dotted with all G slots, so weight bytes are
// read from HBM once per (expert, row tile, slot group).
//
// Arithmetic: per block, sum_i q_w[i] * q_a[i] with dp4a on the raw nibbles,
// then minus 8 * sum_i q_a[i] (exact integer), so the block dot is bit-exact;
// it is scaled by d_w * d_a in fp32 and summed over the lane's blocks, then
// across lanes with shuffles.
#include <cuda_fp16.h>

#include "ft_common.cuh"
#include "ft_internal.h"

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
    int32_t rows;        // rows per tile
    int32_t lanes_per_row;
    int64_t row_tiles;
    int32_t bulk;        // weight rows 16-byte aligned -> bulk copy
};

// Shared-memory carve-up (bytes), in this order:
//   mbarrier (16) | slot ids int32[G] (pad 16) | qa [G][nb][32] | da f32 [G][nb]
//   | suma i32 [G][nb] | weight tile [rows][nb][18] (+16 pad)
__host__ __device__ inline size_t gemv_smem_bytes(int G, int nb, int rows) {
    size_t o = 16;
    o += ((static_cast<size_t>(G) * 4 + 15) / 16) * 16;
    o += static_cast<size_t>(G) * nb * 32;
    o += static_cast<size_t>(G) * nb * 4;
    o += static_cast<size_t>(G) * nb * 4;
    o = (o + 15) / 16 * 16;
    o += static_cast<size_t>(rows) * nb * Q4_0_BYTES + 16;
    return o;
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

template <int G, bool DUMP>
__global__ void __launch_bounds__(256) moe_gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int64_t t = blockIdx.x;
    const int32_t E = a.n_experts;
    if (t >= a.tiles[E]) return;
    const int32_t e = find_expert(a.tiles, E, t);
    const int64_t p0 = static_cast<int64_t>(a.offsets[e]) + (t - a.tiles[e]) * G;
    const int32_t ng = static_cast<int32_t>(min(static_cast<int64_t>(G), a.offsets[e + 1] - p0));
    const int32_t nb = a.nb;

    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* slot = reinterpret_cast<int32_t*>(smem + 16);
    size_t o = 16 + ((static_cast<size_t>(G) * 4 + 15) / 16) * 16;
    uint8_t* qa = smem + o;
    o += static_cast<size_t>(G) * nb * 32;
    float* da = reinterpret_cast<float*>(smem + o);
    o += static_cast<size_t>(G) * nb * 4;
    int32_t* suma = reinterpret_cast<int32_t*>(smem + o);
    o += static_cast<size_t>(G) * nb * 4;
    o = (o + 15) / 16 * 16;
    uint8_t* wt = smem + o;

    const int64_t row_bytes = static_cast<int64_t>(nb) * Q4_0_BYTES;
    const uint8_t* wexp = a.weights + static_cast<int64_t>(e) * a.nrows * row_bytes;

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < G) slot[threadIdx.x] = threadIdx.x < ng ? a.perm[p0 + threadIdx.x] : 0;
    __syncthreads();

    // unpack the G activation rows: int8 block, fp32 d, exact sum of q
    for (int32_t i = threadIdx.x; i < ng * nb; i += blockDim.x) {
        const int32_t g = i / nb, b = i - g * nb;
        const int64_t tok = slot[g] / a.top_k;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.act + (tok * nb + b) * Q8_1_BYTES);
        const uint32_t ds = __ldg(src);
        uint4 q0 = make_uint4(__ldg(src + 1), __ldg(src + 2), __ldg(src + 3), __ldg(src + 4));
        uint4 q1 = make_uint4(__ldg(src + 5), __ldg(src + 6), __ldg(src + 7), __ldg(src + 8));
        uint4* dst = reinterpret_cast<uint4*>(qa + (static_cast<size_t>(g) * nb + b) * 32);
        dst[0] = q0;
        dst[1] = q1;
        da[g * nb + b] = __half2float(__ushort_as_half(static_cast<unsigned short>(ds & 0xFFFFu)));
        int s = 0;
        s = __dp4a(static_cast<int>(q0.x), 0x01010101, s);
        s = __dp4a(static_cast<int>(q0.y), 0x01010101, s);
        s = __dp4a(static_cast<int>(q0.z), 0x01010101, s);
        s = __dp4a(static_cast<int>(q0.w), 0x01010101, s);
        s = __dp4a(static_cast<int>(q1.x), 0x01010101, s);
        s = __dp4a(static_cast<int>(q1.y), 0x01010101, s);
        s = __dp4a(static_cast<int>(q1.z), 0x01010101, s);
        s = __dp4a(static_cast<int>(q1.w), 0x01010101, s);
        suma[g * nb + b] = s;
    }

    const int L = a.lanes_per_row;
    const int rows_per_warp_pass = 32 / L;
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const int sub = static_cast<int>(lane) % L;
    const int rsub = static_cast<int>(lane) / L;
    uint32_t phase = 0;

    for (int64_t y = blockIdx.y; y < a.row_tiles; y += gridDim.y) {
        const int64_t r0 = y * a.rows;
        const int32_t nr = static_cast<int32_t>(min(static_cast<int64_t>(a.rows), a.nrows - r0));
        const uint8_t* src = wexp + r0 * row_bytes;
        const uint32_t bytes = static_cast<uint32_t>(nr * row_bytes);
        if (a.bulk) {
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(bar, bytes);
                bulk_g2s(wt, src, bytes, bar);
            }
        } else {
            // rows not 16-byte aligned: 2-byte loads (blocks are 2-byte aligned)
            const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
            uint16_t* d16 = reinterpret_cast<uint16_t*>(wt);
            for (uint32_t i = threadIdx.x; i < bytes / 2; i += blockDim.x) d16[i] = __ldg(s16 + i);
        }
        __syncthreads();   // activations unpacked (first pass) / fallback tile written
        if (a.bulk && !mbar_wait(bar, phase, a.err)) return;
        phase ^= 1u;

        for (int32_t rl = static_cast<int32_t>(warp) * rows_per_warp_pass + rsub; rl - rsub < nr;
             rl += 8 * rows_per_warp_pass) {
            const bool row_ok = rl < nr;
            float acc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] = 0.0f;
            if (row_ok) {
                const uint32_t rbase = static_cast<uint32_t>(rl) * static_cast<uint32_t>(row_bytes);
                for (int b = sub; b < nb; b += L) {
                    const uint32_t off = rbase + static_cast<uint32_t>(b) * Q4_0_BYTES;
                    const uint32_t sh = off & 2u;
                    const uint32_t* w = reinterpret_cast<const uint32_t*>(wt + (off - sh));
                    const uint32_t W0 = w[0], W1 = w[1], W2 = w[2], W3 = w[3], W4 = w[4];
                    const uint32_t sel = sh ? 0x7654u : 0x5432u;
                    const uint32_t q0 = __byte_perm(W0, W1, sel), q1 = __byte_perm(W1, W2, sel);
                    const uint32_t q2 = __byte_perm(W2, W3, sel), q3 = __byte_perm(W3, W4, sel);
                    const float dw =
                        __half2float(__ushort_as_half(static_cast<unsigned short>((W0 >> (sh * 8)) & 0xFFFFu)));
                    const int l0 = q0 & 0x0F0F0F0F, l1 = q1 & 0x0F0F0F0F, l2 = q2 & 0x0F0F0F0F, l3 = q3 & 0x0F0F0F0F;
                    const int h0 = (q0 >> 4) & 0x0F0F0F0F, h1 = (q1 >> 4) & 0x0F0F0F0F;
                    const int h2 = (q2 >> 4) & 0x0F0F0F0F, h3 = (q3 >> 4) & 0x0F0F0F0F;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        if (g < ng) {
                            const uint4* av = reinterpret_cast<const uint4*>(qa + (static_cast<size_t>(g) * nb + b) * 32);
                            const uint4 A0 = av[0], A1 = av[1];
                            int dot = 0;
                            dot = __dp4a(l0, static_cast<int>(A0.x), dot);
                            dot = __dp4a(l1, static_cast<int>(A0.y), dot);
                            dot = __dp4a(l2, static_cast<int>(A0.z), dot);
                            dot = __dp4a(l3, static_cast<int>(A0.w), dot);
                            dot = __dp4a(h0, static_cast<int>(A1.x), dot);
                            dot = __dp4a(h1, static_cast<int>(A1.y), dot);
                            dot = __dp4a(h2, static_cast<int>(A1.z), dot);
                            dot = __dp4a(h3, static_cast<int>(A1.w), dot);
                            dot -= 8 * suma[g * nb + b];
                            if constexpr (DUMP) {
                                a.dots[(static_cast<int64_t>(slot[g]) * a.nrows + r0 + rl) * nb + b] = dot;
                            } else {
                                acc[g] = fmaf(static_cast<float>(dot), dw * da[g * nb + b], acc[g]);
                            }
                        }
                    }
                }
            }
            if constexpr (!DUMP) {
#pragma unroll
                for (int g = 0; g < G; ++g)
                    for (int o2 = L >> 1; o2 > 0; o2 >>= 1) acc[g] += __shfl_xor_sync(0xFFFFFFFFu, acc[g], o2);
                if (row_ok && sub == 0) {
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        if (g < ng) a.out[static_cast<int64_t>(slot[g]) * a.nrows + r0 + rl] = acc[g];
                }
            }
        }
        __syncthreads();   // tile consumed before the next copy overwrites it
    }
}

GemvPlan plan_gemv(int64_t n_slots, int32_t n_experts, int64_t nrows, int64_t ncols) {
    GemvPlan p{};
    const int64_t nb = ncols / QK;
    const double mean = static_cast<double>(n_slots) / n_experts;
    p.group = mean <= 1.0 ? 1 : mean <= 2.0 ? 2 : mean <= 4.0 ? 4 : 8;
    p.lanes_per_row = nb >= 24 ? 32 : nb >= 12 ? 16 : 8;
    const int64_t row_bytes = nb * Q4_0_BYTES;
    int64_t rows = 49152 / row_bytes;
    rows = rows < 1 ? 1 : rows > 16 ? 16 : rows;
    p.rows = static_cast<int>(rows);
    p.row_tiles = (nrows + rows - 1) / rows;
    p.smem = gemv_smem_bytes(p.group, static_cast<int>(nb), p.rows);
    while (p.smem > 220 * 1024 && p.group > 1) {   // very long rows: fewer slots per tile
        p.group >>= 1;
        p.smem = gemv_smem_bytes(p.group, static_cast<int>(nb), p.rows);
    }
    const int64_t ub = (n_slots + p.group - 1) / p.group + (n_experts < n_slots ? n_experts : n_slots);
    p.grid_x = ub < n_slots ? ub : n_slots;
    return p;
}

template <int G, bool DUMP>
static int launch_gemv_t(const GemvPlan& plan, const GemvArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(plan.grid_x),
                    static_cast<unsigned>(plan.row_tiles < 65535 ? plan.row_tiles : 65535));
    const dim3 block(256);
    if (int st = set_smem_limit(reinterpret_cast<const void*>(moe_gemv_kernel<G, DUMP>), static_cast<int>(plan.smem)))
        return st;
    moe_gemv_kernel<G, DUMP><<<grid, block, plan.smem, s>>>(a);
    return check_launch(DUMP ? "moe_gemv_kernel<dump>" : "moe_gemv_kernel", grid, block, plan.smem);
}

int launch_gemv(const GemvPlan& plan, const uint8_t* weights, const uint8_t* act, const int32_t* perm,
                const int32_t* offsets, const int32_t* tiles, float* out, int32_t* dots, uint32_t* err,
                int64_t n_slots, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols, cudaStream_t s) {
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
    a.rows = plan.rows;
    a.lanes_per_row = plan.lanes_per_row;
    a.row_tiles = plan.row_tiles;
    a.bulk = ((a.nb * Q4_0_BYTES) % 16 == 0) && ((reinterpret_cast<uintptr_t>(weights) & 15u) == 0);
    (void)n_slots;
    const bool dump = dots != nullptr;
    switch (plan.group) {
        case 1: return dump ? launch_gemv_t<1, true>(plan, a, s) : launch_gemv_t<1, false>(plan, a, s);
        case 2: return dump ? launch_gemv_t<2, true>(plan, a, s) : launch_gemv_t<2, false>(plan, a, s);
        case 4: return dump ? launch_gemv_t<4, true>(plan, a, s) : launch_gemv_t<4, false>(plan, a, s);
        default: return dump ? launch_gemv_t<8, true>(plan, a, s) : launch_gemv_t<8, false>(plan, a, s);
    }
}

}  // namespace ft
