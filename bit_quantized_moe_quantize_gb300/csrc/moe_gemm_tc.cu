// Expert-grouped GEMM path of the routed Q4_0 x Q8_1 expert matmul (prefill),
// on the sm_103a tensor cores (tcgen05 MMA into TMEM).
//
// The grouped form follows the expert_offsets layout of nvfp4-megamoe-kernel
// CURRENT_BUG.md (Bug 4: offsets with a leading 0; Bug 2: position -> expert
// by searchsorted(right=True)), but without the fixed-layout padding of
// "Key Architecture: Fixed-Layout Padding": tiles are cut from the router's
// padding-free permutation, so no expert is padded to a fixed row count.
//
// Tile = (expert e, up to 128 routed slots of e, 128 weight rows of e).
// A persistent grid (one CTA per SM) walks the tile list, whose length is
// read on the device from the router's tile prefix; empty experts own no
// tile.  Per CTA, warp-specialized:
//   warp 12  producer: per stage of 8 Q4_0 blocks (K = 256) one 2-D TMA load
//            of the 128 x 144-byte weight box, plus one 288-byte bulk copy per
//            routed slot of its Q8_1 activation row segment (the gather);
//   warps 8-11 unpack: Q4_0 nibbles -> fp16 (q - 8) and int8 q_a -> fp16,
//            both exact, into the K-major 128-byte-swizzled operand layout,
//            plus the fp32 block scales d_w (per row) and d_a (per slot);
//   warp 13  MMA: per 32-value block, two tcgen05.mma kind::f16 (K = 16)
//            M = 128, N = 128 into its own TMEM accumulator (4 buffers);
//   warps 0-7 drain: tcgen05.ld the block's exact integer dot (fp32 holds it
//            exactly: |dot| <= 32512), acc += dot * (d_w * d_a) in fp32
//            registers, and at the end of the tile store the 128 x 128
//            outputs to out[slot][row] (32 consecutive rows per warp store).
//
// Why fp16 operands: every operand value is a small integer (q_w - 8 in
// [-8, 7], q_a in [-127, 127]), exact in fp16, and a 32-term block dot is
// exact in the fp32 accumulator, so the per-block integer dot is bit-exact
// while running at the fp16 tensor rate.  The scales change every 32 values
// along K, so each block needs its own accumulator and a drain; the drain's
// two fp32 operations per (row, slot, block) set this kernel's ceiling.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "ft_common.cuh"
#include "ft_internal.h"

namespace ft {

namespace gemm {
constexpr int BM = kGemmBM;                 // weight rows per tile
constexpr int BN = kGemmBN;                 // slots per tile
constexpr int KB = 8;                       // Q4_0 blocks per raw stage (K = 256)
constexpr int RAW_STAGES = 2;
constexpr int OP_SLOTS = 2;                 // operand slots of 2 blocks (K = 64, one 128-B swizzle atom)
constexpr int NACC = 4;                     // TMEM accumulators, 128 columns each
constexpr int NSC = 8;                      // scale ring depth (blocks)
constexpr int W_RAW_BYTES = BM * KB * Q4_0_BYTES;    // 18432
constexpr int A_RAW_BYTES = BN * KB * Q8_1_BYTES;    // 36864
constexpr int RAW_STAGE_BYTES = W_RAW_BYTES + A_RAW_BYTES;
constexpr int OPA_BYTES = BM * 128;                  // 16384
constexpr int OPB_BYTES = BN * 128;                  // 16384
constexpr int OP_SLOT_BYTES = OPA_BYTES + OPB_BYTES;
constexpr int SC_BYTES = (BM + BN) * 4;
constexpr int N_DRAIN_WARPS = 8, N_UNPACK_WARPS = 4;
constexpr int WARP_PRODUCER = 12, WARP_MMA = 13;
constexpr int THREADS = 14 * 32;
constexpr uint32_t TMEM_COLS = 512;

// smem offsets from a 1024-aligned base
constexpr int OFF_OP = 0;
constexpr int OFF_RAW = OFF_OP + OP_SLOTS * OP_SLOT_BYTES;
constexpr int OFF_SC = OFF_RAW + RAW_STAGES * RAW_STAGE_BYTES;
constexpr int OFF_BAR = OFF_SC + NSC * SC_BYTES;
constexpr int N_BARS = 2 * RAW_STAGES + 2 * OP_SLOTS + 2 * NACC + 2 * NSC;
constexpr int OFF_TMEM = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_TMEM + 16 + 1024;     // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
}  // namespace gemm

struct GemmArgs {
    const uint8_t* act;
    const int32_t* perm;
    const int32_t* offsets;
    const int32_t* tiles;
    float* out;
    int32_t* dots;
    uint32_t* err;
    int64_t nrows;
    int32_t nb;
    int32_t top_k;
    int32_t n_experts;
    int32_t row_tiles;
};

struct TileInfo {
    int32_t e;
    int64_t p0;
    int32_t nvalid;
    int64_t m0;
};

__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int64_t w) {
    TileInfo ti;
    const int64_t st = w / a.row_tiles;
    const int64_t mt = w - st * a.row_tiles;
    int32_t lo = 0, hi = a.n_experts - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (a.tiles[mid] <= st) lo = mid;
        else hi = mid - 1;
    }
    ti.e = lo;
    ti.p0 = static_cast<int64_t>(a.offsets[lo]) + (st - a.tiles[lo]) * gemm::BN;
    ti.nvalid = static_cast<int32_t>(min(static_cast<int64_t>(gemm::BN), a.offsets[lo + 1] - ti.p0));
    ti.m0 = mt * gemm::BM;
    return ti;
}

// Byte offset of 16-byte chunk c of row r in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) {
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

// Four packed nibble bytes -> two fp16x2 words holding (nibble - 8), in order.
__device__ __forceinline__ void nib4_to_h2(uint32_t nib, uint32_t& lo, uint32_t& hi) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    uint32_t a = __byte_perm(nib, 0x64646464u, 0x4140u);
    uint32_t b = __byte_perm(nib, 0x64646464u, 0x4342u);
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
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

template <bool DUMP>
__global__ void __launch_bounds__(gemm::THREADS, 1)
    moe_gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const GemmArgs a) {
    using namespace gemm;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + RAW_STAGES;
    uint64_t* op_full = raw_empty + RAW_STAGES;
    uint64_t* op_empty = op_full + OP_SLOTS;
    uint64_t* acc_full = op_empty + OP_SLOTS;
    uint64_t* acc_empty = acc_full + NACC;
    uint64_t* sc_full = acc_empty + NACC;
    uint64_t* sc_empty = sc_full + NSC;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);

    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const int32_t nb = a.nb;
    const int32_t n_stages = nb / KB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RAW_STAGES; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], N_UNPACK_WARPS * 32);
        }
        for (int i = 0; i < OP_SLOTS; ++i) {
            mbar_init(&op_full[i], N_UNPACK_WARPS * 32);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], N_DRAIN_WARPS);
        }
        for (int i = 0; i < NSC; ++i) {
            mbar_init(&sc_full[i], N_UNPACK_WARPS * 32);
            mbar_init(&sc_empty[i], N_DRAIN_WARPS);
        }
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == WARP_PRODUCER && lane == 0) prefetch_tmap(&wmap);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int64_t total = static_cast<int64_t>(a.tiles[a.n_experts]) * a.row_tiles;

    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ producer
        uint32_t it = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
            const TileInfo ti = decode_tile(a, w);
            int64_t arow[BN / 32];
#pragma unroll
            for (int j = 0; j < BN / 32; ++j) {
                const int n = static_cast<int>(lane) + 32 * j;
                arow[j] = n < ti.nvalid ? static_cast<int64_t>(a.perm[ti.p0 + n] / a.top_k) * nb * Q8_1_BYTES : 0;
            }
            const int32_t wy = static_cast<int32_t>(static_cast<int64_t>(ti.e) * a.nrows + ti.m0);
            for (int32_t ks = 0; ks < n_stages; ++ks, ++it) {
                const uint32_t s = it % RAW_STAGES;
                if (!mbar_wait_warp(&raw_empty[s], ((it / RAW_STAGES) & 1u) ^ 1u, a.err)) { ok = false; break; }
                uint8_t* wraw = smem + OFF_RAW + s * RAW_STAGE_BYTES;
                uint8_t* araw = wraw + W_RAW_BYTES;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&raw_full[s], W_RAW_BYTES + ti.nvalid * (KB * Q8_1_BYTES));
                    tma_load_2d(wraw, &wmap, ks * KB * Q4_0_BYTES, wy, &raw_full[s]);
                }
                __syncwarp();
#pragma unroll
                for (int j = 0; j < BN / 32; ++j) {
                    const int n = static_cast<int>(lane) + 32 * j;
                    if (n < ti.nvalid)
                        bulk_g2s(araw + n * (KB * Q8_1_BYTES),
                                 a.act + arow[j] + static_cast<int64_t>(ks) * (KB * Q8_1_BYTES),
                                 KB * Q8_1_BYTES, &raw_full[s]);
                }
            }
        }
    } else if (warp >= N_DRAIN_WARPS && warp < N_DRAIN_WARPS + N_UNPACK_WARPS) {
        // -------------------------------------------------------------- unpack
        const uint32_t u = threadIdx.x - N_DRAIN_WARPS * 32;   // weight row and slot index, 0..127
        uint32_t it = 0, ou = 0, bc = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
            const TileInfo ti = decode_tile(a, w);
            const bool slot_ok = static_cast<int32_t>(u) < ti.nvalid;
            for (int32_t ks = 0; ks < n_stages && ok; ++ks, ++it) {
                const uint32_t s = it % RAW_STAGES;
                if (!mbar_wait(&raw_full[s], (it / RAW_STAGES) & 1u, a.err)) { ok = false; break; }
                const uint8_t* wraw = smem + OFF_RAW + s * RAW_STAGE_BYTES;
                const uint8_t* araw = wraw + W_RAW_BYTES;
                for (int j = 0; j < KB / 2; ++j, ++ou) {
                    const uint32_t os = ou % OP_SLOTS;
                    if (!mbar_wait(&op_empty[os], ((ou / OP_SLOTS) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    uint8_t* opa = smem + OFF_OP + os * OP_SLOT_BYTES;
                    uint8_t* opb = opa + OPA_BYTES;
                    for (int h = 0; h < 2; ++h, ++bc) {
                        const int bi = 2 * j + h;
                        const uint32_t sc = bc % NSC;
                        if (!mbar_wait(&sc_empty[sc], ((bc / NSC) & 1u) ^ 1u, a.err)) { ok = false; break; }
                        float* dws = reinterpret_cast<float*>(smem + OFF_SC + sc * SC_BYTES);
                        float* das = dws + BM;
                        // weight row u, block bi: 18 bytes at a 2-byte aligned offset
                        {
                            const uint32_t off = u * (KB * Q4_0_BYTES) + bi * Q4_0_BYTES;
                            const uint32_t sh = off & 2u;
                            const uint32_t* wv = reinterpret_cast<const uint32_t*>(wraw + (off - sh));
                            const uint32_t W0 = wv[0], W1 = wv[1], W2 = wv[2], W3 = wv[3], W4 = wv[4];
                            const uint32_t sel = sh ? 0x7654u : 0x5432u;
                            const uint32_t q[4] = {__byte_perm(W0, W1, sel), __byte_perm(W1, W2, sel),
                                                   __byte_perm(W2, W3, sel), __byte_perm(W3, W4, sel)};
                            dws[u] = __half2float(
                                __ushort_as_half(static_cast<unsigned short>((W0 >> (sh * 8)) & 0xFFFFu)));
                            uint32_t hv[16];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                nib4_to_h2(q[i] & 0x0F0F0F0Fu, hv[2 * i], hv[2 * i + 1]);            // values 4i..4i+3
                                nib4_to_h2((q[i] >> 4) & 0x0F0F0F0Fu, hv[8 + 2 * i], hv[8 + 2 * i + 1]);  // 16+4i..
                            }
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                *reinterpret_cast<uint4*>(opa + sw128_off(u, 4 * h + c)) =
                                    make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
                        }
                        // slot u, block bi: 36 bytes, 4-byte aligned
                        if (slot_ok) {
                            const uint32_t* av =
                                reinterpret_cast<const uint32_t*>(araw + u * (KB * Q8_1_BYTES) + bi * Q8_1_BYTES);
                            das[u] = __half2float(__ushort_as_half(static_cast<unsigned short>(av[0] & 0xFFFFu)));
                            uint32_t hv[16];
#pragma unroll
                            for (int i = 0; i < 8; ++i) i8x4_to_h2(av[1 + i], hv[2 * i], hv[2 * i + 1]);
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                *reinterpret_cast<uint4*>(opb + sw128_off(u, 4 * h + c)) =
                                    make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
                        } else {
                            das[u] = 0.0f;
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                *reinterpret_cast<uint4*>(opb + sw128_off(u, 4 * h + c)) = make_uint4(0, 0, 0, 0);
                        }
                        mbar_arrive(&sc_full[sc]);
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
        if (lane == 0) {
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
                        }
                        tc_commit(&op_empty[os]);
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------------- drain
        const uint32_t quarter = warp & 3u, colh = warp >> 2;
        const uint32_t row_l = quarter * 32 + lane;                       // TMEM lane = weight row in tile
        float acc[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) acc[c] = 0.0f;
        uint32_t bc = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
            const TileInfo ti = decode_tile(a, w);
            const int64_t row = ti.m0 + row_l;
            for (int32_t b = 0; b < nb; ++b, ++bc) {
                const uint32_t ab = bc % NACC, sc = bc % NSC;
                if (!mbar_wait_warp(&acc_full[ab], (bc / NACC) & 1u, a.err)) { ok = false; break; }
                if (!mbar_wait_warp(&sc_full[sc], (bc / NSC) & 1u, a.err)) { ok = false; break; }
                tc_fence_after();
                const float* dws = reinterpret_cast<const float*>(smem + OFF_SC + sc * SC_BYTES);
                const float* das = dws + BM + colh * 64;
                const float dw = dws[row_l];
                const uint32_t taddr = tmem_base + ((quarter * 32u) << 16) + ab * BN + colh * 64;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + part * 32, r);
                    tmem_wait_ld();
                    if constexpr (DUMP) {
                        if (row < a.nrows) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const int n = colh * 64 + part * 32 + c;
                                if (n < ti.nvalid) {
                                    const int64_t s = a.perm[ti.p0 + n];
                                    a.dots[(s * a.nrows + row) * nb + b] =
                                        static_cast<int32_t>(__uint_as_float(r[c]));
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 d4 = *reinterpret_cast<const float4*>(das + part * 32 + 4 * c4);
                            acc[part * 32 + 4 * c4 + 0] = fmaf(__uint_as_float(r[4 * c4 + 0]), dw * d4.x, acc[part * 32 + 4 * c4 + 0]);
                            acc[part * 32 + 4 * c4 + 1] = fmaf(__uint_as_float(r[4 * c4 + 1]), dw * d4.y, acc[part * 32 + 4 * c4 + 1]);
                            acc[part * 32 + 4 * c4 + 2] = fmaf(__uint_as_float(r[4 * c4 + 2]), dw * d4.z, acc[part * 32 + 4 * c4 + 2]);
                            acc[part * 32 + 4 * c4 + 3] = fmaf(__uint_as_float(r[4 * c4 + 3]), dw * d4.w, acc[part * 32 + 4 * c4 + 3]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&acc_empty[ab]);
                    mbar_arrive(&sc_empty[sc]);
                }
            }
            if (!ok) break;
            if constexpr (!DUMP) {
                if (row < a.nrows) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int n = colh * 64 + c;
                        if (n < ti.nvalid) {
                            const int64_t s = a.perm[ti.p0 + n];
                            a.out[s * a.nrows + row] = acc[c];
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) acc[c] = 0.0f;
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

int launch_gemm(const uint8_t* weights, const uint8_t* act, const int32_t* perm, const int32_t* offsets,
                const int32_t* tiles, float* out, int32_t* dots, uint32_t* err, int64_t n_slots, int32_t top_k,
                int32_t n_experts, int64_t nrows, int64_t ncols, int64_t tokens, cudaStream_t s) {
    using namespace gemm;
    (void)tokens;
    if (n_slots == 0) return FT_OK;
    const int64_t nb = ncols / QK;
    auto encode = get_encode_fn();
    if (!encode) return fail(FT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    CUtensorMap wmap;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(nb * Q4_0_BYTES), static_cast<cuuint64_t>(n_experts * nrows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(nb * Q4_0_BYTES)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(KB * Q4_0_BYTES), static_cast<cuuint32_t>(BM)};
    const cuuint32_t estride[2] = {1, 1};
    CUresult cr = encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(weights), gdim, gstride, box,
                         estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(FT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(cr));

    GemmArgs ga{};
    ga.act = act;
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
    ga.row_tiles = static_cast<int32_t>((nrows + BM - 1) / BM);

    const int sms = sm_count();
    const int64_t slot_tiles_ub = (n_slots + BN - 1) / BN + (n_experts < n_slots ? n_experts : n_slots);
    const int64_t tiles_ub = slot_tiles_ub * ga.row_tiles;
    const dim3 grid(static_cast<unsigned>(tiles_ub < sms ? tiles_ub : sms));
    const dim3 block(THREADS);
    if (dots) {
        if (int st = set_smem_limit(reinterpret_cast<const void*>(moe_gemm_tc_kernel<true>), SMEM_BYTES)) return st;
        moe_gemm_tc_kernel<true><<<grid, block, SMEM_BYTES, s>>>(wmap, ga);
        return check_launch("moe_gemm_tc_kernel<dump>", grid, block, SMEM_BYTES);
    }
    if (int st = set_smem_limit(reinterpret_cast<const void*>(moe_gemm_tc_kernel<false>), SMEM_BYTES)) return st;
    moe_gemm_tc_kernel<false><<<grid, block, SMEM_BYTES, s>>>(wmap, ga);
    return check_launch("moe_gemm_tc_kernel", grid, block, SMEM_BYTES);
}

}  // namespace ft
