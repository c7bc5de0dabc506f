// Pieces of the expert-grouped GEMM path: the kernel arguments, the tile
// decode over the router's tile prefix, the nibble -> fp16 conversion, the
// drain's scale layout and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "ft_common.cuh"
#include "ft_internal.h"

namespace ft {

struct GemmArgs {
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
    // layer 1 with the gated activation in the epilogue (act_mid != nullptr):
    // the weight rows are n_inter gate rows then n_inter up rows per expert,
    // and the epilogue writes Q8_1 rows of act(gate) * up to act_mid
    uint8_t* act_mid;
    int64_t n_inter;
    int32_t act_kind;
};

struct TileInfo {
    int32_t e;
    int64_t p0;
    int32_t nvalid;
    int64_t m0;
};

// Work item w -> (expert e, first router position p0 of its slot tile, valid
// slots in the tile, first weight row m0).  The slot tile is found as the
// largest e with tiles[e] <= st, i.e. searchsorted(right=True) over the tile
// prefix (nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 2), so empty experts own
// no tile.
template <int BN>
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
    ti.p0 = static_cast<int64_t>(a.offsets[lo]) + (st - a.tiles[lo]) * BN;
    ti.nvalid = static_cast<int32_t>(min(static_cast<int64_t>(BN), a.offsets[lo + 1] - ti.p0));
    ti.m0 = mt * kGemmBM;
    return ti;
}

// Four packed nibble bytes -> two fp16x2 words holding (nibble - OFF), in order
// (OFF 8 for Q4_0, 0 for the K-quants' levels).  0x64nn is the fp16 1024 + nn,
// so one subtraction of 1024 + OFF gives nn - OFF exactly.
template <int OFF = 8>
__device__ __forceinline__ void nib4_to_h2(uint32_t nib, uint32_t& lo, uint32_t& hi) {
    static_assert(OFF >= 0 && OFF < 256, "level offset");
    const __half2 bias = __halves2half2(__ushort_as_half(0x6400 + OFF), __ushort_as_half(0x6400 + OFF));
    uint32_t a = __byte_perm(nib, 0x64646464u, 0x4140u);
    uint32_t b = __byte_perm(nib, 0x64646464u, 0x4342u);
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

// Position of slot c (0 <= c < BN) of a block's fp32 activation scales in the
// drain's read order: for each group of CW columns and each column-pair index
// q = (c % 8) / 2, a run of CW/4 floats {d_a[8 i + 2 q + e]} at a pitch of
// CW/4 + 4 floats, so that the four 16-byte reads a warp's lane quads issue at
// once fall in four different bank groups.
template <int CW>
__device__ __forceinline__ uint32_t da_index(uint32_t c) {
    constexpr uint32_t QP = CW / 4 + 4;
    const uint32_t cc = c % CW;
    return (c / CW) * (4 * QP) + ((cc & 7u) >> 1) * QP + (cc >> 3) * 2 + (cc & 1u);
}

// 2-D tensor map over a row-major array (inner extent `inner` elements, rows
// `row_bytes` apart), box box_inner x box_outer.
int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz, const char* what);

}  // namespace ft
