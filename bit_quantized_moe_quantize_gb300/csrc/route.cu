// Router: stable counting sort of the flat (token, top-k) slots by expert id.
//
// Produces counts[E], offsets[E+1] with a leading 0 (nvfp4-megamoe-kernel
// CURRENT_BUG.md, Bug 4: the grouped GEMM takes expert_offsets[1:E+1]) and
// the padding-free permutation perm[S]: perm[offsets[e] + r] is the r-th slot
// of expert e in ascending slot order.  Positions in [offsets[e],
// offsets[e+1]) belong to e, the searchsorted(right=True) map of Bug 2, so
// empty experts own no position.  The same pass also writes, per matmul path,
// the prefix over experts of the number of slot tiles (ceil(count / group)),
// which lets the matmul kernels enumerate their tiles on the device.
//
// A fixed number of launches for a given shape, whatever the data: no host
// read-back, no allocation, nothing that depends on device values on the
// host side, so the router can be captured in a CUDA graph (CURRENT_BUG.md,
// "Cudagraph Constraints").  No atomics on global counters: each warp owns a
// chunk of 256 slots and a private histogram row, so every result is
// deterministic.
//
//   1. route_hist:    per chunk, histogram of expert ids -> hist[chunk][e]
//   2. route_scan:    one CTA: counts, offsets, tile prefixes, and hist
//                     rewritten in place as each chunk's first position per e
//   3. route_scatter: per chunk, stable placement with __match_any_sync ranks
//
// Batches of at most 32 chunks whose histograms fit in shared memory run the
// same three steps inside one CTA (route_small_kernel), with the histogram in
// shared memory: one launch instead of three, which is most of the routing
// time when the batch is small.  Decode-sized batches (at most 512 slots) run
// them in a single warp (route_warp_kernel), with no CTA-wide barrier.
#include <mutex>

#include "ft_common.cuh"
#include "ft_internal.h"

namespace ft {

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Step 1 for one warp and its chunk: histogram of the chunk's expert ids in
// row[E] (shared memory), bad ids flagged in err.
__device__ void route_hist_chunk(const int32_t* __restrict__ ids, int64_t n_slots, int32_t n_experts, int64_t chunk,
                                 int32_t* row, uint32_t* err, int32_t expert_start, int32_t n_global) {
    const uint32_t lane = lane_id();
    for (int32_t e = lane; e < n_experts; e += 32) row[e] = 0;
    __syncwarp();
    bool saw_bad = false;
    for (int step = 0; step < kRouteChunk / 32; ++step) {
        const int64_t s = chunk * kRouteChunk + step * 32 + lane;
        const int32_t g = s < n_slots ? ids[s] : -1;              // global expert id
        const int64_t el = static_cast<int64_t>(g) - expert_start;  // routed expert (this shard's numbering)
        const bool valid = s < n_slots && el >= 0 && el < n_experts;
        const int32_t e = static_cast<int32_t>(el);
        saw_bad |= (s < n_slots) && (g < 0 || g >= n_global);     // only ids no shard owns are errors
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
        if (valid && lane == static_cast<uint32_t>(__ffs(peers) - 1)) row[e] += __popc(peers);
        __syncwarp();
    }
    if (__any_sync(0xFFFFFFFFu, saw_bad) && lane == 0) atomicOr(err, FT_DEVERR_BAD_EXPERT_ID);
    __syncwarp();
}

__global__ void __launch_bounds__(32 * kRouteWarps)
    route_hist_kernel(const int32_t* __restrict__ ids, int64_t n_slots, int32_t n_experts, int64_t n_chunks,
                      int32_t* __restrict__ hist, uint32_t* err, int32_t expert_start, int32_t n_global) {
    extern __shared__ int32_t sh_hist[];
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
    if (chunk >= n_chunks) return;
    int32_t* row = sh_hist + static_cast<int64_t>(warp) * n_experts;
    route_hist_chunk(ids, n_slots, n_experts, chunk, row, err, expert_start, n_global);
    int32_t* grow = hist + chunk * n_experts;
    for (int32_t e = lane; e < n_experts; e += 32) grow[e] = row[e];
}

// Exclusive scan of v[0..n) in shared memory by the whole CTA (blockDim 1024);
// returns the total.  scratch holds 32 ints.
__device__ int32_t block_exclusive_scan(int32_t* v, int32_t n, int32_t* scratch) {
    const int32_t tid = threadIdx.x, nt = blockDim.x;
    const int32_t per = (n + nt - 1) / nt;
    const int32_t lo = min(n, tid * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int32_t i = lo; i < hi; ++i) local += v[i];
    // inclusive warp scan of the per-thread sums
    const uint32_t lane = lane_id(), warp = tid >> 5;
    int32_t inc = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= static_cast<uint32_t>(o)) inc += y;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int32_t nw = nt >> 5;
        int32_t w = lane < static_cast<uint32_t>(nw) ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= static_cast<uint32_t>(o)) w += y;
        }
        if (lane < static_cast<uint32_t>(nw)) scratch[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int32_t total = scratch[(nt >> 5) - 1];
    int32_t run = inc - local + (warp > 0 ? scratch[warp - 1] : 0);
    for (int32_t i = lo; i < hi; ++i) {
        const int32_t x = v[i];
        v[i] = run;
        run += x;
    }
    __syncthreads();
    return total;
}

// Step 2 by one CTA of 1024 threads on hist[n_chunks][E] (global or shared
// memory).  sh: part[P][E] + tot[E] + tiles[E] + 32 ints.
__device__ void route_scan_body(int32_t* hist, int64_t n_chunks, int32_t n_experts, int32_t* __restrict__ counts,
                                int32_t* __restrict__ offsets, int32_t* __restrict__ tiles_gemv, int32_t gemv_group,
                                int32_t* __restrict__ tiles_gemm, int32_t gemm_group, int32_t* sh) {
    const int32_t E = n_experts, nt = blockDim.x, tid = threadIdx.x;
    const int32_t P = E >= nt ? 1 : nt / E;                 // parts per expert
    int32_t* part = sh;                                     // [P][E]
    int32_t* tot = part + static_cast<int64_t>(P) * E;      // [E]
    int32_t* tl = tot + E;                                  // [E]
    int32_t* scratch = tl + E;                              // [32]
    const int64_t per = (n_chunks + P - 1) / P;

    // pass 1: partial sums over chunk ranges
    for (int32_t idx = tid; idx < P * E; idx += nt) {
        const int32_t e = idx % E, p = idx / E;
        const int64_t c0 = p * per, c1 = min(n_chunks, c0 + per);
        int32_t acc = 0;
        for (int64_t c = c0; c < c1; ++c) acc += hist[c * E + e];
        part[p * E + e] = acc;
    }
    __syncthreads();
    // per expert: exclusive prefix over parts, and the total
    for (int32_t e = tid; e < E; e += nt) {
        int32_t run = 0;
        for (int32_t p = 0; p < P; ++p) {
            const int32_t x = part[p * E + e];
            part[p * E + e] = run;
            run += x;
        }
        tot[e] = run;
        counts[e] = run;
    }
    __syncthreads();
    // tile counts per path, before tot is overwritten by its scan
    if (tiles_gemv)
        for (int32_t e = tid; e < E; e += nt) tl[e] = (tot[e] + gemv_group - 1) / gemv_group;
    __syncthreads();
    if (tiles_gemv) {
        const int32_t t = block_exclusive_scan(tl, E, scratch);
        for (int32_t e = tid; e < E; e += nt) tiles_gemv[e] = tl[e];
        if (tid == 0) tiles_gemv[E] = t;
    }
    __syncthreads();
    if (tiles_gemm)
        for (int32_t e = tid; e < E; e += nt) tl[e] = (tot[e] + gemm_group - 1) / gemm_group;
    __syncthreads();
    if (tiles_gemm) {
        const int32_t t = block_exclusive_scan(tl, E, scratch);
        for (int32_t e = tid; e < E; e += nt) tiles_gemm[e] = tl[e];
        if (tid == 0) tiles_gemm[E] = t;
    }
    __syncthreads();
    const int32_t total = block_exclusive_scan(tot, E, scratch);
    for (int32_t e = tid; e < E; e += nt) offsets[e] = tot[e];
    if (tid == 0) offsets[E] = total;
    __syncthreads();
    // pass 2: hist[c][e] := first position of chunk c's slots of expert e
    for (int32_t idx = tid; idx < P * E; idx += nt) {
        const int32_t e = idx % E, p = idx / E;
        const int64_t c0 = p * per, c1 = min(n_chunks, c0 + per);
        int32_t run = tot[e] + part[p * E + e];
        for (int64_t c = c0; c < c1; ++c) {
            const int32_t x = hist[c * E + e];
            hist[c * E + e] = run;
            run += x;
        }
    }
}

// One CTA of 1024 threads.  Shared: part[P][E] + tot[E] + tiles[E] + 32.
__global__ void __launch_bounds__(1024)
    route_scan_kernel(int32_t* __restrict__ hist, int64_t n_chunks, int32_t n_experts, int32_t* __restrict__ counts,
                      int32_t* __restrict__ offsets, int32_t* __restrict__ tiles_gemv, int32_t gemv_group,
                      int32_t* __restrict__ tiles_gemm, int32_t gemm_group) {
    extern __shared__ int32_t sh[];
    route_scan_body(hist, n_chunks, n_experts, counts, offsets, tiles_gemv, gemv_group, tiles_gemm, gemm_group, sh);
}

// Step 3 for one warp and its chunk: cur[E] (shared memory) starts as the
// chunk's first position per expert.
__device__ void route_scatter_chunk(const int32_t* __restrict__ ids, int64_t n_slots, int32_t n_experts,
                                    int64_t chunk, int32_t* cur, int32_t* __restrict__ perm,
                                    uint32_t* __restrict__ zero_rows, int64_t row_words, int32_t expert_start) {
    const uint32_t lane = lane_id();
    for (int step = 0; step < kRouteChunk / 32; ++step) {
        const int64_t s = chunk * kRouteChunk + step * 32 + lane;
        const int64_t el = static_cast<int64_t>(s < n_slots ? ids[s] : -1) - expert_start;
        const bool valid = s < n_slots && el >= 0 && el < n_experts;
        const int32_t e = static_cast<int32_t>(el);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
        int32_t pos = 0;
        if (valid) pos = cur[e] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (valid && lane == static_cast<uint32_t>(__ffs(peers) - 1)) cur[e] += __popc(peers);
        if (valid) perm[pos] = static_cast<int32_t>(s);
        if (!valid && s < n_slots && zero_rows != nullptr) {
            uint32_t* row = zero_rows + s * row_words;
            for (int64_t r = 0; r < row_words; ++r) row[r] = 0u;
        }
        __syncwarp();
    }
}

// Positions past the valid slots are -1 (threads tid, tid + nt, ...).
__device__ __forceinline__ void route_perm_tail(const int32_t* __restrict__ offsets, int32_t n_experts,
                                                int64_t n_slots, int32_t* __restrict__ perm, int64_t tid, int64_t nt) {
    const int64_t n_valid = offsets[n_experts];
    for (int64_t p = n_valid + tid; p < n_slots; p += nt) perm[p] = -1;
}

__global__ void __launch_bounds__(32 * kRouteWarps)
    route_scatter_kernel(const int32_t* __restrict__ ids, int64_t n_slots, int32_t n_experts, int64_t n_chunks,
                         const int32_t* __restrict__ base, const int32_t* __restrict__ offsets,
                         int32_t* __restrict__ perm, uint32_t* __restrict__ zero_rows, int64_t row_words,
                         int32_t expert_start) {
    extern __shared__ int32_t sh_cursor[];
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    route_perm_tail(offsets, n_experts, n_slots, perm, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                    static_cast<int64_t>(gridDim.x) * blockDim.x);
    const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
    if (chunk >= n_chunks) return;
    int32_t* cur = sh_cursor + static_cast<int64_t>(warp) * n_experts;
    const int32_t* brow = base + chunk * n_experts;
    for (int32_t e = lane; e < n_experts; e += 32) cur[e] = brow[e];
    __syncwarp();
    route_scatter_chunk(ids, n_slots, n_experts, chunk, cur, perm, zero_rows, row_words, expert_start);
}

// All three steps in one CTA of 1024 threads (32 warps, one chunk each) for
// n_chunks <= 32.  Shared: hist[n_chunks][E], then the scan's part/tot/tiles.
__global__ void __launch_bounds__(1024)
    route_small_kernel(const int32_t* __restrict__ ids, int64_t n_slots, int32_t n_experts, int64_t n_chunks,
                       int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                       int32_t* __restrict__ tiles_gemv, int32_t gemv_group, int32_t* __restrict__ tiles_gemm,
                       int32_t gemm_group, uint32_t* err, uint32_t* __restrict__ zero_rows, int64_t row_words,
                       int32_t expert_start, int32_t n_global) {
    extern __shared__ int32_t sh_small[];
    int32_t* hist = sh_small;                                            // [n_chunks][E]
    int32_t* scan_sh = sh_small + n_chunks * static_cast<int64_t>(n_experts);
    const uint32_t warp = threadIdx.x >> 5;
    if (warp < n_chunks)
        route_hist_chunk(ids, n_slots, n_experts, warp, hist + warp * n_experts, err, expert_start, n_global);
    __syncthreads();
    route_scan_body(hist, n_chunks, n_experts, counts, offsets, tiles_gemv, gemv_group, tiles_gemm, gemm_group,
                    scan_sh);
    __syncthreads();
    route_perm_tail(offsets, n_experts, n_slots, perm, threadIdx.x, blockDim.x);
    if (warp < n_chunks)
        route_scatter_chunk(ids, n_slots, n_experts, warp, hist + warp * n_experts, perm, zero_rows, row_words,
                            expert_start);
}

// All three steps in ONE warp, for decode-sized batches (S <= kRouteWarpSlots,
// E <= kRouteWarpExperts): the histogram and the scatter cursors live in
// shared memory, the scans are warp scans over each lane's contiguous range
// of experts, and nothing waits on a CTA-wide barrier.  The slot ids stay in
// registers between the histogram and the scatter.  Same outputs, bit for
// bit, as the multi-warp kernels.
constexpr int kRouteWarpSlots = 512;
constexpr int kRouteWarpExperts = 2048;

__device__ __forceinline__ int32_t warp_inclusive_scan(int32_t v) {
    const uint32_t lane = lane_id();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= static_cast<uint32_t>(o)) v += y;
    }
    return v;
}

__global__ void __launch_bounds__(32)
    route_warp_kernel(const int32_t* __restrict__ ids, int32_t n_slots, int32_t n_experts,
                      int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                      int32_t* __restrict__ tiles_gemv, int32_t gemv_group, int32_t* __restrict__ tiles_gemm,
                      int32_t gemm_group, uint32_t* err, uint32_t* __restrict__ zero_rows, int64_t row_words,
                      int32_t expert_start, int32_t n_global) {
    extern __shared__ int32_t sh_warp[];
    int32_t* cnt = sh_warp;                 // [E]
    int32_t* cur = sh_warp + n_experts;     // [E]
    constexpr int STEPS = kRouteWarpSlots / 32;
    const uint32_t lane = lane_id();
    for (int32_t e = lane; e < n_experts; e += 32) cnt[e] = 0;
    __syncwarp();
    int32_t el[STEPS];
    bool saw_bad = false;
#pragma unroll
    for (int step = 0; step < STEPS; ++step) {
        const int32_t s = step * 32 + static_cast<int32_t>(lane);
        el[step] = -1;
        if (step * 32 < n_slots) {                                   // warp-uniform
            const int32_t g = s < n_slots ? ids[s] : -1;
            const int64_t x = static_cast<int64_t>(g) - expert_start;
            const bool valid = s < n_slots && x >= 0 && x < n_experts;
            saw_bad |= (s < n_slots) && (g < 0 || g >= n_global);
            el[step] = valid ? static_cast<int32_t>(x) : -1;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, el[step]);
            if (valid && lane == static_cast<uint32_t>(__ffs(peers) - 1)) cnt[el[step]] += __popc(peers);
            __syncwarp();
        }
    }
    if (__any_sync(0xFFFFFFFFu, saw_bad) && lane == 0) atomicOr(err, FT_DEVERR_BAD_EXPERT_ID);
    // exclusive scans over experts: lane l owns the contiguous range [lo, hi)
    const int32_t per = (n_experts + 31) / 32;
    const int32_t lo = min(n_experts, static_cast<int32_t>(lane) * per), hi = min(n_experts, lo + per);
    int32_t sc = 0, sv = 0, sm = 0;
    for (int32_t e = lo; e < hi; ++e) {
        const int32_t c = cnt[e];
        sc += c;
        sv += (c + gemv_group - 1) / gemv_group;
        sm += (c + gemm_group - 1) / gemm_group;
    }
    int32_t rc = warp_inclusive_scan(sc) - sc, rv = warp_inclusive_scan(sv) - sv, rm = warp_inclusive_scan(sm) - sm;
    for (int32_t e = lo; e < hi; ++e) {
        const int32_t c = cnt[e];
        counts[e] = c;
        offsets[e] = rc;
        cur[e] = rc;
        if (tiles_gemv) tiles_gemv[e] = rv;
        if (tiles_gemm) tiles_gemm[e] = rm;
        rc += c;
        rv += (c + gemv_group - 1) / gemv_group;
        rm += (c + gemm_group - 1) / gemm_group;
    }
    if (lane == 31) {
        offsets[n_experts] = rc;
        if (tiles_gemv) tiles_gemv[n_experts] = rv;
        if (tiles_gemm) tiles_gemm[n_experts] = rm;
    }
    const int32_t n_valid = __shfl_sync(0xFFFFFFFFu, rc, 31);
    __syncwarp();
    // stable scatter: equal ids ranked by lane within each step of 32 slots
#pragma unroll
    for (int step = 0; step < STEPS; ++step) {
        const int32_t s = step * 32 + static_cast<int32_t>(lane);
        if (step * 32 < n_slots) {
            const bool valid = el[step] >= 0;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, el[step]);
            int32_t pos = 0;
            if (valid) pos = cur[el[step]] + __popc(peers & lanemask_lt());
            __syncwarp();
            if (valid && lane == static_cast<uint32_t>(__ffs(peers) - 1)) cur[el[step]] += __popc(peers);
            if (valid) perm[pos] = s;
            if (!valid && s < n_slots && zero_rows != nullptr) {
                uint32_t* row = zero_rows + static_cast<int64_t>(s) * row_words;
                for (int64_t r = 0; r < row_words; ++r) row[r] = 0u;
            }
            __syncwarp();
        }
    }
    for (int32_t p = n_valid + static_cast<int32_t>(lane); p < n_slots; p += 32) perm[p] = -1;
}

int launch_route(const int32_t* ids, int64_t n_slots, int32_t n_experts, const RouteBuffers& b,
                 int32_t gemv_group, int32_t gemm_group, uint32_t* zero_rows, int64_t row_words, cudaStream_t s) {
    {
        const int big = 160 * 1024;
        if (int st = set_smem_limit(reinterpret_cast<const void*>(route_hist_kernel), big)) return st;
        if (int st = set_smem_limit(reinterpret_cast<const void*>(route_scan_kernel), big)) return st;
        if (int st = set_smem_limit(reinterpret_cast<const void*>(route_scatter_kernel), big)) return st;
    }
    const int64_t n_chunks = route_chunks(n_slots);
    const int32_t start = b.expert_start, n_global = b.n_global > 0 ? b.n_global : n_experts;
    const int32_t P = n_experts >= 1024 ? 1 : 1024 / n_experts;
    const size_t scan_sm = (static_cast<size_t>(P) * n_experts + 2 * static_cast<size_t>(n_experts) + 32) *
                           sizeof(int32_t);
    if (n_slots <= kRouteWarpSlots && n_experts <= kRouteWarpExperts) {
        const size_t sm = 2 * static_cast<size_t>(n_experts) * sizeof(int32_t);
        route_warp_kernel<<<1, 32, sm, s>>>(ids, static_cast<int32_t>(n_slots), n_experts, b.counts, b.offsets, b.perm,
                                            b.tiles_gemv, gemv_group, b.tiles_gemm, gemm_group, b.err, zero_rows,
                                            row_words, start, n_global);
        return check_launch("route_warp_kernel", dim3(1), dim3(32), sm);
    }
    if (n_chunks <= 32 && n_chunks * n_experts <= 16384) {
        const size_t sm = static_cast<size_t>(n_chunks) * n_experts * sizeof(int32_t) + scan_sm;
        if (int st = set_smem_limit(reinterpret_cast<const void*>(route_small_kernel), static_cast<int>(sm))) return st;
        route_small_kernel<<<1, 1024, sm, s>>>(ids, n_slots, n_experts, n_chunks, b.counts, b.offsets, b.perm,
                                               b.tiles_gemv, gemv_group, b.tiles_gemm, gemm_group, b.err, zero_rows,
                                               row_words, start, n_global);
        return check_launch("route_small_kernel", dim3(1), dim3(1024), sm);
    }
    const int64_t ctas = (n_chunks + kRouteWarps - 1) / kRouteWarps;
    const dim3 block(32 * kRouteWarps);
    const size_t sm_rows = static_cast<size_t>(kRouteWarps) * n_experts * sizeof(int32_t);
    if (ctas > 0) {
        const dim3 grid(static_cast<unsigned>(ctas));
        route_hist_kernel<<<grid, block, sm_rows, s>>>(ids, n_slots, n_experts, n_chunks, b.hist, b.err, start,
                                                       n_global);
        if (int st = check_launch("route_hist_kernel", grid, block, sm_rows)) return st;
    }
    route_scan_kernel<<<1, 1024, scan_sm, s>>>(b.hist, n_chunks, n_experts, b.counts, b.offsets, b.tiles_gemv,
                                               gemv_group, b.tiles_gemm, gemm_group);
    if (int st = check_launch("route_scan_kernel", dim3(1), dim3(1024), scan_sm)) return st;
    if (ctas > 0) {
        const dim3 grid(static_cast<unsigned>(ctas));
        route_scatter_kernel<<<grid, block, sm_rows, s>>>(ids, n_slots, n_experts, n_chunks, b.hist, b.offsets,
                                                          b.perm, zero_rows, row_words, start);
        if (int st = check_launch("route_scatter_kernel", grid, block, sm_rows)) return st;
    }
    return FT_OK;
}

// --------------------------------------------------- allocation-free router
// For callers that must not allocate device memory (see
// ft_moe_route_offsets_noalloc in ft_moe.h): the histogram scratch is this
// fixed array, plus one word that receives bad-id flags when the caller
// passes no error word.  Host code must not use the array's name as a
// pointer - on the host it is only a stand-in for the symbol - so its device
// address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) int32_t g_route_noalloc_scratch[FT_ROUTE_NOALLOC_SCRATCH_WORDS + 64];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
int32_t* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
int noalloc_scratch(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(FT_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fail(FT_ERR_CUDA, "cudaGetSymbolAddress(route scratch): %s", cudaGetErrorString(e));
        g_noalloc_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_addr[dev];
    return FT_OK;
}
}  // namespace

}  // namespace ft

extern "C" int ft_moe_route_offsets_noalloc(const int32_t* topk_ids, int64_t tokens, int32_t top_k,
                                            int32_t n_experts, int32_t* counts, int32_t* offsets, int32_t* perm,
                                            uint32_t* dev_err, void* stream) {
    using namespace ft;
    if (tokens < 0) return fail(FT_ERR_ARG, "tokens must be >= 0 (got %lld)", (long long)tokens);
    if (n_experts < 1 || n_experts > FT_MAX_EXPERTS)
        return fail(FT_ERR_ARG, "n_experts must be in [1, %d] (got %d)", FT_MAX_EXPERTS, n_experts);
    if (top_k < 1 || top_k > n_experts)
        return fail(FT_ERR_ARG, "top_k must be in [1, n_experts=%d] (got %d)", n_experts, top_k);
    if (tokens > INT32_MAX / top_k)
        return fail(FT_ERR_SIZE, "tokens * top_k = %lld * %d must be < 2^31", (long long)tokens, top_k);
    const int64_t n_slots = tokens * top_k;
    const int64_t words = route_chunks(n_slots) * static_cast<int64_t>(n_experts);
    if (words > FT_ROUTE_NOALLOC_SCRATCH_WORDS)
        return fail(FT_ERR_SIZE,
                    "ft_moe_route_offsets_noalloc: %lld slots and %d experts need %lld scratch words, more than the "
                    "%d built into the library; use ft_moe_route_offsets",
                    (long long)n_slots, n_experts, (long long)words, FT_ROUTE_NOALLOC_SCRATCH_WORDS);
    if (!counts || !offsets || (n_slots > 0 && (!topk_ids || !perm))) return fail(FT_ERR_ARG, "null pointer");
    if ((reinterpret_cast<uintptr_t>(topk_ids) | reinterpret_cast<uintptr_t>(counts) |
         reinterpret_cast<uintptr_t>(offsets) | reinterpret_cast<uintptr_t>(perm)) & 3u)
        return fail(FT_ERR_ALIGN, "int32 arrays must be 4-byte aligned");
    int32_t* scratch = nullptr;
    if (int st = noalloc_scratch(&scratch)) return st;
    RouteBuffers rb{};
    rb.counts = counts;
    rb.offsets = offsets;
    rb.perm = perm;
    rb.hist = scratch;
    rb.tiles_gemv = nullptr;
    rb.tiles_gemm = nullptr;
    rb.err = dev_err ? dev_err : reinterpret_cast<uint32_t*>(scratch + FT_ROUTE_NOALLOC_SCRATCH_WORDS);
    return launch_route(topk_ids, n_slots, n_experts, rb, 1, 1, nullptr, 0, static_cast<cudaStream_t>(stream));
}

