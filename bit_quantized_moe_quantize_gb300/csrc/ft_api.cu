// C ABI of libft_moe.so: argument validation, workspace, path dispatch and
// launch checks around the kernels.  See include/ft_moe.h for the contract.
//
// Every size product is formed in 64-bit (mlxcel PR #652, "Fix": the int32
// product m * n that overflowed and yielded a zero grid), and every kernel
// launch is followed by a check of its status that names the kernel and its
// grid (FreeToken PR #185, "Fix": FT_MOE_VEC_LAUNCH_CHECK after each launch,
// so a rejected geometry is reported where it happens instead of by the next
// unrelated CUDA call).
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "../../include/ft_moe.h"
#include "ft_internal.h"

namespace ft {

static thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

// ---------------------------------------------------------------- profiling
struct Prof {
    std::mutex mu;
    bool on = false;
    int max_calls = 0;
    cudaEvent_t* ev = nullptr;       // [max_calls][5]: quant b/e, route b, matmul b/e
    int n_quant = 0, n_mm = 0;
    bool quant_open = false, mm_open = false;
    int64_t launches = 0;
};
static Prof g_prof;

void prof_count_launch() {
    if (g_prof.on) {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        ++g_prof.launches;
    }
}

void prof_mark(ProfPoint p, cudaStream_t s) {
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    Prof& P = g_prof;
    switch (p) {
        case kProfQuantBegin:
            if (P.n_quant < P.max_calls) {
                cudaEventRecord(P.ev[P.n_quant * 5 + 0], s);
                P.quant_open = true;
            }
            break;
        case kProfQuantEnd:
            if (P.quant_open) {
                cudaEventRecord(P.ev[P.n_quant * 5 + 1], s);
                P.quant_open = false;
                ++P.n_quant;
            }
            break;
        case kProfRouteBegin:
            if (P.n_mm < P.max_calls) {
                cudaEventRecord(P.ev[P.n_mm * 5 + 2], s);
                P.mm_open = true;
            }
            break;
        case kProfMatmulBegin:
            if (P.mm_open) cudaEventRecord(P.ev[P.n_mm * 5 + 3], s);
            break;
        case kProfMatmulEnd:
            if (P.mm_open) {
                cudaEventRecord(P.ev[P.n_mm * 5 + 4], s);
                P.mm_open = false;
                ++P.n_mm;
            }
            break;
    }
}

int check_launch(const char* kernel, dim3 grid, dim3 block, size_t smem) {
    prof_count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return FT_OK;
    return fail(FT_ERR_LAUNCH, "launch of %s failed: %s (grid %u x %u x %u, block %u x %u x %u, smem %zu)", kernel,
                cudaGetErrorString(e), grid.x, grid.y, grid.z, block.x, block.y, block.z, smem);
}

static int cuda_fail(cudaError_t e, const char* what) {
    return fail(FT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static std::mutex g_attr_mu;

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

int set_smem_limit(const void* kernel, int bytes) {
    struct Entry {
        const void* k;
        int dev;
        int bytes;
    };
    static Entry done[256];
    static int n_done = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_attr_mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].k == kernel && done[i].dev == dev && done[i].bytes >= bytes) return FT_OK;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    for (int i = 0; i < n_done; ++i)
        if (done[i].k == kernel && done[i].dev == dev) {
            done[i].bytes = bytes;
            return FT_OK;
        }
    if (n_done < 256) done[n_done++] = Entry{kernel, dev, bytes};
    return FT_OK;
}

// ------------------------------------------------------------- validation
static bool mul_ok(int64_t a, int64_t b, int64_t* r) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *r = a * b;
    return true;
}

struct Shape {
    int64_t tokens, n_slots, nrows, ncols, nb;
    int32_t top_k, n_experts;
    int32_t act_div;   // activation row of slot s: s / act_div (top_k: one row per token; 1: one per slot)
    // expert-parallel shard: ids are global in [0, n_global); this call holds
    // experts [expert_start, expert_start + n_experts) (0 and n_experts otherwise)
    int32_t expert_start, n_global;
    int32_t wtype;     // FT_TYPE_* of the weights
    // routed slots per held expert on average (what the tile plans go by)
    double mean() const { return static_cast<double>(n_slots) / n_global; }
};

// Checks the routing arguments; fills n_slots.
static int check_route_args(int64_t tokens, int32_t top_k, int32_t n_experts, Shape* sh) {
    if (tokens < 0) return fail(FT_ERR_ARG, "tokens must be >= 0 (got %lld)", (long long)tokens);
    if (n_experts < 1 || n_experts > FT_MAX_EXPERTS)
        return fail(FT_ERR_ARG, "n_experts must be in [1, %d] (got %d)", FT_MAX_EXPERTS, n_experts);
    if (top_k < 1 || top_k > n_experts)
        return fail(FT_ERR_ARG, "top_k must be in [1, n_experts=%d] (got %d)", n_experts, top_k);
    int64_t s;
    if (!mul_ok(tokens, top_k, &s) || s > INT32_MAX)
        return fail(FT_ERR_SIZE, "tokens * top_k = %lld * %d must be < 2^31", (long long)tokens, top_k);
    sh->tokens = tokens;
    sh->top_k = top_k;
    sh->n_experts = n_experts;
    sh->n_slots = s;
    sh->act_div = top_k;
    sh->expert_start = 0;
    sh->n_global = n_experts;
    sh->wtype = FT_TYPE_Q4_0;
    return FT_OK;
}

static int check_matmul_args(int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols,
                             Shape* sh) {
    if (int st = check_route_args(tokens, top_k, n_experts, sh)) return st;
    if (ncols <= 0 || ncols % 32 != 0)
        return fail(FT_ERR_ARG, "ncols must be a positive multiple of 32 (got %lld)", (long long)ncols);
    if (ncols > FT_MAX_NCOLS) return fail(FT_ERR_SIZE, "ncols must be <= %d (got %lld)", FT_MAX_NCOLS, (long long)ncols);
    if (nrows <= 0) return fail(FT_ERR_ARG, "nrows must be > 0 (got %lld)", (long long)nrows);
    int64_t en, wbytes, obytes;
    if (!mul_ok(n_experts, nrows, &en) || en > INT32_MAX)
        return fail(FT_ERR_SIZE, "n_experts * nrows must be < 2^31");
    if (!mul_ok(en, (ncols / 32) * 34, &wbytes)) return fail(FT_ERR_SIZE, "weight size overflows int64");
    if (!mul_ok(sh->n_slots, nrows, &obytes) || obytes > INT64_MAX / 4)
        return fail(FT_ERR_SIZE, "output size overflows int64");
    sh->nrows = nrows;
    sh->ncols = ncols;
    sh->nb = ncols / 32;
    return FT_OK;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static int get_stream_capturing(cudaStream_t s, bool* capturing) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    *capturing = cs != cudaStreamCaptureStatusNone;
    return FT_OK;
}

// -------------------------------------------------------------- workspace
// Per device: one cudaMalloc'ed block.  Layout (each part 256-byte aligned):
//   err word | counts[E] | offsets[E+1] | perm[S] | tiles_gemv[E+1] |
//   tiles_gemm[E+1] | hist[nchunks][E] | (tensor-core path only:)
//   xh[S_pad][ncols] fp16 | da[S_pad][ncols/32] fp16 | (Q4_K weights there:)
//   sa[S_pad][ncols/32] fp32 | (layer 1 with the
//   activation fused, on the GEMV path:) h[S][2 n_inter] fp32 | (the fp16
//   entry point, unless it runs in one launch:) act[T][ncols/32] Q8_1
struct WsLayout {
    size_t err, counts, offsets, perm, tiles_gemv, tiles_gemm, hist, xh, da, sa, h, act, total;
};

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

static WsLayout ws_layout(int64_t n_slots, int32_t n_experts, int64_t gemm_ncols = 0, size_t h_bytes = 0,
                          size_t act_bytes = 0, bool gemm_sums = false) {
    WsLayout L{};
    size_t o = 0;
    L.err = o;
    o = al256(o + 4);
    L.counts = o;
    o = al256(o + 4 * static_cast<size_t>(n_experts));
    L.offsets = o;
    o = al256(o + 4 * (static_cast<size_t>(n_experts) + 1));
    L.perm = o;
    o = al256(o + 4 * static_cast<size_t>(n_slots));
    L.tiles_gemv = o;
    o = al256(o + 4 * (static_cast<size_t>(n_experts) + 1));
    L.tiles_gemm = o;
    o = al256(o + 4 * (static_cast<size_t>(n_experts) + 1));
    L.hist = o;
    o = al256(o + 4 * static_cast<size_t>(route_chunks(n_slots)) * n_experts);
    const size_t rows = gemm_ncols ? static_cast<size_t>(gemm_rows(n_slots)) : 0;
    L.xh = o;
    o = al256(o + 2 * rows * static_cast<size_t>(gemm_ncols));
    L.da = o;
    o = al256(o + 2 * rows * static_cast<size_t>(gemm_ncols / 32));
    L.sa = o;
    o = al256(o + (gemm_sums ? 4 * rows * static_cast<size_t>(gemm_ncols / 32) : 0));
    L.h = o;
    o = al256(o + h_bytes);
    L.act = o;
    o = al256(o + act_bytes);
    L.total = o;
    return L;
}

// A guard block of kGuardBytes after the end of every workspace, filled with
// kGuardByte when the workspace is allocated and checked by
// ft_moe_read_device_error: a kernel writing past the end of the workspace
// changes it.
constexpr size_t kGuardBytes = 256;
constexpr int kGuardByte = 0xA5;

struct DeviceWs {
    void* base = nullptr;
    size_t bytes = 0;   // usable bytes; the guard block follows them
};

constexpr int kMaxDevices = 64;
static DeviceWs g_ws[kMaxDevices];
static std::mutex g_ws_mu;

static int current_device(int* dev) {
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (*dev < 0 || *dev >= kMaxDevices) return fail(FT_ERR_CUDA, "device ordinal %d out of range", *dev);
    return FT_OK;
}

// Ensures the current device's workspace holds `need` bytes; returns its base.
static int ws_acquire(size_t need, cudaStream_t s, uint8_t** base) {
    int dev;
    if (int st = current_device(&dev)) return st;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    DeviceWs& w = g_ws[dev];
    if (w.bytes < need) {
        bool capturing = false;
        if (int st = get_stream_capturing(s, &capturing)) return st;
        if (capturing)
            return fail(FT_ERR_WORKSPACE,
                        "workspace of %zu bytes needed but %zu reserved, and the stream is being captured; call "
                        "ft_moe_reserve before capture",
                        need, w.bytes);
        if (w.base) {
            cudaError_t e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize before workspace growth");
            cudaFree(w.base);
            w.base = nullptr;
            w.bytes = 0;
        }
        void* p = nullptr;
        cudaError_t e = cudaMalloc(&p, need + kGuardBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
        e = cudaMemset(p, 0, need);
        if (e == cudaSuccess) e = cudaMemset(static_cast<uint8_t*>(p) + need, kGuardByte, kGuardBytes);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFree(p);
            return cuda_fail(e, "cudaMemset(workspace)");
        }
        w.base = p;
        w.bytes = need;
    }
    *base = static_cast<uint8_t*>(w.base);
    return FT_OK;
}

// ------------------------------------------------------------------ paths
static int g_path = -1;   // -1: not yet read from the environment
static std::mutex g_path_mu;

static int path_setting() {
    std::lock_guard<std::mutex> lk(g_path_mu);
    if (g_path < 0) {
        g_path = FT_PATH_AUTO;
        const char* v = std::getenv("FT_MOE_PATH");
        if (v && std::strcmp(v, "gemv") == 0) g_path = FT_PATH_GEMV;
        if (v && std::strcmp(v, "gemm") == 0) g_path = FT_PATH_GEMM;
        if (v && std::strcmp(v, "gemv_dp4a") == 0) g_path = FT_PATH_GEMV_DP4A;
    }
    return g_path;
}

// The tensor-core path loads 8-block weight boxes (rows 16-byte aligned) of
// 128 rows, so it needs ncols % 256 == 0 and at least 128 weight rows overall.
static bool gemm_shape_ok(const Shape& sh) {
    return sh.ncols % 256 == 0 && static_cast<int64_t>(sh.n_experts) * sh.nrows >= kGemmBM;
}

// Host-side choice from the shape only (no device read): the tensor-core path
// pays off once experts see enough slots to fill a 128-column MMA tile.
static bool gemm_type_ok(int wtype) { return wtype == FT_TYPE_Q4_0 || wtype == FT_TYPE_Q4_K; }

// Routed slots per expert on average from which the tensor-core path is
// chosen: 40 where the GEMV would run 16-slot mma.sync tiles (Q4_0 or Q4_K
// whose activation tile fits; measured on Q4_0: those beat the GEMM up to 32
// slots per expert on the three workload shapes by 1.1-1.5x and lose from
// 48), else 16 (the dp4a tiles).
static double gemm_min_mean(const Shape& sh, int setting) {
    if ((sh.wtype != FT_TYPE_Q4_0 && sh.wtype != FT_TYPE_Q4_K) || setting == FT_PATH_GEMV_DP4A) return 16.0;
    const double m = sh.mean() > 16.0 ? sh.mean() : 16.0;
    return plan_gemv(sh.n_slots, sh.n_experts, sh.nrows, sh.ncols, m, sh.wtype, true).mma ? 40.0 : 16.0;
}

static int choose_path(const Shape& sh, int setting) {
    if (setting == FT_PATH_GEMV || setting == FT_PATH_GEMV_DP4A) return FT_PATH_GEMV;
    if (!gemm_type_ok(sh.wtype)) return setting == FT_PATH_GEMM ? FT_PATH_GEMM : FT_PATH_GEMV;
    if (setting == FT_PATH_GEMM) return FT_PATH_GEMM;
    if (!gemm_shape_ok(sh)) return FT_PATH_GEMV;
    return sh.mean() >= gemm_min_mean(sh, setting) ? FT_PATH_GEMM : FT_PATH_GEMV;
}

// Slots above which the GEMV path is never chosen by itself (the tensor-core
// path takes over at gemm_min_mean routed slots per expert on average).
static int64_t gemv_max_slots(const Shape& sh) {
    const int setting = path_setting();
    if (setting == FT_PATH_GEMV || setting == FT_PATH_GEMV_DP4A || !gemm_shape_ok(sh) || !gemm_type_ok(sh.wtype))
        return sh.n_slots;
    const int64_t lim = static_cast<int64_t>(gemm_min_mean(sh, setting)) * sh.n_global;
    return sh.n_slots < lim ? sh.n_slots : lim;
}

// af != nullptr: layer 1 with the gated activation fused (sh.nrows = 2
// af->n_inter, out unused): the tensor-core path applies it in its epilogue;
// the GEMV path writes the layer-1 result to workspace and runs the
// activation/requantize step on it.
// Bytes of the Q8_1 activation rows of a call (T rows of ncols / 32 blocks).
static size_t act_rows_bytes(const Shape& sh) {
    return static_cast<size_t>(sh.tokens) * static_cast<size_t>(sh.nb) * 36;
}

// x16 != nullptr: the activations come as fp16 rows [tokens][ncols] (act is
// unused): a decode-sized batch on the GEMV path runs as one launch that
// routes and quantizes per CTA; anything else quantizes into workspace first.
static int run_matmul(const void* weights, const void* act, const int32_t* topk_ids, float* out, int32_t* dots,
                      const Shape& sh, cudaStream_t s, const ActFuse* af = nullptr, const void* x16 = nullptr) {
    const int path = choose_path(sh, path_setting());
    if (path == FT_PATH_GEMM && !gemm_type_ok(sh.wtype))
        return fail(FT_ERR_ARG, "the tensor-core path takes Q4_0 and Q4_K weights only (weight type %d)", sh.wtype);
    const bool gemm_sums = path == FT_PATH_GEMM && sh.wtype == FT_TYPE_Q4_K;
    if (path == FT_PATH_GEMM && !gemm_shape_ok(sh))
        return fail(FT_ERR_ARG, "the tensor-core path needs ncols %% 256 == 0 and n_experts * nrows >= 128 (got %lld, %lld)",
                    (long long)sh.ncols, (long long)sh.n_experts * sh.nrows);
    const bool h_in_ws = af && path == FT_PATH_GEMV;
    const GemvPlan gp = plan_gemv(sh.n_slots, sh.n_experts, sh.nrows, sh.ncols, sh.mean(), sh.wtype,
                                  path_setting() != FT_PATH_GEMV_DP4A);
    // the one-launch decode step is the row-per-lane kernel: not where the
    // routed matmul runs mma.sync tiles (its result must equal quantize +
    // matmul bit for bit; gemv_fused_ok rejects such plans)
    const bool one_launch = x16 && !af && !dots && path == FT_PATH_GEMV && sh.wtype == FT_TYPE_Q4_0 &&
                            sh.act_div == sh.top_k && sh.n_global == sh.n_experts && aligned(x16, 16) &&
                            gp.smem <= 227 * 1024 && gemv_fused_ok(gp, sh.n_slots, sh.n_experts, sh.ncols);
    const WsLayout L = ws_layout(sh.n_slots, sh.n_experts, path == FT_PATH_GEMM ? sh.ncols : 0,
                                 h_in_ws ? 4 * static_cast<size_t>(sh.n_slots) * sh.nrows : 0,
                                 x16 && !one_launch ? act_rows_bytes(sh) : 0, gemm_sums);
    uint8_t* ws = nullptr;
    if (int st = ws_acquire(L.total, s, &ws)) return st;
    if (one_launch) {
        prof_mark(kProfRouteBegin, s);
        prof_mark(kProfMatmulBegin, s);
        const int st = launch_gemv_fused(gp, static_cast<const uint8_t*>(weights), static_cast<const uint16_t*>(x16),
                                         topk_ids, out, reinterpret_cast<uint32_t*>(ws + L.err), sh.n_slots,
                                         sh.top_k, sh.n_experts, sh.nrows, sh.ncols, s);
        prof_mark(kProfMatmulEnd, s);
        return st;
    }
    if (x16) {
        prof_mark(kProfQuantBegin, s);
        const int st = launch_quantize_q8_1(x16, ws + L.act, sh.tokens, sh.ncols, s);
        prof_mark(kProfQuantEnd, s);
        if (st) return st;
        act = ws + L.act;
    }
    if (h_in_ws) out = reinterpret_cast<float*>(ws + L.h);
    RouteBuffers rb{};
    rb.counts = reinterpret_cast<int32_t*>(ws + L.counts);
    rb.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    rb.perm = reinterpret_cast<int32_t*>(ws + L.perm);
    rb.hist = reinterpret_cast<int32_t*>(ws + L.hist);
    rb.tiles_gemv = reinterpret_cast<int32_t*>(ws + L.tiles_gemv);
    rb.tiles_gemm = reinterpret_cast<int32_t*>(ws + L.tiles_gemm);
    rb.err = reinterpret_cast<uint32_t*>(ws + L.err);

    const int tile_width = gemm_tile_width(sh.mean());
    if (path == FT_PATH_GEMV && (gp.smem > 227 * 1024 || gp.stages < 1))
        return fail(FT_ERR_SIZE, "GEMV tile needs %zu bytes of shared memory (%d ring stages of %lld-column rows fit)",
                    gp.smem, gp.stages, (long long)sh.ncols);
    // rows of slots with a bad expert id are zeroed by the router: block dots,
    // outputs, or (fused on the tensor-core path) the slot's Q8_1 row
    const bool fused_tc = af && path == FT_PATH_GEMM;
    uint32_t* zero_rows = dots       ? reinterpret_cast<uint32_t*>(dots)
                          : fused_tc ? reinterpret_cast<uint32_t*>(af->act_mid)
                                     : reinterpret_cast<uint32_t*>(out);
    const int64_t row_words = dots ? sh.nrows * sh.nb : fused_tc ? af->n_inter / 32 * 9 : sh.nrows;   // 9 words per Q8_1 block
    prof_mark(kProfRouteBegin, s);
    rb.expert_start = sh.expert_start;
    rb.n_global = sh.n_global;
    if (int st = launch_route(topk_ids, sh.n_slots, sh.n_experts, rb, gp.group, tile_width,
                              zero_rows, row_words, s))
        return st;
    if (path == FT_PATH_GEMM && sh.n_slots > 0) {
        if (int st = launch_gather(static_cast<const uint8_t*>(act), rb.perm, rb.offsets, sh.n_experts, sh.act_div,
                                   sh.nb, sh.n_slots, reinterpret_cast<uint16_t*>(ws + L.xh),
                                   reinterpret_cast<uint16_t*>(ws + L.da), s,
                                   gemm_sums ? reinterpret_cast<float*>(ws + L.sa) : nullptr))
            return st;
    }
    prof_mark(kProfMatmulBegin, s);
    int st;
    if (path == FT_PATH_GEMV) {
        st = launch_gemv(gp, static_cast<const uint8_t*>(weights), static_cast<const uint8_t*>(act), rb.perm,
                         rb.offsets, rb.tiles_gemv, out, dots, rb.err, sh.n_slots, sh.act_div, sh.n_experts, sh.nrows,
                         sh.ncols, s, sh.wtype);
        if (st == FT_OK && h_in_ws)
            st = launch_act_mul_quantize_q8_1(out, af->act_mid, sh.n_slots, af->n_inter, af->kind, s);
    } else {
        st = launch_gemm(static_cast<const uint8_t*>(weights), static_cast<const uint8_t*>(act), rb.perm,
                         rb.offsets, rb.tiles_gemm, fused_tc ? nullptr : out, dots, rb.err, sh.n_slots, sh.act_div,
                         sh.n_experts, sh.nrows, sh.ncols, reinterpret_cast<uint16_t*>(ws + L.xh),
                         reinterpret_cast<uint16_t*>(ws + L.da), tile_width, s, af,
                         gemm_sums ? reinterpret_cast<const float*>(ws + L.sa) : nullptr);
    }
    prof_mark(kProfMatmulEnd, s);
    return st;
}

}  // namespace ft

using namespace ft;

extern "C" {

int ft_abi_version(void) { return FT_MOE_ABI_VERSION; }

const char* ft_last_error(void) { return g_last_error.c_str(); }

int ft_quantize_q8_1(const void* x_fp16, void* act_q8_1, int64_t tokens, int64_t ncols, void* stream) {
    g_last_error.clear();
    if (tokens < 0) return fail(FT_ERR_ARG, "tokens must be >= 0");
    if (ncols <= 0 || ncols % 32 != 0) return fail(FT_ERR_ARG, "ncols must be a positive multiple of 32");
    int64_t n;
    if (!mul_ok(tokens, ncols, &n) || n > INT64_MAX / 4) return fail(FT_ERR_SIZE, "tokens * ncols overflows");
    if (tokens == 0) return FT_OK;
    if (!x_fp16 || !act_q8_1) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(x_fp16, 8) || !aligned(act_q8_1, 4))
        return fail(FT_ERR_ALIGN, "x_fp16 must be 8-byte and act_q8_1 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_mark(kProfQuantBegin, s);
    const int st = launch_quantize_q8_1(x_fp16, act_q8_1, tokens, ncols, s);
    prof_mark(kProfQuantEnd, s);
    return st;
}

int ft_moe_route_offsets(const int32_t* topk_ids, int64_t tokens, int32_t top_k, int32_t n_experts, int32_t* counts,
                         int32_t* offsets, int32_t* perm, uint32_t* dev_err, void* stream) {
    g_last_error.clear();
    Shape sh{};
    if (int st = check_route_args(tokens, top_k, n_experts, &sh)) return st;
    if (!counts || !offsets || (sh.n_slots > 0 && (!topk_ids || !perm))) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(topk_ids, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm, 4))
        return fail(FT_ERR_ALIGN, "int32 arrays must be 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const WsLayout L = ws_layout(sh.n_slots, sh.n_experts);
    uint8_t* ws = nullptr;
    if (int st = ws_acquire(L.total, s, &ws)) return st;
    RouteBuffers rb{};
    rb.counts = counts;
    rb.offsets = offsets;
    rb.perm = perm;
    rb.hist = reinterpret_cast<int32_t*>(ws + L.hist);
    rb.tiles_gemv = nullptr;
    rb.tiles_gemm = nullptr;
    rb.err = dev_err ? dev_err : reinterpret_cast<uint32_t*>(ws + L.err);
    return launch_route(topk_ids, sh.n_slots, sh.n_experts, rb, 1, 1, nullptr, 0, s);
}

static int matmul_entry(const void* weights, const void* act, const int32_t* topk_ids, float* out, int32_t* dots,
                        int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols,
                        void* stream, bool act_per_slot = false, int32_t expert_start = 0, int32_t n_local = 0,
                        int32_t wtype = FT_TYPE_Q4_0) {
    g_last_error.clear();
    Shape sh{};
    // n_experts counts every expert the ids may name; an expert-parallel shard
    // (n_local > 0) holds experts [expert_start, expert_start + n_local) of them
    if (int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh)) return st;
    if (act_per_slot) sh.act_div = 1;
    if (weight_block_bytes(wtype) == 0) return fail(FT_ERR_ARG, "unknown weight type %d", wtype);
    if (ncols % weight_block_values(wtype) != 0)
        return fail(FT_ERR_ARG, "weight type %d needs ncols %% %d == 0 (got %lld)", wtype, weight_block_values(wtype),
                    (long long)ncols);
    sh.wtype = wtype;
    if (n_local > 0) {
        if (expert_start < 0 || static_cast<int64_t>(expert_start) + n_local > n_experts)
            return fail(FT_ERR_ARG, "the shard's experts [%d, %lld) must lie in [0, n_experts_global=%d)", expert_start,
                        (long long)expert_start + n_local, n_experts);
        sh.expert_start = expert_start;
        sh.n_experts = n_local;
    }
    if (sh.n_slots == 0) return FT_OK;
    if (!weights || !act || !topk_ids || (!out && !dots)) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(weights, 16) || !aligned(act, 16))
        return fail(FT_ERR_ALIGN, "weights and act must be 16-byte aligned");
    if (!aligned(topk_ids, 4) || !aligned(out, 4) || !aligned(dots, 4))
        return fail(FT_ERR_ALIGN, "topk_ids / out / dots must be 4-byte aligned");
    if (dots) {
        int64_t n;
        if (!mul_ok(sh.n_slots * sh.nrows, sh.nb, &n) || n > INT32_MAX)
            return fail(FT_ERR_SIZE, "dots array would exceed 2^31 elements");
    }
    return run_matmul(weights, act, topk_ids, out, dots, sh, static_cast<cudaStream_t>(stream));
}

int ft_moe_q4_0_q8_1(const void* weights, const void* act, const int32_t* topk_ids, float* out, int64_t tokens,
                     int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols, void* stream) {
    if (!out) {
        g_last_error.clear();
        Shape sh{};
        if (int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh)) return st;
        if (sh.n_slots == 0) return FT_OK;
        return fail(FT_ERR_ARG, "null pointer");
    }
    return matmul_entry(weights, act, topk_ids, out, nullptr, tokens, top_k, n_experts, nrows, ncols, stream);
}

int ft_moe_q4_0_fp16(const void* weights, const void* x_fp16, const int32_t* topk_ids, float* out, int64_t tokens,
                     int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols, void* stream) {
    g_last_error.clear();
    Shape sh{};
    if (int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh)) return st;
    if (sh.n_slots == 0) return FT_OK;
    if (!weights || !x_fp16 || !topk_ids || !out) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(weights, 16)) return fail(FT_ERR_ALIGN, "weights must be 16-byte aligned");
    if (!aligned(x_fp16, 8) || !aligned(topk_ids, 4) || !aligned(out, 4))
        return fail(FT_ERR_ALIGN, "x_fp16 must be 8-byte, topk_ids and out 4-byte aligned");
    return run_matmul(weights, nullptr, topk_ids, out, nullptr, sh, static_cast<cudaStream_t>(stream), nullptr, x_fp16);
}

int ft_moe_q4_0_q8_1_ep(const void* weights_local, const void* act, const int32_t* topk_ids, float* out,
                        int64_t tokens, int32_t top_k, int32_t n_experts_global, int32_t expert_start,
                        int32_t n_experts_local, int64_t nrows, int64_t ncols, void* stream) {
    if (n_experts_local < 1) {
        g_last_error.clear();
        return fail(FT_ERR_ARG, "n_experts_local must be >= 1 (got %d)", n_experts_local);
    }
    if (!out) {
        g_last_error.clear();
        Shape sh{};
        if (int st = check_matmul_args(tokens, top_k, n_experts_global, nrows, ncols, &sh)) return st;
        if (sh.n_slots == 0) return FT_OK;
        return fail(FT_ERR_ARG, "null pointer");
    }
    return matmul_entry(weights_local, act, topk_ids, out, nullptr, tokens, top_k, n_experts_global, nrows, ncols,
                        stream, false, expert_start, n_experts_local);
}

int ft_moe_q4_0_q8_1_slots(const void* weights, const void* act_slots, const int32_t* topk_ids, float* out,
                           int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols,
                           void* stream) {
    if (!out) {
        g_last_error.clear();
        Shape sh{};
        if (int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh)) return st;
        if (sh.n_slots == 0) return FT_OK;
        return fail(FT_ERR_ARG, "null pointer");
    }
    return matmul_entry(weights, act_slots, topk_ids, out, nullptr, tokens, top_k, n_experts, nrows, ncols, stream,
                        true);
}

int ft_act_mul_quantize_q8_1(const float* h, void* act_q8_1, int64_t rows, int64_t n_inter, int32_t act_kind,
                             void* stream) {
    g_last_error.clear();
    if (rows < 0) return fail(FT_ERR_ARG, "rows must be >= 0 (got %lld)", (long long)rows);
    if (n_inter <= 0 || n_inter % 32 != 0)
        return fail(FT_ERR_ARG, "n_inter must be a positive multiple of 32 (got %lld)", (long long)n_inter);
    if (act_kind != FT_ACT_SILU && act_kind != FT_ACT_GELU_TANH)
        return fail(FT_ERR_ARG, "act_kind must be FT_ACT_SILU or FT_ACT_GELU_TANH (got %d)", act_kind);
    int64_t n;
    if (!mul_ok(rows, 2 * n_inter, &n) || n > INT64_MAX / 8) return fail(FT_ERR_SIZE, "rows * n_inter overflows");
    if (rows == 0) return FT_OK;
    if (!h || !act_q8_1) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(h, 16) || !aligned(act_q8_1, 4))
        return fail(FT_ERR_ALIGN, "h must be 16-byte and act_q8_1 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_mark(kProfQuantBegin, s);
    const int st = launch_act_mul_quantize_q8_1(h, act_q8_1, rows, n_inter, act_kind, s);
    prof_mark(kProfQuantEnd, s);
    return st;
}

int ft_moe_q4_0_q8_1_act(const void* w13, const void* act, const int32_t* topk_ids, void* act_mid, int64_t tokens,
                         int32_t top_k, int32_t n_experts, int64_t n_inter, int64_t hidden, int32_t act_kind,
                         void* stream) {
    g_last_error.clear();
    Shape sh{};
    if (n_inter <= 0 || n_inter % 32 != 0 || n_inter > INT64_MAX / 4)
        return fail(FT_ERR_ARG, "n_inter must be a positive multiple of 32 (got %lld)", (long long)n_inter);
    if (int st = check_matmul_args(tokens, top_k, n_experts, 2 * n_inter, hidden, &sh)) return st;
    if (act_kind != FT_ACT_SILU && act_kind != FT_ACT_GELU_TANH)
        return fail(FT_ERR_ARG, "act_kind must be FT_ACT_SILU or FT_ACT_GELU_TANH (got %d)", act_kind);
    if (sh.n_slots == 0) return FT_OK;
    if (!w13 || !act || !topk_ids || !act_mid) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(w13, 16) || !aligned(act, 16)) return fail(FT_ERR_ALIGN, "w13 and act must be 16-byte aligned");
    if (!aligned(topk_ids, 4) || !aligned(act_mid, 4))
        return fail(FT_ERR_ALIGN, "topk_ids and act_mid must be 4-byte aligned");
    const ActFuse af{static_cast<uint8_t*>(act_mid), n_inter, act_kind};
    return run_matmul(w13, act, topk_ids, nullptr, nullptr, sh, static_cast<cudaStream_t>(stream), &af);
}

int ft_moe_ffn_q4_0_q8_1(const void* w13, const void* w2, const void* act, const int32_t* topk_ids, float* h,
                         void* act_mid, float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                         int64_t hidden, int64_t n_inter, int32_t act_kind, void* stream) {
    g_last_error.clear();
    Shape sh{};
    if (n_inter <= 0 || n_inter > INT64_MAX / 2) return fail(FT_ERR_ARG, "n_inter must be > 0");
    if (int st = check_matmul_args(tokens, top_k, n_experts, 2 * n_inter, hidden, &sh)) return st;
    if (int st = check_matmul_args(tokens, top_k, n_experts, hidden, n_inter, &sh)) return st;
    if (act_kind != FT_ACT_SILU && act_kind != FT_ACT_GELU_TANH)
        return fail(FT_ERR_ARG, "act_kind must be FT_ACT_SILU or FT_ACT_GELU_TANH (got %d)", act_kind);
    if (sh.n_slots == 0) return FT_OK;
    if (!act_mid || !out) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(h, 16) || !aligned(act_mid, 16)) return fail(FT_ERR_ALIGN, "h and act_mid must be 16-byte aligned");
    if (h) {
        if (int st = matmul_entry(w13, act, topk_ids, h, nullptr, tokens, top_k, n_experts, 2 * n_inter, hidden,
                                  stream))
            return st;
        if (int st = ft_act_mul_quantize_q8_1(h, act_mid, sh.n_slots, n_inter, act_kind, stream)) return st;
    } else if (int st = ft_moe_q4_0_q8_1_act(w13, act, topk_ids, act_mid, tokens, top_k, n_experts, n_inter, hidden,
                                             act_kind, stream)) {
        return st;
    }
    return matmul_entry(w2, act_mid, topk_ids, out, nullptr, tokens, top_k, n_experts, hidden, n_inter, stream, true);
}

int ft_moe_ffn_reserve(int64_t max_tokens, int32_t max_top_k, int32_t n_experts, int64_t hidden, int64_t n_inter) {
    g_last_error.clear();
    Shape s1{}, s2{};
    if (n_inter <= 0 || n_inter > INT64_MAX / 4) return fail(FT_ERR_ARG, "n_inter must be > 0");
    if (int st = check_matmul_args(max_tokens, max_top_k, n_experts, 2 * n_inter, hidden, &s1)) return st;
    if (int st = check_matmul_args(max_tokens, max_top_k, n_experts, hidden, n_inter, &s2)) return st;
    // layer 1 on the tensor-core path, layer 1 fused on the GEMV path (its
    // result in workspace, at most the slots that path is chosen for), layer 2
    size_t need = ws_layout(s1.n_slots, n_experts, gemm_shape_ok(s1) ? hidden : 0).total;
    const size_t fused_gemv =
        ws_layout(s1.n_slots, n_experts, 0, 4 * static_cast<size_t>(gemv_max_slots(s1)) * 2 * n_inter).total;
    const size_t l2 = ws_layout(s2.n_slots, n_experts, gemm_shape_ok(s2) ? n_inter : 0).total;
    need = need > fused_gemv ? need : fused_gemv;
    need = need > l2 ? need : l2;
    uint8_t* base = nullptr;
    return ws_acquire(need, nullptr, &base);
}

int ft_moe_gguf_q8_1(int32_t wtype, const void* weights, const void* act, const int32_t* topk_ids, float* out,
                     int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols, void* stream) {
    if (weight_block_bytes(wtype) == 0) {
        g_last_error.clear();
        return fail(FT_ERR_ARG, "unknown weight type %d", wtype);
    }
    if (!out) {
        g_last_error.clear();
        Shape sh{};
        if (int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh)) return st;
        if (sh.n_slots == 0) return FT_OK;
        return fail(FT_ERR_ARG, "null pointer");
    }
    return matmul_entry(weights, act, topk_ids, out, nullptr, tokens, top_k, n_experts, nrows, ncols, stream, false,
                        0, 0, wtype);
}

int ft_repack_q4_0_soa(const void* weights, void* qs, void* d, int64_t n_blocks, void* stream) {
    g_last_error.clear();
    if (n_blocks < 0) return fail(FT_ERR_ARG, "n_blocks must be >= 0 (got %lld)", (long long)n_blocks);
    if (n_blocks > INT64_MAX / 18) return fail(FT_ERR_SIZE, "n_blocks * 18 overflows int64");
    if (n_blocks == 0) return FT_OK;
    if (!weights || !qs || !d) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(weights, 2) || !aligned(qs, 16) || !aligned(d, 2))
        return fail(FT_ERR_ALIGN, "weights and d must be 2-byte, qs 16-byte aligned");
    return launch_repack_q4_0_soa(weights, qs, d, n_blocks, static_cast<cudaStream_t>(stream));
}

int ft_moe_block_dots(const void* weights, const void* act, const int32_t* topk_ids, int32_t* dots, int64_t tokens,
                      int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols, void* stream) {
    if (!dots) {
        g_last_error.clear();
        Shape sh{};
        if (int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh)) return st;
        if (sh.n_slots == 0) return FT_OK;
        return fail(FT_ERR_ARG, "null pointer");
    }
    return matmul_entry(weights, act, topk_ids, nullptr, dots, tokens, top_k, n_experts, nrows, ncols, stream);
}

size_t ft_moe_workspace_bytes(int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols) {
    Shape sh{};
    std::string keep = g_last_error;
    const int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh);
    g_last_error = keep;
    if (st) return 0;
    return ws_layout(sh.n_slots, sh.n_experts, gemm_shape_ok(sh) ? sh.ncols : 0, 0, act_rows_bytes(sh),
                     gemm_shape_ok(sh))
        .total;
}

int ft_moe_reserve(int64_t max_tokens, int32_t max_top_k, int32_t n_experts, int64_t nrows, int64_t ncols) {
    g_last_error.clear();
    Shape sh{};
    if (int st = check_matmul_args(max_tokens, max_top_k, n_experts, nrows, ncols, &sh)) return st;
    uint8_t* base = nullptr;
    return ws_acquire(ws_layout(sh.n_slots, sh.n_experts, gemm_shape_ok(sh) ? sh.ncols : 0, 0, act_rows_bytes(sh),
                                gemm_shape_ok(sh))
                          .total,
                      nullptr, &base);
}

int ft_moe_release(void) {
    g_last_error.clear();
    int dev;
    if (int st = current_device(&dev)) return st;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    DeviceWs& w = g_ws[dev];
    if (w.base) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        e = cudaFree(w.base);
        w.base = nullptr;
        w.bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
    }
    return FT_OK;
}

int ft_moe_read_device_error(void* stream, uint32_t* flags_out) {
    g_last_error.clear();
    if (!flags_out) return fail(FT_ERR_ARG, "null pointer");
    *flags_out = 0;
    int dev;
    if (int st = current_device(&dev)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    DeviceWs& w = g_ws[dev];
    if (!w.base) return FT_OK;
    uint32_t v = 0;
    e = cudaMemcpy(&v, w.base, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
    e = cudaMemset(w.base, 0, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
    uint8_t guard[kGuardBytes];
    uint8_t* gdev = static_cast<uint8_t*>(w.base) + w.bytes;
    e = cudaMemcpy(guard, gdev, kGuardBytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(workspace guard)");
    for (size_t i = 0; i < kGuardBytes; ++i)
        if (guard[i] != kGuardByte) {
            v |= FT_DEVERR_WORKSPACE_GUARD;
            e = cudaMemset(gdev, kGuardByte, kGuardBytes);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(workspace guard)");
            break;
        }
    *flags_out = v;
    return v ? fail(FT_ERR_DEVICE_FLAG, "device error flags 0x%x", v) : FT_OK;
}

int ft_debug_stream_read(const void* buf, int64_t bytes, void* stream) {
    g_last_error.clear();
    if (bytes < 0 || bytes % 16 != 0)
        return fail(FT_ERR_ARG, "bytes must be a non-negative multiple of 16 (got %lld)", (long long)bytes);
    if (bytes == 0) return FT_OK;
    if (!buf) return fail(FT_ERR_ARG, "null pointer");
    if (!aligned(buf, 16)) return fail(FT_ERR_ALIGN, "buf must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = nullptr;
    if (int st = ws_acquire(ws_layout(0, 1).total, s, &ws)) return st;
    // the sink is the workspace's error word: written only on an impossible sum
    return launch_stream_read(buf, bytes / 16, reinterpret_cast<uint32_t*>(ws + ws_layout(0, 1).counts), s);
}

int ft_debug_wait_timeout(int64_t limit_ns, void* stream) {
    g_last_error.clear();
    if (limit_ns < 1000 || limit_ns > 1000000000)
        return fail(FT_ERR_ARG, "limit_ns must be in [1000, 1000000000] (got %lld)", (long long)limit_ns);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = nullptr;
    if (int st = ws_acquire(ws_layout(0, 1).total, s, &ws)) return st;
    return launch_wait_timeout_probe(reinterpret_cast<uint32_t*>(ws + ws_layout(0, 1).err), limit_ns, s);
}

int ft_profile_enable(int32_t max_calls) {
    g_last_error.clear();
    if (max_calls < 0) return fail(FT_ERR_ARG, "max_calls must be >= 0");
    std::lock_guard<std::mutex> lk(g_prof.mu);
    Prof& P = g_prof;
    if (P.ev) {
        for (int i = 0; i < P.max_calls * 5; ++i) cudaEventDestroy(P.ev[i]);
        delete[] P.ev;
        P.ev = nullptr;
    }
    P.on = false;
    P.max_calls = 0;
    P.n_quant = P.n_mm = 0;
    P.quant_open = P.mm_open = false;
    P.launches = 0;
    if (max_calls == 0) return FT_OK;
    P.ev = new cudaEvent_t[static_cast<size_t>(max_calls) * 5];
    for (int i = 0; i < max_calls * 5; ++i) {
        const cudaError_t e = cudaEventCreate(&P.ev[i]);
        if (e != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(P.ev[j]);
            delete[] P.ev;
            P.ev = nullptr;
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    P.max_calls = max_calls;
    P.on = true;
    return FT_OK;
}

int ft_profile_read(double* quantize_ms, double* route_ms, double* matmul_ms, int64_t* n_calls,
                    int64_t* n_launches) {
    g_last_error.clear();
    std::lock_guard<std::mutex> lk(g_prof.mu);
    Prof& P = g_prof;
    double q = 0, r = 0, m = 0;
    for (int i = 0; i < P.n_quant; ++i) {
        float ms = 0;
        cudaError_t e = cudaEventSynchronize(P.ev[i * 5 + 1]);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, P.ev[i * 5 + 0], P.ev[i * 5 + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "reading quantizer events");
        q += ms;
    }
    for (int i = 0; i < P.n_mm; ++i) {
        float a = 0, b = 0;
        cudaError_t e = cudaEventSynchronize(P.ev[i * 5 + 4]);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&a, P.ev[i * 5 + 2], P.ev[i * 5 + 3]);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&b, P.ev[i * 5 + 3], P.ev[i * 5 + 4]);
        if (e != cudaSuccess) return cuda_fail(e, "reading matmul events");
        r += a;
        m += b;
    }
    if (quantize_ms) *quantize_ms = q;
    if (route_ms) *route_ms = r;
    if (matmul_ms) *matmul_ms = m;
    if (n_calls) *n_calls = P.n_mm;
    if (n_launches) *n_launches = P.launches;
    P.n_quant = P.n_mm = 0;
    P.quant_open = P.mm_open = false;
    P.launches = 0;
    return FT_OK;
}

int ft_moe_set_path(int32_t path) {
    if (path != FT_PATH_AUTO && path != FT_PATH_GEMV && path != FT_PATH_GEMM && path != FT_PATH_GEMV_DP4A) return -1;
    const int prev = path_setting();
    std::lock_guard<std::mutex> lk(g_path_mu);
    g_path = path;
    return prev;
}

int ft_moe_selected_path(int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols) {
    return ft_moe_gguf_selected_path(FT_TYPE_Q4_0, tokens, top_k, n_experts, nrows, ncols);
}

int ft_moe_gguf_selected_path(int32_t wtype, int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                              int64_t ncols) {
    Shape sh{};
    std::string keep = g_last_error;
    const int st = check_matmul_args(tokens, top_k, n_experts, nrows, ncols, &sh);
    g_last_error = keep;
    if (st || weight_block_bytes(wtype) == 0 || ncols % weight_block_values(wtype) != 0) return -1;
    sh.wtype = wtype;
    return choose_path(sh, path_setting());
}

}  // extern "C"
