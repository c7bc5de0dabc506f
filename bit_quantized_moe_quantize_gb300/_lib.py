"""ctypes binding of libft_moe.so: argument marshalling only.

Every function here checks tensor dtypes, devices and shapes, then passes raw
device pointers and the current CUDA stream to the C ABI declared in
``include/ft_moe.h``.  No arithmetic of the routed matmul happens in Python,
and there is no fallback: if the library is missing or was built from other
sources, loading raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libft_moe.so")

FT_OK, FT_ERR_ARG, FT_ERR_SIZE, FT_ERR_ALIGN, FT_ERR_LAUNCH, FT_ERR_WORKSPACE, FT_ERR_CUDA, FT_ERR_DEVICE_FLAG = range(8)
STATUS_NAMES = {0: "FT_OK", 1: "FT_ERR_ARG", 2: "FT_ERR_SIZE", 3: "FT_ERR_ALIGN", 4: "FT_ERR_LAUNCH",
                5: "FT_ERR_WORKSPACE", 6: "FT_ERR_CUDA", 7: "FT_ERR_DEVICE_FLAG"}
FT_DEVERR_BAD_EXPERT_ID = 0x1
FT_DEVERR_WAIT_TIMEOUT = 0x2
FT_DEVERR_WORKSPACE_GUARD = 0x4
FT_PATH_AUTO, FT_PATH_GEMV, FT_PATH_GEMM, FT_PATH_GEMV_DP4A = 0, 1, 2, 3
PATHS = {"auto": FT_PATH_AUTO, "gemv": FT_PATH_GEMV, "gemm": FT_PATH_GEMM, "gemv_dp4a": FT_PATH_GEMV_DP4A}

EXPORTS = ("ft_quantize_q8_1", "ft_moe_route_offsets", "ft_moe_q4_0_q8_1", "ft_moe_workspace_bytes",
           "ft_moe_reserve", "ft_moe_release", "ft_moe_read_device_error", "ft_moe_set_path",
           "ft_moe_selected_path", "ft_moe_gguf_selected_path", "ft_moe_block_dots", "ft_last_error", "ft_abi_version", "ft_profile_enable",
           "ft_profile_read", "ft_moe_route_offsets_noalloc", "ft_moe_q4_0_q8_1_slots",
           "ft_moe_q4_0_q8_1_ep", "ft_act_mul_quantize_q8_1", "ft_moe_ffn_q4_0_q8_1", "ft_moe_gguf_q8_1",
           "ft_repack_q4_0_soa", "ft_debug_wait_timeout", "ft_moe_q4_0_q8_1_act", "ft_moe_ffn_reserve",
           "ft_moe_q4_0_fp16", "ft_debug_stream_read")


class FtError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library, refusing a build whose source hash is stale."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _build
        if not os.path.exists(path):
            raise FtError(FT_ERR_CUDA, f"{path} is missing: run bit_quantized_moe_quantize_gb300.build.build()")
        if path == LIB_PATH and not _build.is_current():
            raise FtError(FT_ERR_CUDA, f"{path} was built from other sources: rebuild it")
        L = ctypes.CDLL(path)
        i64, i32, vp, u32p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)
        L.ft_quantize_q8_1.argtypes = [vp, vp, i64, i64, vp]
        L.ft_moe_route_offsets.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp, vp]
        L.ft_moe_route_offsets_noalloc.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp, vp]
        L.ft_moe_q4_0_q8_1.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, vp]
        L.ft_moe_q4_0_q8_1_slots.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, vp]
        L.ft_moe_q4_0_fp16.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, vp]
        L.ft_moe_q4_0_q8_1_ep.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i32, i64, i64, vp]
        L.ft_moe_block_dots.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, vp]
        L.ft_act_mul_quantize_q8_1.argtypes = [vp, vp, i64, i64, i32, vp]
        L.ft_moe_gguf_q8_1.argtypes = [i32, vp, vp, vp, vp, i64, i32, i32, i64, i64, vp]
        L.ft_repack_q4_0_soa.argtypes = [vp, vp, vp, i64, vp]
        L.ft_debug_wait_timeout.argtypes = [i64, vp]
        L.ft_debug_stream_read.argtypes = [vp, i64, vp]
        L.ft_moe_ffn_q4_0_q8_1.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i64, i64, i32, vp]
        L.ft_moe_q4_0_q8_1_act.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, i32, vp]
        L.ft_moe_ffn_reserve.argtypes = [i64, i32, i32, i64, i64]
        L.ft_moe_workspace_bytes.argtypes = [i64, i32, i32, i64, i64]
        L.ft_moe_workspace_bytes.restype = ctypes.c_size_t
        L.ft_moe_reserve.argtypes = [i64, i32, i32, i64, i64]
        L.ft_moe_release.argtypes = []
        L.ft_moe_read_device_error.argtypes = [vp, u32p]
        L.ft_moe_set_path.argtypes = [i32]
        L.ft_moe_selected_path.argtypes = [i64, i32, i32, i64, i64]
        L.ft_moe_gguf_selected_path.argtypes = [i32, i64, i32, i32, i64, i64]
        L.ft_last_error.argtypes = []
        L.ft_last_error.restype = ctypes.c_char_p
        L.ft_abi_version.argtypes = []
        L.ft_profile_enable.argtypes = [i32]
        dp, lp = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)
        L.ft_profile_read.argtypes = [dp, dp, dp, lp, lp]
        for name in EXPORTS:
            getattr(L, name).restype = getattr(L, name).restype or ctypes.c_int
        L.ft_moe_workspace_bytes.restype = ctypes.c_size_t
        L.ft_last_error.restype = ctypes.c_char_p
        _lib = L
        return L


def last_error() -> str:
    return load().ft_last_error().decode()


def _check(status: int):
    if status != FT_OK:
        raise FtError(status, last_error())


# ------------------------------------------------------------------ tensors
def _torch():
    import torch
    return torch


def _stream(t):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dev(t, dtype, name, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def quantize_q8_1(x, out=None):
    """fp16 [T, K] -> Q8_1 uint8 [T, K/32, 36] (ft_quantize_q8_1)."""
    torch = _torch()
    px = _dev(x, torch.float16, "x", 2)
    T, K = x.shape
    if out is None:
        out = torch.empty((T, K // 32, 36), dtype=torch.uint8, device=x.device)
    po = _dev(out, torch.uint8, "out")
    _check(load().ft_quantize_q8_1(px, po, T, K, _stream(x)))
    return out


def route_offsets(topk_ids, n_experts, counts=None, offsets=None, perm=None, dev_err=None):
    """int32 [T, k] -> (counts [E], offsets [E+1], perm [T*k]) (ft_moe_route_offsets)."""
    torch = _torch()
    pid = _dev(topk_ids, torch.int32, "topk_ids", 2)
    T, k = topk_ids.shape
    dev = topk_ids.device
    counts = torch.empty(n_experts, dtype=torch.int32, device=dev) if counts is None else counts
    offsets = torch.empty(n_experts + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    perm = torch.empty(T * k, dtype=torch.int32, device=dev) if perm is None else perm
    pe = ctypes.c_void_p(0) if dev_err is None else _dev(dev_err, torch.int32, "dev_err")
    _check(load().ft_moe_route_offsets(pid, T, k, n_experts, _dev(counts, torch.int32, "counts"),
                                       _dev(offsets, torch.int32, "offsets"), _dev(perm, torch.int32, "perm"),
                                       pe, _stream(topk_ids)))
    return counts, offsets, perm


def _matmul_shape(weights, act, topk_ids):
    torch = _torch()
    _dev(weights, torch.uint8, "weights", 4)
    _dev(act, torch.uint8, "act", 3)
    _dev(topk_ids, torch.int32, "topk_ids", 2)
    E, N, nb, wb = weights.shape
    T, nb2, ab = act.shape
    if wb != 18 or ab != 36 or nb != nb2 or topk_ids.shape[0] != T:
        raise ValueError(f"shape mismatch: weights {tuple(weights.shape)} act {tuple(act.shape)} "
                         f"topk_ids {tuple(topk_ids.shape)}")
    return E, N, nb * 32, T, topk_ids.shape[1]


def moe_q4_0_q8_1(weights, act, topk_ids, out=None):
    """Routed matmul: Q4_0 [E,N,K/32,18] x Q8_1 [T,K/32,36] -> fp32 [T, k, N] (ft_moe_q4_0_q8_1)."""
    torch = _torch()
    E, N, K, T, k = _matmul_shape(weights, act, topk_ids)
    if out is None:
        out = torch.empty((T, k, N), dtype=torch.float32, device=weights.device)
    po = _dev(out, torch.float32, "out")
    _check(load().ft_moe_q4_0_q8_1(ctypes.c_void_p(weights.data_ptr()), ctypes.c_void_p(act.data_ptr()),
                                   ctypes.c_void_p(topk_ids.data_ptr()), po, T, k, E, N, K, _stream(weights)))
    return out


def moe_q4_0_q8_1_slots(weights, act_slots, topk_ids, out=None):
    """Routed matmul with one activation row per slot: Q4_0 [E,N,K/32,18] x
    Q8_1 [T*k,K/32,36] (row s for slot s = t*k + j) -> fp32 [T, k, N]
    (ft_moe_q4_0_q8_1_slots)."""
    torch = _torch()
    _dev(weights, torch.uint8, "weights", 4)
    _dev(act_slots, torch.uint8, "act_slots", 3)
    _dev(topk_ids, torch.int32, "topk_ids", 2)
    E, N, nb, wb = weights.shape
    S, nb2, ab = act_slots.shape
    T, k = topk_ids.shape
    if wb != 18 or ab != 36 or nb != nb2 or S != T * k:
        raise ValueError(f"shape mismatch: weights {tuple(weights.shape)} act_slots {tuple(act_slots.shape)} "
                         f"topk_ids {tuple(topk_ids.shape)}")
    if out is None:
        out = torch.empty((T, k, N), dtype=torch.float32, device=weights.device)
    po = _dev(out, torch.float32, "out")
    _check(load().ft_moe_q4_0_q8_1_slots(ctypes.c_void_p(weights.data_ptr()), ctypes.c_void_p(act_slots.data_ptr()),
                                         ctypes.c_void_p(topk_ids.data_ptr()), po, T, k, E, N, nb * 32,
                                         _stream(weights)))
    return out


def moe_q4_0_q8_1_ep(weights_local, act, topk_ids, n_experts_global, expert_start, out=None):
    """Routed matmul on an expert-parallel shard (ft_moe_q4_0_q8_1_ep):
    weights_local Q4_0 [E_local,N,K/32,18] holds experts [expert_start,
    expert_start + E_local) of n_experts_global; topk_ids hold global ids;
    rows of slots routed elsewhere are 0."""
    torch = _torch()
    E_local, N, K, T, k = _matmul_shape(weights_local, act, topk_ids)
    if out is None:
        out = torch.empty((T, k, N), dtype=torch.float32, device=weights_local.device)
    po = _dev(out, torch.float32, "out")
    _check(load().ft_moe_q4_0_q8_1_ep(ctypes.c_void_p(weights_local.data_ptr()), ctypes.c_void_p(act.data_ptr()),
                                      ctypes.c_void_p(topk_ids.data_ptr()), po, T, k, int(n_experts_global),
                                      int(expert_start), E_local, N, K, _stream(weights_local)))
    return out


# GGUF weight types: GGML type number, bytes per stored block, weights per block
WEIGHT_TYPES = {"q4_0": (2, 18, 32), "q4_1": (3, 20, 32), "q5_0": (6, 22, 32), "q5_1": (7, 24, 32),
                "q8_0": (8, 34, 32), "q4_k": (12, 144, 256), "q5_k": (13, 176, 256),
                "q6_k": (14, 210, 256), "q2_k": (10, 84, 256), "q3_k": (11, 110, 256)}


def moe_gguf_q8_1(wtype, weights, act, topk_ids, out=None):
    """Routed matmul with weights of a GGUF type (ft_moe_gguf_q8_1): weights uint8
    [E, N, K/32 (K/256 for the K-quants), bytes of the type] x Q8_1 [T, K/32, 36]
    -> fp32 [T, k, N]."""
    torch = _torch()
    tid, bb, per = WEIGHT_TYPES[wtype]
    _dev(weights, torch.uint8, "weights", 4)
    _dev(act, torch.uint8, "act", 3)
    _dev(topk_ids, torch.int32, "topk_ids", 2)
    E, N, nb, wb = weights.shape
    T, nb2, ab = act.shape
    if wb != bb or ab != 36 or nb * per != nb2 * 32 or topk_ids.shape[0] != T:
        raise ValueError(f"shape mismatch for {wtype}: weights {tuple(weights.shape)} act {tuple(act.shape)} "
                         f"topk_ids {tuple(topk_ids.shape)}")
    k = topk_ids.shape[1]
    if out is None:
        out = torch.empty((T, k, N), dtype=torch.float32, device=weights.device)
    po = _dev(out, torch.float32, "out")
    _check(load().ft_moe_gguf_q8_1(tid, ctypes.c_void_p(weights.data_ptr()), ctypes.c_void_p(act.data_ptr()),
                                   ctypes.c_void_p(topk_ids.data_ptr()), po, T, k, E, N, nb * per, _stream(weights)))
    return out


def repack_q4_0_soa(weights, qs=None, d=None):
    """Q4_0 blocks uint8 [..., 18] -> (nibble bytes uint8 [n, 16], fp16 scales [n])
    (ft_repack_q4_0_soa)."""
    torch = _torch()
    _dev(weights, torch.uint8, "weights")
    if weights.shape[-1] != 18:
        raise ValueError(f"weights must end in 18-byte Q4_0 blocks, got {tuple(weights.shape)}")
    n = weights.numel() // 18
    qs = torch.empty((n, 16), dtype=torch.uint8, device=weights.device) if qs is None else qs
    d = torch.empty(n, dtype=torch.float16, device=weights.device) if d is None else d
    _check(load().ft_repack_q4_0_soa(ctypes.c_void_p(weights.data_ptr()), _dev(qs, torch.uint8, "qs"),
                                     _dev(d, torch.float16, "d"), n, _stream(weights)))
    return qs, d


ACT_SILU = 0
ACT_GELU_TANH = 1


def act_mul_quantize_q8_1(h, act_kind, out=None):
    """fp32 [..., 2I] (gate | up) -> Q8_1 uint8 [rows, I/32, 36] of act(gate) * up,
    rows = h.numel() / 2I (ft_act_mul_quantize_q8_1)."""
    torch = _torch()
    ph = _dev(h, torch.float32, "h")
    two_i = h.shape[-1]
    if two_i % 64:
        raise ValueError(f"the last dim of h must be 2 * n_inter with n_inter % 32 == 0 (got {two_i})")
    rows = h.numel() // two_i
    if out is None:
        out = torch.empty((rows, two_i // 64, 36), dtype=torch.uint8, device=h.device)
    po = _dev(out, torch.uint8, "out")
    if out.numel() != rows * (two_i // 64) * 36:
        raise ValueError(f"out must hold {rows} x {two_i // 64} Q8_1 blocks")
    _check(load().ft_act_mul_quantize_q8_1(ph, po, rows, two_i // 2, int(act_kind), _stream(h)))
    return out


def moe_q4_0_fp16(weights, x, topk_ids, out=None):
    """The whole hot path from fp16 rows (ft_moe_q4_0_fp16): Q4_0 [E, N, K/32, 18]
    x fp16 [T, K] -> fp32 [T, k, N]; one launch for decode-sized batches."""
    torch = _torch()
    _dev(weights, torch.uint8, "weights", 4)
    px = _dev(x, torch.float16, "x", 2)
    _dev(topk_ids, torch.int32, "topk_ids", 2)
    E, N, nb, wb = weights.shape
    T, K = x.shape
    if wb != 18 or nb * 32 != K or topk_ids.shape[0] != T:
        raise ValueError(f"shape mismatch: weights {tuple(weights.shape)} x {tuple(x.shape)} "
                         f"topk_ids {tuple(topk_ids.shape)}")
    k = topk_ids.shape[1]
    if out is None:
        out = torch.empty((T, k, N), dtype=torch.float32, device=weights.device)
    po = _dev(out, torch.float32, "out")
    _check(load().ft_moe_q4_0_fp16(ctypes.c_void_p(weights.data_ptr()), px, ctypes.c_void_p(topk_ids.data_ptr()),
                                   po, T, k, E, N, K, _stream(weights)))
    return out


def moe_q4_0_q8_1_act(w13, act, topk_ids, act_kind, out=None):
    """Layer 1 with the gated activation fused (ft_moe_q4_0_q8_1_act): w13 Q4_0
    [E, 2I, H/32, 18] (gate rows, then up rows), act Q8_1 [T, H/32, 36] ->
    Q8_1 uint8 [T*k, I/32, 36] of act(gate) * up per slot."""
    torch = _torch()
    E, two_i, H, T, k = _matmul_shape(w13, act, topk_ids)
    if two_i % 64:
        raise ValueError(f"w13 must hold 2 * n_inter rows with n_inter % 32 == 0 (got {two_i})")
    I = two_i // 2
    if out is None:
        out = torch.empty((T * k, I // 32, 36), dtype=torch.uint8, device=w13.device)
    po = _dev(out, torch.uint8, "out")
    if out.numel() != T * k * (I // 32) * 36:
        raise ValueError(f"out must hold {T * k} x {I // 32} Q8_1 blocks")
    _check(load().ft_moe_q4_0_q8_1_act(ctypes.c_void_p(w13.data_ptr()), ctypes.c_void_p(act.data_ptr()),
                                       ctypes.c_void_p(topk_ids.data_ptr()), po, T, k, E, I, H, int(act_kind),
                                       _stream(w13)))
    return out


def moe_ffn_q4_0_q8_1(w13, w2, act, topk_ids, act_kind, out=None, h=None, act_mid=None, keep_h=True):
    """Both expert layers per slot (ft_moe_ffn_q4_0_q8_1): w13 Q4_0 [E, 2I, H/32, 18]
    (gate rows, then up rows), w2 Q4_0 [E, H, I/32, 18], act Q8_1 [T, H/32, 36]
    -> out fp32 [T, k, H]; returns (out, h [T, k, 2I] fp32, act_mid [T*k, I/32, 36]).
    keep_h=False (and h None): layer 1 with the activation fused, h is None."""
    torch = _torch()
    E, two_i, H, T, k = _matmul_shape(w13, act, topk_ids)
    _dev(w2, torch.uint8, "w2", 4)
    if w2.shape[0] != E or w2.shape[1] != H or w2.shape[3] != 18 or 2 * w2.shape[2] * 32 != two_i:
        raise ValueError(f"shape mismatch: w13 {tuple(w13.shape)} w2 {tuple(w2.shape)}")
    I = two_i // 2
    dev = w13.device
    out = torch.empty((T, k, H), dtype=torch.float32, device=dev) if out is None else out
    if h is None and keep_h:
        h = torch.empty((T, k, two_i), dtype=torch.float32, device=dev)
    act_mid = torch.empty((T * k, I // 32, 36), dtype=torch.uint8, device=dev) if act_mid is None else act_mid
    ph = ctypes.c_void_p(0) if h is None else _dev(h, torch.float32, "h")
    _check(load().ft_moe_ffn_q4_0_q8_1(ctypes.c_void_p(w13.data_ptr()), ctypes.c_void_p(w2.data_ptr()),
                                       ctypes.c_void_p(act.data_ptr()), ctypes.c_void_p(topk_ids.data_ptr()),
                                       ph, _dev(act_mid, torch.uint8, "act_mid"),
                                       _dev(out, torch.float32, "out"), T, k, E, H, I, int(act_kind),
                                       _stream(w13)))
    return out, h, act_mid


def ffn_reserve(max_tokens, max_top_k, n_experts, hidden, n_inter):
    """Workspace for both expert layers up to these sizes (ft_moe_ffn_reserve)."""
    _check(load().ft_moe_ffn_reserve(max_tokens, max_top_k, n_experts, hidden, n_inter))


def block_dots(weights, act, topk_ids, out=None):
    """Diagnostic: int32 [T*k, N, K/32] per-block integer dots (ft_moe_block_dots)."""
    torch = _torch()
    E, N, K, T, k = _matmul_shape(weights, act, topk_ids)
    if out is None:
        out = torch.empty((T * k, N, K // 32), dtype=torch.int32, device=weights.device)
    po = _dev(out, torch.int32, "out")
    _check(load().ft_moe_block_dots(ctypes.c_void_p(weights.data_ptr()), ctypes.c_void_p(act.data_ptr()),
                                    ctypes.c_void_p(topk_ids.data_ptr()), po, T, k, E, N, K, _stream(weights)))
    return out


def workspace_bytes(tokens, top_k, n_experts, nrows, ncols) -> int:
    return int(load().ft_moe_workspace_bytes(tokens, top_k, n_experts, nrows, ncols))


def reserve(max_tokens, max_top_k, n_experts, nrows, ncols):
    _check(load().ft_moe_reserve(max_tokens, max_top_k, n_experts, nrows, ncols))


def release():
    _check(load().ft_moe_release())


def read_device_error(stream=None) -> int:
    """Synchronize, return and clear the library's device error word (no raise)."""
    torch = _torch()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream if stream is None else stream)
    flags = ctypes.c_uint32(0)
    st = load().ft_moe_read_device_error(s, ctypes.byref(flags))
    if st not in (FT_OK, FT_ERR_DEVICE_FLAG):
        raise FtError(st, last_error())
    return int(flags.value)


def debug_stream_read(buf, nbytes=None, stream=None):
    """Measurement hook (ft_debug_stream_read): stream the first nbytes (default:
    all, rounded down to 16) of a CUDA tensor through the SMs, nothing written."""
    torch = _torch()
    if not isinstance(buf, torch.Tensor) or not buf.is_cuda or not buf.is_contiguous():
        raise TypeError("buf must be a contiguous CUDA tensor")
    n = buf.numel() * buf.element_size() if nbytes is None else int(nbytes)
    n -= n % 16
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream if stream is None else stream)
    _check(load().ft_debug_stream_read(ctypes.c_void_p(buf.data_ptr()), n, s))


def debug_wait_timeout(limit_ns: int, stream=None):
    """Test hook (ft_debug_wait_timeout): a kernel whose bounded wait gives up
    after limit_ns; the flag it raises is read with read_device_error()."""
    torch = _torch()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream if stream is None else stream)
    _check(load().ft_debug_wait_timeout(int(limit_ns), s))


def set_path(path) -> int:
    p = PATHS[path] if isinstance(path, str) else int(path)
    prev = load().ft_moe_set_path(p)
    if prev < 0:
        raise ValueError(f"unknown path {path!r}")
    return prev


def selected_path(tokens, top_k, n_experts, nrows, ncols, wtype="q4_0") -> int:
    """The path (FT_PATH_GEMV / FT_PATH_GEMM) the matmul would take for this shape
    and weight type under the current setting, or -1."""
    if wtype == "q4_0":
        return int(load().ft_moe_selected_path(tokens, top_k, n_experts, nrows, ncols))
    return int(load().ft_moe_gguf_selected_path(WEIGHT_TYPES[wtype][0], tokens, top_k, n_experts, nrows, ncols))


def profile_enable(max_calls: int):
    """Record CUDA events around this library's kernels for the next max_calls calls (0 stops)."""
    _check(load().ft_profile_enable(int(max_calls)))


def profile_read() -> dict:
    """Synchronize on the recorded events; summed kernel times (ms), calls and launches; resets."""
    q, r, m = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    n, nl = ctypes.c_int64(), ctypes.c_int64()
    _check(load().ft_profile_read(ctypes.byref(q), ctypes.byref(r), ctypes.byref(m), ctypes.byref(n),
                                  ctypes.byref(nl)))
    return {"quantize_ms": q.value, "route_ms": r.value, "matmul_ms": m.value, "calls": n.value,
            "launches": nl.value}
