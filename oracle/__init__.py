"""ctypes binding of the CPU oracle (ft_oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the CPU-baseline
leg of the benchmark may import this package; the CUDA library and its Python
binding never do.  The shared object is built with gcc into ``_build/`` under
a name that carries the source hash, so a stale build is never picked up.
"""

from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ft_oracle.c")
_HDR = os.path.join(_HERE, "ft_oracle.h")
_LOCK = threading.Lock()
_LIB = None

QK = 32
Q4_0_BYTES = 18
Q8_1_BYTES = 36


def _source_hash(src=_SRC) -> str:
    h = hashlib.sha256()
    for p in (src, _HDR):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def build(src: str = _SRC, out_dir: str | None = None, extra_flags=()) -> str:
    """Compile the oracle (or a copy of it) with gcc; returns the .so path."""
    out_dir = out_dir or os.path.join(_HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, f"liboracle_{_source_hash(src)}.so")
    if not os.path.exists(so):
        tmp = so + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
               "-I", _HERE, *extra_flags, src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, so)
    return so


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Numpy-facing wrapper around one loaded oracle shared object."""

    def __init__(self, so_path: str):
        L = ctypes.CDLL(so_path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_double.restype = ctypes.c_double
        L.oracle_float_to_half.argtypes = [ctypes.c_float]
        L.oracle_float_to_half.restype = ctypes.c_uint16
        L.oracle_quantize_q4_0.argtypes = [vp, i64, vp]
        L.oracle_dequantize_q4_0.argtypes = [vp, i64, vp]
        L.oracle_quantize_q8_1.argtypes = [vp, i64, i64, vp]
        L.oracle_dequantize_q8_1.argtypes = [vp, i64, vp]
        L.oracle_route.argtypes = [vp, i64, i32, vp, vp, vp]
        L.oracle_route.restype = i64
        L.oracle_block_dot.argtypes = [vp, vp]
        L.oracle_block_dot.restype = i32
        L.oracle_moe_q4_0_q8_1.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64]
        L.oracle_moe_sample.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, vp, vp, i64, vp]
        L.oracle_moe_slots_q4_0_q8_1.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64]
        L.oracle_moe_ep_q4_0_q8_1.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i32, i64, i64]
        L.oracle_moe_block_dots.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, vp]
        L.oracle_moe_dequant_bruteforce.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, vp]
        L.oracle_act_mul.argtypes = [vp, i64, i64, i32, vp]
        L.oracle_repack_q4_0_soa.argtypes = [vp, i64, vp, vp]
        L.oracle_gguf_block_bytes.argtypes = [i32]
        L.oracle_gguf_block_bytes.restype = i32
        L.oracle_dequantize_gguf.argtypes = [i32, vp, i64, vp]
        L.oracle_gguf_block_dot.argtypes = [i32, vp, vp]
        L.oracle_gguf_block_dot.restype = i32
        L.oracle_moe_gguf_q8_1.argtypes = [i32, vp, vp, vp, vp, i64, i32, i32, i64, i64]
        L.oracle_act_mul_quantize_q8_1.argtypes = [vp, i64, i64, i32, vp]
        self.lib = L
        self.path = so_path

    # fp16 ------------------------------------------------------------
    def half_to_double(self, h: int) -> float:
        return self.lib.oracle_half_to_double(int(h))

    def float_to_half(self, f: float) -> int:
        return int(self.lib.oracle_float_to_half(float(np.float32(f))))

    # formats ---------------------------------------------------------
    def quantize_q4_0(self, w: np.ndarray) -> np.ndarray:
        w = np.ascontiguousarray(w, dtype=np.float32)
        assert w.shape[-1] % QK == 0
        nb = w.size // QK
        out = np.empty((nb, Q4_0_BYTES), dtype=np.uint8)
        self.lib.oracle_quantize_q4_0(_p(w), nb, _p(out))
        return out.reshape(*w.shape[:-1], w.shape[-1] // QK, Q4_0_BYTES)

    def dequantize_q4_0(self, blocks: np.ndarray) -> np.ndarray:
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
        nb = blocks.size // Q4_0_BYTES
        out = np.empty(nb * QK, dtype=np.float64)
        self.lib.oracle_dequantize_q4_0(_p(blocks), nb, _p(out))
        return out.reshape(*blocks.shape[:-2], blocks.shape[-2] * QK)

    def quantize_q8_1(self, x_fp16: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x_fp16, dtype=np.float16)
        T, K = x.shape
        assert K % QK == 0
        out = np.empty((T, K // QK, Q8_1_BYTES), dtype=np.uint8)
        self.lib.oracle_quantize_q8_1(_p(x.view(np.uint16)), T, K, _p(out))
        return out

    def dequantize_q8_1(self, blocks: np.ndarray) -> np.ndarray:
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
        nb = blocks.size // Q8_1_BYTES
        out = np.empty(nb * QK, dtype=np.float64)
        self.lib.oracle_dequantize_q8_1(_p(blocks), nb, _p(out))
        return out.reshape(*blocks.shape[:-2], blocks.shape[-2] * QK)

    # other GGUF weight types -----------------------------------------
    GGUF = {"q4_0": 2, "q4_1": 3, "q5_0": 6, "q5_1": 7, "q8_0": 8, "q4_k": 12, "q5_k": 13, "q6_k": 14, "q2_k": 10, "q3_k": 11}
    KQUANTS = (10, 11, 12, 13, 14)

    def gguf_block_bytes(self, wtype) -> int:
        return int(self.lib.oracle_gguf_block_bytes(self.GGUF.get(wtype, wtype)))

    def dequantize_gguf(self, wtype, blocks: np.ndarray) -> np.ndarray:
        t = self.GGUF.get(wtype, wtype)
        bb = self.gguf_block_bytes(t)
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
        assert blocks.shape[-1] == bb
        nb = blocks.size // bb
        per = 256 if t in self.KQUANTS else QK
        out = np.empty(nb * per, dtype=np.float64)
        self.lib.oracle_dequantize_gguf(t, _p(blocks), nb, _p(out))
        return out.reshape(*blocks.shape[:-2], blocks.shape[-2] * per)

    def gguf_block_dot(self, wtype, w_block: np.ndarray, a_block: np.ndarray) -> int:
        t = self.GGUF.get(wtype, wtype)
        w = np.ascontiguousarray(w_block, dtype=np.uint8)
        a = np.ascontiguousarray(a_block, dtype=np.uint8)
        assert w.size == self.gguf_block_bytes(t) and a.size == Q8_1_BYTES
        return int(self.lib.oracle_gguf_block_dot(t, _p(w), _p(a)))

    def moe_gguf(self, wtype, weights, act, topk_ids) -> np.ndarray:
        """weights [E, N, K/32, bytes of the type] x Q8_1 act [T, K/32, 36] -> fp32 [T, k, N]."""
        t = self.GGUF.get(wtype, wtype)
        w = np.ascontiguousarray(weights, dtype=np.uint8)
        a = np.ascontiguousarray(act, dtype=np.uint8)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        E, N, nb, bb = w.shape
        assert bb == self.gguf_block_bytes(t)
        per = 256 if t in self.KQUANTS else QK
        T, k = ids.shape
        assert a.shape == (T, nb * per // QK, Q8_1_BYTES)
        out = np.empty((T, k, N), dtype=np.float32)
        self.lib.oracle_moe_gguf_q8_1(t, _p(w), _p(a), _p(ids), _p(out), T, k, E, N, nb * per)
        return out

    # SoA repack --------------------------------------------------------
    def repack_q4_0_soa(self, blocks: np.ndarray):
        """Q4_0 blocks [..., 18] -> (nibble bytes uint8 [n, 16], scales fp16 [n])."""
        b = np.ascontiguousarray(blocks, dtype=np.uint8)
        n = b.size // Q4_0_BYTES
        qs = np.empty((n, 16), dtype=np.uint8)
        d = np.empty(n, dtype=np.uint16)
        self.lib.oracle_repack_q4_0_soa(_p(b), n, _p(qs), _p(d))
        return qs, d.view(np.float16)

    # gated activation ------------------------------------------------
    ACT_SILU = 0
    ACT_GELU_TANH = 1

    def act_mul(self, h: np.ndarray, kind: int) -> np.ndarray:
        """a = act(h[..., :I]) * h[..., I:] in fp64, rounded to fp32."""
        h = np.ascontiguousarray(h, dtype=np.float32)
        two_i = h.shape[-1]
        assert two_i % 2 == 0
        rows = h.size // two_i if two_i else 0
        out = np.empty((*h.shape[:-1], two_i // 2), dtype=np.float32)
        self.lib.oracle_act_mul(_p(h), rows, two_i // 2, int(kind), _p(out))
        return out

    def act_mul_quantize_q8_1(self, h: np.ndarray, kind: int) -> np.ndarray:
        """Q8_1 rows [..., I/32, 36] of act_mul(h, kind)."""
        h = np.ascontiguousarray(h, dtype=np.float32)
        two_i = h.shape[-1]
        assert two_i % (2 * QK) == 0
        rows = h.size // two_i if two_i else 0
        out = np.empty((*h.shape[:-1], two_i // 2 // QK, Q8_1_BYTES), dtype=np.uint8)
        self.lib.oracle_act_mul_quantize_q8_1(_p(h), rows, two_i // 2, int(kind), _p(out))
        return out

    def moe_ffn(self, w13, w2, act, topk_ids, kind: int):
        """Both expert layers of the routed MoE block, per slot: h = W13 x (gate |
        up rows), a = Q8_1(act(gate) * up), out = W2 a -> [T, k, hidden] fp32,
        with h and a returned too."""
        h = self.moe(w13, act, topk_ids)
        T, k = np.asarray(topk_ids).shape
        a = self.act_mul_quantize_q8_1(h.reshape(T * k, -1), kind)
        out = self.moe_slots(w2, a, topk_ids)
        return out, h, a

    # route -----------------------------------------------------------
    def route(self, topk_ids: np.ndarray, n_experts: int):
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(-1)
        S = ids.size
        counts = np.empty(n_experts, dtype=np.int32)
        offsets = np.empty(n_experts + 1, dtype=np.int32)
        perm = np.empty(S, dtype=np.int32)
        bad = self.lib.oracle_route(_p(ids), S, n_experts, _p(counts), _p(offsets), _p(perm))
        return counts, offsets, perm, int(bad)

    # dot -------------------------------------------------------------
    def block_dot(self, w_block: np.ndarray, a_block: np.ndarray) -> int:
        w = np.ascontiguousarray(w_block, dtype=np.uint8)
        a = np.ascontiguousarray(a_block, dtype=np.uint8)
        assert w.size == Q4_0_BYTES and a.size == Q8_1_BYTES
        return int(self.lib.oracle_block_dot(_p(w), _p(a)))

    @staticmethod
    def _shape(weights, act, topk_ids):
        E, N, nb, _ = weights.shape
        T = act.shape[0]
        k = topk_ids.shape[1]
        return E, N, nb * QK, T, k

    def moe(self, weights, act, topk_ids) -> np.ndarray:
        weights = np.ascontiguousarray(weights, dtype=np.uint8)
        act = np.ascontiguousarray(act, dtype=np.uint8)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        E, N, K, T, k = self._shape(weights, act, ids)
        out = np.empty((T, k, N), dtype=np.float32)
        self.lib.oracle_moe_q4_0_q8_1(_p(weights), _p(act), _p(ids), _p(out), T, k, E, N, K)
        return out

    def moe_slots(self, weights, act_slots, topk_ids) -> np.ndarray:
        """Per-slot activations: act_slots is Q8_1 [T*k][K/32], row s for slot s."""
        weights = np.ascontiguousarray(weights, dtype=np.uint8)
        act_slots = np.ascontiguousarray(act_slots, dtype=np.uint8)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        E, N, nb, _ = weights.shape
        T, k = ids.shape
        assert act_slots.shape == (T * k, nb, 36), act_slots.shape
        K = nb * QK
        out = np.empty((T, k, N), dtype=np.float32)
        self.lib.oracle_moe_slots_q4_0_q8_1(_p(weights), _p(act_slots), _p(ids), _p(out), T, k, E, N, K)
        return out

    def moe_ep(self, weights_local, act, topk_ids, n_global, expert_start) -> np.ndarray:
        """Expert-parallel shard: weights_local = experts [expert_start, expert_start + E_local)
        of n_global; topk_ids hold global ids; non-local slots give zero rows."""
        weights_local = np.ascontiguousarray(weights_local, dtype=np.uint8)
        act = np.ascontiguousarray(act, dtype=np.uint8)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        E_local, N, K, T, k = self._shape(weights_local, act, ids)
        out = np.empty((T, k, N), dtype=np.float32)
        self.lib.oracle_moe_ep_q4_0_q8_1(_p(weights_local), _p(act), _p(ids), _p(out), T, k, n_global,
                                         expert_start, E_local, N, K)
        return out

    def moe_sample(self, weights, act, topk_ids, slots, rows) -> np.ndarray:
        weights = np.ascontiguousarray(weights, dtype=np.uint8)
        act = np.ascontiguousarray(act, dtype=np.uint8)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        E, N, K, T, k = self._shape(weights, act, ids)
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        assert slots.shape == rows.shape
        assert slots.size == 0 or (slots.min() >= 0 and slots.max() < T * k)
        assert rows.size == 0 or (rows.min() >= 0 and rows.max() < N)
        out = np.empty(slots.size, dtype=np.float64)
        self.lib.oracle_moe_sample(_p(weights), _p(act), _p(ids), T, k, E, N, K,
                                   _p(slots), _p(rows), slots.size, _p(out))
        return out

    def moe_block_dots(self, weights, act, topk_ids) -> np.ndarray:
        weights = np.ascontiguousarray(weights, dtype=np.uint8)
        act = np.ascontiguousarray(act, dtype=np.uint8)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        E, N, K, T, k = self._shape(weights, act, ids)
        out = np.empty((T * k, N, K // QK), dtype=np.int32)
        self.lib.oracle_moe_block_dots(_p(weights), _p(act), _p(ids), T, k, E, N, K, _p(out))
        return out

    def moe_dequant_bruteforce(self, weights, act, topk_ids) -> np.ndarray:
        weights = np.ascontiguousarray(weights, dtype=np.uint8)
        act = np.ascontiguousarray(act, dtype=np.uint8)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        E, N, K, T, k = self._shape(weights, act, ids)
        out = np.empty((T, k, N), dtype=np.float64)
        self.lib.oracle_moe_dequant_bruteforce(_p(weights), _p(act), _p(ids), T, k, E, N, K, _p(out))
        return out


def get() -> Oracle:
    """The oracle built from the committed source (built once per process)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = Oracle(build())
        return _LIB
