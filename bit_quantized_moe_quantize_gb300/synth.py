"""Seeded synthetic inputs for the routed Q4_0 x Q8_1 MoE expert matmul.

This module only draws random numbers and stores them in the layouts the
library consumes.  It holds none of the matmul, activation-quantizer or
router arithmetic: both the CUDA path and the CPU oracle receive what this
module returns, and nothing else is shared between them.

The one encoding step here is the storage format of the synthetic *weights*:
expert weights are drawn in fp32 and stored as GGUF Q4_0 blocks, because the
routed matmul consumes Q4_0 weights as an input (the pages serve GGUF Q4_0
checkpoints: FreeToken PR #185, section "Tested on").  The CUDA path never
quantizes weights.  The oracle carries its own, independently written Q4_0
quantizer and a test checks that both produce identical bytes.

Workloads (shapes, seeds, value distributions):

* tiny layer          E=8,   k=2, K=256,  N=128,   T=16                 seed 0
* prefill             E=128, k=8, K=2816, N=1408,  T in {2048,4096,8191} seed 1
  (the shape of the kernel benchmark on FreeToken PR #185, "Performance")
* launch-limit        E=8,   k=2, K=256,  N=128,   T in {8192,16384}    seed 2
  (T*k = 65536 and 131072 slots, past the 65535 grid.z cap of "Problem")
* qwen3-30b-a3b shape E=128, k=8, K=2048, N=768,   T in {1,8,64,512,8192},
  Zipf(1.1) expert popularity                                           seed 3
* mixtral-8x7b shape  E=8,   k=2, K=4096, N=14336, T in {1,32,32768},
  1% outlier channels x20                                               seed 4
  (the two model shapes whose long prompts failed on mlxcel PR #652)

Weights are fp32 N(0, 0.02) stored as Q4_0, activations fp16 N(0, 1), routing
draws k distinct experts per token (uniform, or sequential weighted draws
without replacement for the Zipf workload, done with the equivalent
Gumbel-top-k construction).
"""

from __future__ import annotations

import dataclasses

import numpy as np

QK = 32                 # values per quantization block
Q4_0_BYTES = 18         # fp16 d + 16 bytes of nibbles
Q8_1_BYTES = 36         # fp16 d + fp16 s + 32 int8


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_experts: int
    top_k: int
    ncols: int
    nrows: int
    tokens: tuple
    routing: str = "uniform"      # "uniform" | "zipf"
    zipf_s: float = 1.1
    outlier_frac: float = 0.0
    outlier_scale: float = 20.0
    seed: int = 0
    w_std: float = 0.02


WORKLOADS = {
    "tiny": Workload("tiny", 8, 2, 256, 128, (16,), seed=0),
    "prefill": Workload("prefill", 128, 8, 2816, 1408, (2048, 4096, 8191), seed=1),
    "launch_limit": Workload("launch_limit", 8, 2, 256, 128, (8192, 16384), seed=2),
    "qwen3_30b_a3b": Workload("qwen3_30b_a3b", 128, 8, 2048, 768, (1, 8, 64, 512, 8192),
                              routing="zipf", seed=3),
    "mixtral_8x7b": Workload("mixtral_8x7b", 8, 2, 4096, 14336, (1, 32, 32768),
                             outlier_frac=0.01, seed=4),
}

# stream ids inside one workload seed
_S_WEIGHTS, _S_ACT, _S_ROUTE, _S_OUTLIER, _S_RANK, _S_GGUF = 0, 1, 2, 3, 4, 5

# the other GGUF weight types with 32-weight blocks: bytes per block, offset of
# the code bytes, whether the block stores an fp16 m after d, GGML type number
GGUF_TYPES = {"q4_0": (18, 2, False, 2), "q4_1": (20, 4, True, 3), "q5_0": (22, 2, False, 6),
              "q5_1": (24, 4, True, 7), "q8_0": (34, 2, False, 8),
              "q4_k": (144, 4, False, 12), "q5_k": (176, 4, False, 13), "q6_k": (210, 0, False, 14),
              "q2_k": (84, 0, False, 10), "q3_k": (110, 0, False, 11)}
KQUANTS = ("q4_k", "q5_k", "q6_k", "q2_k", "q3_k")     # 256 weights per (super-)block; the others hold 32


def _rng(seed: int, stream: int, *extra: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, *extra])))


def encode_q4_0(w: np.ndarray) -> np.ndarray:
    """Store fp32 weights (last axis a multiple of 32) as GGUF Q4_0 bytes.

    Per 32-block: m = the element of largest magnitude (first on ties, sign
    kept), d = m / -8 in fp32, q = clamp(round_half_away(w / d) + 8, 0, 15)
    (q = 8 when d == 0), stored as fp16 d followed by 16 bytes whose low
    nibble is q[j] and high nibble q[j+16].  Returns uint8 [..., K/32, 18].
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    lead = w.shape[:-1]
    blocks = w.reshape(-1, QK)
    nb = blocks.shape[0]
    idx = np.argmax(np.abs(blocks), axis=1)
    m = blocks[np.arange(nb), idx]
    d = (m / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (blocks / d[:, None]).astype(np.float64)     # fp32 division, widened exactly
    r = np.trunc(quot + np.copysign(0.5, quot))               # half away from zero, exact in fp64
    q = np.clip(np.where(d[:, None] == 0, 0.0, r) + 8.0, 0, 15).astype(np.uint8)
    out = np.empty((nb, Q4_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(nb, 2)
    out[:, 2:] = q[:, :16] | (q[:, 16:] << 4)
    return out.reshape(*lead, w.shape[-1] // QK, Q4_0_BYTES)


def make_weights(wl: Workload, chunk_rows: int = 1 << 16) -> np.ndarray:
    """Q4_0 expert weights, uint8 [E, N, K/32, 18]."""
    E, N, K = wl.n_experts, wl.nrows, wl.ncols
    out = np.empty((E, N, K // QK, Q4_0_BYTES), dtype=np.uint8)
    rng = _rng(wl.seed, _S_WEIGHTS)
    flat = out.reshape(E * N, K // QK, Q4_0_BYTES)
    for r0 in range(0, E * N, chunk_rows):
        r1 = min(E * N, r0 + chunk_rows)
        w = rng.standard_normal((r1 - r0, K), dtype=np.float32) * np.float32(wl.w_std)
        flat[r0:r1] = encode_q4_0(w)
    return out


def make_weights_gguf(wl: Workload, wtype: str, chunk_rows: int = 1 << 16) -> np.ndarray:
    """Expert weights as random valid blocks of a GGUF type, uint8
    [E, N, K/32, bytes] (K/256 super-blocks for the K-quants).

    Q4_0 goes through make_weights.  For the others every code byte (nibbles,
    5th-bit words, int8 codes, packed 6-bit sub-block scales and mins) is
    uniform random, d = fp16(0.0005 + 0.002 |z|) and, for the types with an
    offset, m = fp16(-d * L / 2 * (1 + 0.1 z')) with L the number of levels,
    so that the weights centre near zero like trained ones; the K-quants take
    0.05 of that d and dmin = fp16(d L / 2 |1 + 0.1 z'|) (the 6-bit sub-block
    scale and min multiply both); Q6_K takes random int8 scales and
    d = fp16(0.00002 (0.5 + |z|)).  Random bytes are valid blocks
    of these formats; no weight quantization is involved.
    """
    if wtype == "q4_0":
        return make_weights(wl, chunk_rows)
    bb, code0, has_m, tid = GGUF_TYPES[wtype]
    E, N, K = wl.n_experts, wl.nrows, wl.ncols
    nb = K // (256 if wtype in KQUANTS else QK)
    out = np.empty((E * N, nb, bb), dtype=np.uint8)
    rng = _rng(wl.seed, _S_GGUF, tid)
    levels = {"q4_1": 16, "q5_1": 32}.get(wtype, 0)
    for r0 in range(0, E * N, chunk_rows):
        r1 = min(E * N, r0 + chunk_rows)
        n = r1 - r0
        if wtype in ("q2_k", "q3_k"):     # random code, mask and scale bytes, fp16 d (and dmin) last
            head = 80 if wtype == "q2_k" else 108
            out[r0:r1, :, 0:head] = rng.integers(0, 256, size=(n, nb, head), dtype=np.uint8)
            dd = np.float32(0.0005 if wtype == "q2_k" else 0.00015) * (
                np.float32(0.5) + np.abs(rng.standard_normal((n, nb), dtype=np.float32)))
            out[r0:r1, :, head:head + 2] = dd.astype(np.float16).view(np.uint8).reshape(n, nb, 2)
            if wtype == "q2_k":      # dmin ~ d * 1.5 centres scale * q - min near zero
                dm = dd * np.float32(1.5)
                out[r0:r1, :, 82:84] = dm.astype(np.float16).view(np.uint8).reshape(n, nb, 2)
            continue
        if wtype == "q6_k":     # random code and scale bytes, fp16 d last
            out[r0:r1, :, 0:208] = rng.integers(0, 256, size=(n, nb, 208), dtype=np.uint8)
            d6 = np.float32(0.00002) * (np.float32(0.5) + np.abs(rng.standard_normal((n, nb), dtype=np.float32)))
            out[r0:r1, :, 208:210] = d6.astype(np.float16).view(np.uint8).reshape(n, nb, 2)
            continue
        d = (np.float32(0.0005) + np.float32(0.002) * np.abs(rng.standard_normal((n, nb), dtype=np.float32)))
        if wtype in KQUANTS:      # super-block scales of the 6-bit sub-block scales and mins
            d = d * np.float32(0.05)
            half_levels = np.float32(8 if wtype == "q4_k" else 16)
            dmin = d * half_levels * np.abs(np.float32(1) + np.float32(0.1) * rng.standard_normal((n, nb), dtype=np.float32))
            out[r0:r1, :, 2:4] = dmin.astype(np.float16).view(np.uint8).reshape(n, nb, 2)
        out[r0:r1, :, 0:2] = d.astype(np.float16).view(np.uint8).reshape(n, nb, 2)
        if has_m:
            z = rng.standard_normal((n, nb), dtype=np.float32)
            m = -d * np.float32(levels / 2) * (np.float32(1) + np.float32(0.1) * z)
            out[r0:r1, :, 2:4] = m.astype(np.float16).view(np.uint8).reshape(n, nb, 2)
        out[r0:r1, :, code0:] = rng.integers(0, 256, size=(n, nb, bb - code0), dtype=np.uint8)
    return out.reshape(E, N, nb, bb)


def make_activations(wl: Workload, tokens: int) -> np.ndarray:
    """fp16 activations [T, K]; outlier channels are scaled before fp16 rounding."""
    K = wl.ncols
    x = _rng(wl.seed, _S_ACT, tokens).standard_normal((tokens, K), dtype=np.float32)
    if wl.outlier_frac > 0:
        n_out = int(np.floor(wl.outlier_frac * K))
        ch = _rng(wl.seed, _S_OUTLIER).choice(K, size=n_out, replace=False)
        x[:, ch] *= np.float32(wl.outlier_scale)
    return x.astype(np.float16)


def make_topk_ids(wl: Workload, tokens: int) -> np.ndarray:
    """int32 [T, k]: k distinct experts per token, in draw order."""
    E, k = wl.n_experts, wl.top_k
    rng = _rng(wl.seed, _S_ROUTE, tokens)
    u = rng.random((tokens, E))
    if wl.routing == "uniform":
        keys = u
    elif wl.routing == "zipf":
        rank = np.empty(E, dtype=np.float64)
        rank[_rng(wl.seed, _S_RANK).permutation(E)] = np.arange(1, E + 1)
        logp = -wl.zipf_s * np.log(rank)
        # Gumbel-top-k == sequential weighted draws without replacement
        keys = logp[None, :] - np.log(-np.log(np.clip(u, 1e-300, 1.0)))
    else:
        raise ValueError(wl.routing)
    ids = np.argsort(-keys, axis=1, kind="stable")[:, :k]
    return np.ascontiguousarray(ids.astype(np.int32))


def make_case(name: str, tokens: int, with_weights: bool = True):
    wl = WORKLOADS[name]
    return dict(
        workload=wl,
        tokens=tokens,
        weights=make_weights(wl) if with_weights else None,
        x=make_activations(wl, tokens),
        topk_ids=make_topk_ids(wl, tokens),
    )


def custom_workload(n_experts, top_k, ncols, nrows, seed, routing="uniform", **kw) -> Workload:
    return Workload("custom", n_experts, top_k, ncols, nrows, (), routing=routing, seed=seed, **kw)
