"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the workload definitions and arithmetic
fix.  ``test_oracle_pins.py`` runs them on the committed oracle (all must
pass) and on mutated copies of it (each mutant must fail at least one), which
shows the pins are sensitive to the plausible mistakes they are meant to catch.

Block formats (GGUF, restated): Q4_0 = fp16 d + 16 bytes, weight j < 16 in the
low nibble of byte j, weight j + 16 in its high nibble, value (q - 8) d;
Q8_1 = fp16 d + fp16 s + 32 int8 q, value q d, s = d * sum(q).
"""

from __future__ import annotations

import numpy as np

QK = 32


# ------------------------------------------------------------------ helpers
def q4_block(d_bits: int, q: list[int]) -> np.ndarray:
    """Assemble one Q4_0 block from fp16 bits and 32 nibble values (test-side, by hand)."""
    assert len(q) == 32
    b = np.zeros(18, dtype=np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    for j in range(16):
        b[2 + j] = (q[j] & 15) | ((q[j + 16] & 15) << 4)
    return b


def q8_block(d_bits: int, s_bits: int, q: list[int]) -> np.ndarray:
    b = np.zeros(36, dtype=np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    b[2], b[3] = s_bits & 0xFF, s_bits >> 8
    b[4:] = np.asarray(q, dtype=np.int8).view(np.uint8)
    return b


def numpy_decode_q4_0(w: np.ndarray) -> np.ndarray:
    """Independent vectorised decode of Q4_0 bytes [..., nb, 18] -> fp64 [..., nb*32]."""
    d = np.ascontiguousarray(w[..., 0:2]).view(np.float16)[..., 0].astype(np.float64)
    qs = w[..., 2:].astype(np.int64)
    q = np.concatenate([qs & 15, qs >> 4], axis=-1) - 8
    v = q * d[..., None]
    return v.reshape(*w.shape[:-2], w.shape[-2] * QK)


def numpy_decode_q8_1(a: np.ndarray) -> np.ndarray:
    d = np.ascontiguousarray(a[..., 0:2]).view(np.float16)[..., 0].astype(np.float64)
    q = np.ascontiguousarray(a[..., 4:]).view(np.int8).astype(np.float64)
    v = q * d[..., None]
    return v.reshape(*a.shape[:-2], a.shape[-2] * QK)


def tiny_case(seed=0, E=6, k=2, K=128, N=24, T=7, x_scale=1.0):
    from bit_quantized_moe_quantize_gb300 import synth
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
    x = (rng.standard_normal((T, K)) * x_scale).astype(np.float16)
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    return synth.encode_q4_0(w), x, ids


# ------------------------------------------------------------------- fp16
def pin_fp16(o):
    special = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6,
                        2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26,
                        1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 0.1, 1 / 3, 2048.5, 4097.0],
                       dtype=np.float32)
    rng = np.random.default_rng(1)
    rand = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 18, 20000))).astype(np.float32)
    for f in np.concatenate([special, -special, rand]):
        with np.errstate(over="ignore"):
            want = int(np.float32(f).astype(np.float16).view(np.uint16))
        got = o.float_to_half(f)
        assert got == want, (float(f), hex(got), hex(want))
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b, r in zip(bits, ref):
        if np.isnan(r):
            continue
        assert o.half_to_double(int(b)) == r, hex(int(b))


# ------------------------------------------------------------------- Q4_0
def pin_q4_0_hand(o):
    # largest magnitude -1.0 first at index 0 -> d = 0.125 (fp16 0x3000); w = (q - 8) d
    q = [i // 2 for i in range(32)]
    w = np.array([(qi - 8) * 0.125 for qi in q], dtype=np.float32)
    got = o.quantize_q4_0(w[None, :])[0, 0]
    want = np.array([0x00, 0x30] + [(j // 2) | ((j // 2 + 8) << 4) for j in range(16)],
                    dtype=np.uint8)
    assert np.array_equal(got, want), (got, want)
    # positive extreme: m = +2 -> d = -0.25 (0xB400); 2 -> q 0, 1 -> 4, -1 -> 12, 0 -> 8
    w = np.zeros(32, dtype=np.float32)
    w[0], w[1], w[17] = 2.0, 1.0, -1.0
    got = o.quantize_q4_0(w[None, :])[0, 0]
    want = np.full(18, 0x88, dtype=np.uint8)
    want[0], want[1] = 0x00, 0xB4
    want[2] = 0x80 | 0x0            # qs[0]: low q[0] = 0, high q[16] = 8
    want[3] = (12 << 4) | 4         # qs[1]: low q[1] = 4, high q[17] = 12
    assert np.array_equal(got, want), (got, want)
    # opposite extreme saturates: m = +1 first, -1 -> round(8) + 8 = 16 -> 15
    w = np.zeros(32, dtype=np.float32)
    w[0], w[5] = 1.0, -1.0
    got = o.quantize_q4_0(w[None, :])[0, 0]
    assert got[2] & 15 == 0 and got[2 + 5] & 15 == 15
    # all zero -> d = +0 / -8 = -0.0 in IEEE arithmetic (fp16 0x8000), every nibble 8
    got = o.quantize_q4_0(np.zeros((1, 32), np.float32))[0, 0]
    assert np.array_equal(got, np.array([0x00, 0x80] + [0x88] * 16, dtype=np.uint8))


def pin_q4_0_nearest_level(o):
    """q is the nearest level to w/d (ties away from zero), clamped: brute-force search."""
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((64, 32)) * 0.02).astype(np.float32)
    w[3, 7] = -np.abs(w[3]).max() * 1.5  # a negative extreme
    blocks = o.quantize_q4_0(w)[:, 0]
    for bi in range(w.shape[0]):
        m = w[bi][np.argmax(np.abs(w[bi]))]
        d = np.float32(m) / np.float32(-8.0)
        d16 = int(np.float32(d).astype(np.float16).view(np.uint16))
        assert int(blocks[bi, 0]) | (int(blocks[bi, 1]) << 8) == d16
        for i in range(32):
            r = float(np.float32(w[bi, i]) / d)
            best, bestd = None, None
            for c in range(-8, 8 + 1):
                dist = abs(r - c)
                if bestd is None or dist < bestd - 1e-12 or (abs(dist - bestd) <= 1e-12 and abs(c) > abs(best)):
                    best, bestd = c, dist
            qwant = min(15, max(0, best + 8))
            byte = blocks[bi, 2 + (i % 16)]
            qgot = (byte & 15) if i < 16 else (byte >> 4)
            assert qgot == qwant, (bi, i, qgot, qwant)
        # the extreme element always maps to level 0
        i = int(np.argmax(np.abs(w[bi])))
        byte = blocks[bi, 2 + (i % 16)]
        assert ((byte & 15) if i < 16 else (byte >> 4)) == 0


def pin_q4_0_matches_generator(o):
    from bit_quantized_moe_quantize_gb300 import synth
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((3, 5, 256)) * 0.02).astype(np.float32)
    w[0, 0, :32] = 0.0
    w[1, 2, 40] = -w[1, 2, 32:64].max() * 3
    assert np.array_equal(o.quantize_q4_0(w), synth.encode_q4_0(w))


def pin_q4_0_dequant(o):
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((10, 64)) * 0.02).astype(np.float32)
    blocks = o.quantize_q4_0(w)
    deq = o.dequantize_q4_0(blocks)
    assert np.array_equal(deq, numpy_decode_q4_0(blocks))
    # round trip: within half a level of w/d (plus the fp16 rounding of d), except where
    # w/d lies past 7.5, the top level 7 being the last one (then within one level)
    wb = w.reshape(10, 2, 32)
    d32 = np.array([[np.float32(b[np.argmax(np.abs(b))]) / np.float32(-8) for b in row] for row in wb])
    r = wb.astype(np.float64) / d32[..., None]
    err = np.abs(deq.reshape(10, 2, 32) - wb.astype(np.float64))
    ad = np.abs(d32)[..., None]
    sat = r > 7.5
    bound = np.where(sat, 1.0, 0.5) * ad * (1 + 1e-6) + 8 * ad * 2.0 ** -11
    assert np.all(err <= bound)
    assert np.all(np.abs(r) <= 8 * (1 + 1e-6))


# ------------------------------------------------------------------- Q8_1
def _q8_numpy_fp32(x16: np.ndarray):
    """fp32 replay of the activation quantizer as the workload defines it."""
    x = x16.astype(np.float32).reshape(-1, 32)
    amax = np.abs(x).max(axis=1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (x / d[:, None]).astype(np.float64)
    q = np.where(amax[:, None] == 0, 0, np.trunc(r + np.copysign(0.5, r)))
    q = np.clip(q, -127, 127).astype(np.int64)
    s = (d * q.sum(axis=1).astype(np.float32)).astype(np.float32)
    return d.astype(np.float16), s.astype(np.float16), q


def pin_q8_1_hand(o):
    # all 2.0: d = fp16(2/127), every q = 127, s = fp16(d32 * 4064) = 64.0
    x = np.full((1, 32), 2.0, dtype=np.float16)
    blk = o.quantize_q8_1(x)[0, 0]
    assert np.all(blk[4:].view(np.int8) == 127)
    d = np.frombuffer(blk[0:2].tobytes(), np.float16)[0]
    s = np.frombuffer(blk[2:4].tobytes(), np.float16)[0]
    assert d == np.float16(2.0 / 127.0)
    assert s == np.float16(64.0)
    # zero block: every byte 0
    blk = o.quantize_q8_1(np.zeros((1, 32), np.float16))[0, 0]
    assert not blk.any()
    # one nonzero element -0.5 at index 9: q[9] = -127, the rest 0, s = -d*127 = -0.5
    x = np.zeros((1, 32), np.float16)
    x[0, 9] = -0.5
    blk = o.quantize_q8_1(x)[0, 0]
    q = blk[4:].view(np.int8)
    assert q[9] == -127 and np.count_nonzero(q) == 1
    assert np.frombuffer(blk[2:4].tobytes(), np.float16)[0] == np.float16(-0.5)
    # amax = 127 -> d32 = 1 exactly, so q = x for integer x
    x = np.zeros((1, 32), np.float16)
    x[0, :8] = [127, -127, 1, -1, 2, 50, -99, 3]
    blk = o.quantize_q8_1(x)[0, 0]
    assert blk[0] == 0x00 and blk[1] == 0x3C                       # d = 1.0
    assert blk[4:].view(np.int8)[:8].tolist() == [127, -127, 1, -1, 2, 50, -99, 3]
    assert np.frombuffer(blk[2:4].tobytes(), np.float16)[0] == np.float16(-44.0)
    # amax = 63.5 -> d32 = 0.5 exactly, so q = 2x
    x = np.zeros((1, 32), np.float16)
    x[0, 30:32] = [63.5, 0.5]
    x[0, 0:3] = [-63.5, -0.5, 10.0]
    blk = o.quantize_q8_1(x)[0, 0]
    assert blk[0] == 0x00 and blk[1] == 0x38                       # d = 0.5
    q = blk[4:].view(np.int8)
    assert q[[0, 1, 2, 30, 31]].tolist() == [-127, -1, 20, 127, 1]
    assert np.count_nonzero(q) == 5


def pin_q8_1_numpy(o):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 256)).astype(np.float16)
    x[2, 32:64] = 0
    x[3, :] *= np.float16(20)
    x[4, 64:96] = np.float16(6e-5)   # tiny block: d lands in fp16 subnormals
    blk = o.quantize_q8_1(x).reshape(-1, 36)
    d, s, q = _q8_numpy_fp32(x)
    assert np.array_equal(blk[:, 0:2].copy().view(np.float16)[:, 0].view(np.uint16), d.view(np.uint16))
    assert np.array_equal(blk[:, 2:4].copy().view(np.float16)[:, 0].view(np.uint16), s.view(np.uint16))
    assert np.array_equal(blk[:, 4:].view(np.int8).astype(np.int64), q)


def pin_q8_1_error_bound(o):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((16, 512)).astype(np.float16)
    blk = o.quantize_q8_1(x)
    deq = o.dequantize_q8_1(blk)
    assert np.array_equal(deq, numpy_decode_q8_1(blk))
    xb = x.astype(np.float64).reshape(-1, 32)
    amax = np.abs(xb).max(axis=1)
    d32 = amax / 127.0
    err = np.abs(deq.reshape(-1, 32) - xb)
    # half a level plus the fp16 rounding of d applied to |q| <= 127
    bound = 0.5 * d32 * (1 + 1e-6) + 127 * d32 * 2.0 ** -11
    assert np.all(err <= bound[:, None])
    q = blk.reshape(-1, 36)[:, 4:].view(np.int8)
    assert np.all(np.abs(q).max(axis=1) == 127)


# ------------------------------------------------------------------ route
def pin_route(o):
    rng = np.random.default_rng(7)
    for S, E in [(0, 4), (1, 1), (37, 5), (500, 16), (64, 128)]:
        ids = rng.integers(0, E, S).astype(np.int32)
        counts, offsets, perm, bad = o.route(ids, E)
        assert bad == 0
        assert np.array_equal(counts, np.bincount(ids, minlength=E))
        assert offsets[0] == 0 and offsets[-1] == S
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(perm, np.argsort(ids, kind="stable"))
    ids = np.array([3, -1, 0, 7, 3, 9, 0], dtype=np.int32)
    counts, offsets, perm, bad = o.route(ids, 4)
    assert bad == 3
    assert counts.tolist() == [2, 0, 0, 2]
    assert offsets.tolist() == [0, 2, 2, 2, 4]
    assert perm.tolist() == [2, 6, 0, 4, -1, -1, -1]


# -------------------------------------------------------------------- dot
def pin_block_dot_hand(o):
    zero_d = 0x3C00   # fp16 1.0 (the scales do not enter the integer dot)
    assert o.block_dot(q4_block(zero_d, [9] * 32), q8_block(zero_d, 0, [1] * 32)) == 32
    assert o.block_dot(q4_block(zero_d, [0] * 32), q8_block(zero_d, 0, [127] * 32)) == -32512
    assert o.block_dot(q4_block(zero_d, [15] * 32), q8_block(zero_d, 0, [-127] * 32)) == -28448
    # single nonzero weight in the high-nibble half: only a[20] matters
    qw = [8] * 32
    qw[20] = 15
    qa = list(range(-16, 16))
    assert o.block_dot(q4_block(zero_d, qw), q8_block(zero_d, 0, qa)) == 7 * qa[20]
    # single nonzero weight in the low-nibble half
    qw = [8] * 32
    qw[3] = 1
    assert o.block_dot(q4_block(zero_d, qw), q8_block(zero_d, 0, qa)) == -7 * qa[3]


def pin_moe_closed_form_vs_bruteforce(o):
    for seed, T in [(10, 7), (11, 1), (12, 13)]:
        w, x, ids = tiny_case(seed=seed, T=T)
        act = o.quantize_q8_1(x)
        y = o.moe(w, act, ids).astype(np.float64)
        bf = o.moe_dequant_bruteforce(w, act, ids)
        scale = np.abs(bf).max()
        assert np.all(np.abs(y - bf) <= 1e-6 * np.abs(bf) + 1e-12 * scale)
        ys = o.moe_sample(w, act, ids, np.arange(T * ids.shape[1]), np.zeros(T * ids.shape[1], np.int64))
        assert np.all(np.abs(ys - bf[:, :, 0].reshape(-1)) <= 1e-12 * scale)


def pin_moe_numpy_einsum(o):
    """Decode both operands independently in numpy and contract with einsum."""
    for seed, T, k in [(20, 9, 2), (21, 4, 3)]:
        w, x, ids = tiny_case(seed=seed, T=T, k=k)
        act = o.quantize_q8_1(x)
        W = numpy_decode_q4_0(w)                   # [E, N, K]
        A = numpy_decode_q8_1(act)                 # [T, K]
        want = np.einsum("tjnk,tk->tjn", W[ids], A)
        got = o.moe(w, act, ids).astype(np.float64)
        tol = 1e-6 * np.abs(want) + 1e-9 * np.abs(want).max()
        assert np.all(np.abs(got - want) <= tol)


def pin_moe_block_dots(o):
    w, x, ids = tiny_case(seed=30, T=3, K=64, N=5)
    act = o.quantize_q8_1(x)
    dots = o.moe_block_dots(w, act, ids)
    qs = w[..., 2:].astype(np.int64)
    Wq = np.concatenate([qs & 15, qs >> 4], axis=-1) - 8          # [E, N, nb, 32] levels
    Aq = np.ascontiguousarray(act[..., 4:]).view(np.int8).astype(np.int64)   # [T, nb, 32]
    flat = ids.reshape(-1)
    for s in range(flat.size):
        e, t = flat[s], s // ids.shape[1]
        want = (Wq[e] * Aq[t][None]).sum(axis=-1)                # [N, nb]
        assert np.array_equal(dots[s], want)


def pin_moe_split_invariance(o):
    w, x, ids = tiny_case(seed=40, T=11)
    act = o.quantize_q8_1(x)
    y = o.moe(w, act, ids)
    y1 = o.moe(w, act[:5], ids[:5])
    y2 = o.moe(w, act[5:], ids[5:])
    assert np.array_equal(y, np.concatenate([y1, y2]))


def pin_moe_bad_ids(o):
    w, x, ids = tiny_case(seed=50, T=4)
    ids = ids.copy()
    ids[1, 0] = -3
    ids[2, 1] = w.shape[0]
    act = o.quantize_q8_1(x)
    y = o.moe(w, act, ids)
    assert not y[1, 0].any() and not y[2, 1].any()
    assert y[0].any() and y[3].any()


def pin_moe_slots_numpy_einsum(o):
    """Per-slot activations (one Q8_1 row per routed slot): independent numpy
    decode of both operands and einsum, with every slot's row different."""
    for seed, T, k in [(60, 6, 2), (61, 3, 3)]:
        w, x, ids = tiny_case(seed=seed, T=T * k, k=1)        # T*k distinct activation rows
        ids = tiny_case(seed=seed + 100, T=T, k=k)[2]          # routing of T tokens x k slots
        act_slots = o.quantize_q8_1(x)                          # [T*k, nb, 36]
        W = numpy_decode_q4_0(w)                                # [E, N, K]
        A = numpy_decode_q8_1(act_slots)                        # [T*k, K]
        want = np.einsum("snk,sk->sn", W[ids.reshape(-1)], A).reshape(T, k, -1)
        got = o.moe_slots(w, act_slots, ids).astype(np.float64)
        tol = 1e-6 * np.abs(want) + 1e-9 * np.abs(want).max()
        assert np.all(np.abs(got - want) <= tol)


def pin_moe_slots_replicated_rows(o):
    """Slot s given its token's row (row s // k) reproduces the per-token
    matmul bit for bit."""
    w, x, ids = tiny_case(seed=62, T=7, k=3)
    act = o.quantize_q8_1(x)
    act_slots = np.repeat(act, ids.shape[1], axis=0)
    assert np.array_equal(o.moe_slots(w, act_slots, ids), o.moe(w, act, ids))


def pin_moe_ep_shards_sum_to_full(o):
    """A partition of the experts into shards: the shards' outputs (zero rows for
    slots routed elsewhere) add up to the full matmul bit for bit, and a single
    shard holding every expert is the full matmul."""
    w, x, ids = tiny_case(seed=64, E=6, T=9, k=2)
    act = o.quantize_q8_1(x)
    full = o.moe(w, act, ids)
    E = w.shape[0]
    for bounds in [(0, 2, 6), (0, 1, 4, 6), (0, 6)]:
        total = np.zeros_like(full)
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            part = o.moe_ep(w[lo:hi], act, ids, E, lo)
            local = (ids >= lo) & (ids < hi)
            assert not part[~local].any()                     # non-local slots are zero rows
            total += part
        assert np.array_equal(total, full)


# ------------------------------------------------------- gated activation
def _act_inputs(seed, rows=5, n_inter=96):
    rng = np.random.default_rng(seed)
    h = (rng.standard_normal((rows, 2 * n_inter)) * 3).astype(np.float32)
    h[0, :8] = [0.0, -0.0, 1e-30, -1e-30, 40.0, -40.0, 1000.0, -1000.0]
    h[1, :n_inter] = np.linspace(-12, 12, n_inter, dtype=np.float32)
    return h


def _ulp32(x):
    return np.spacing(np.abs(x).astype(np.float32)).astype(np.float64)


def pin_act_library(o):
    """act_mul against library activations in fp64 (torch.nn.functional.silu and
    gelu(approximate="tanh")), up half applied after: within one fp32 ulp, plus
    1e-15 |g u| for the cancellation in 1 + tanh(.) deep in the negative tail,
    where two fp64 tanh routines may differ by an ulp of 1."""
    import torch
    import torch.nn.functional as F
    h = _act_inputs(11)
    n = h.shape[1] // 2
    g = torch.from_numpy(h[:, :n].astype(np.float64))
    u = h[:, n:].astype(np.float64)
    for kind, fn in ((o.ACT_SILU, F.silu), (o.ACT_GELU_TANH, lambda t: F.gelu(t, approximate="tanh"))):
        ref = fn(g).numpy() * u
        a = o.act_mul(h, kind).astype(np.float64)
        tol = _ulp32(ref) + 1e-15 * np.abs(g.numpy() * u) + 1e-45
        assert np.all(np.abs(a - ref) <= tol), kind
        if kind == o.ACT_SILU:                  # no cancellation in either evaluation
            assert np.mean(a == ref.astype(np.float32)) > 0.98


def pin_act_tail_accuracy(o):
    """Both activations against 50-digit evaluations of their definitions
    (mpmath), tanh form as written for GELU: every fp32 result within one ulp,
    including the negative tails where the exact values are tiny (GELU below
    g = -6, where 1 + tanh(y) cancels in fp64; SiLU down to g = -80)."""
    import mpmath
    mpmath.mp.dps = 50
    g = np.concatenate([np.linspace(-12, 12, 481), np.linspace(-80, -12, 69)]).astype(np.float32)
    h = np.concatenate([g, np.full_like(g, 1.5)])[None, :]
    c = mpmath.sqrt(mpmath.mpf(2) / mpmath.pi)
    for kind in (o.ACT_SILU, o.ACT_GELU_TANH):
        a = o.act_mul(h, kind)[0]
        for gi, ai in zip(g.tolist(), a.tolist()):
            x = mpmath.mpf(gi)
            if kind == o.ACT_SILU:
                ex = x / (1 + mpmath.exp(-x))
            else:
                ex = x / 2 * (1 + mpmath.tanh(c * (x + mpmath.mpf("0.044715") * x ** 3)))
            ex = float(ex * mpmath.mpf(1.5))
            assert abs(ai - ex) <= float(np.spacing(np.float32(abs(ex)))) + 1e-45, (kind, gi, ai, ex)


def pin_act_gelu_vs_erf(o):
    """The tanh form stays within 5e-4 of the exact GELU x * Phi(x) (its known
    approximation error is 4.7e-4); a dropped cubic term is off by 3e-2."""
    from scipy.special import erf
    g = np.linspace(-10, 10, 4001).astype(np.float32)
    h = np.concatenate([g, np.ones_like(g)])[None, :]
    a = o.act_mul(h, o.ACT_GELU_TANH)[0].astype(np.float64)
    gd = g.astype(np.float64)
    exact = 0.5 * gd * (1.0 + erf(gd / np.sqrt(2.0)))
    assert np.abs(a - exact).max() < 5e-4


def pin_act_odd_identity(o):
    """Both activations satisfy f(x) - f(-x) = x (1 - sigmoid(x) = sigmoid(-x),
    tanh odd); with up = 1 each output carries one fp32 rounding."""
    g = np.concatenate([np.linspace(-30, 30, 601), [1e-3, 0.25, 7.5]]).astype(np.float32)
    n = g.size
    h = np.zeros((2, 2 * n), np.float32)
    h[0, :n], h[1, :n] = g, -g
    h[:, n:] = 1.0
    for kind in (o.ACT_SILU, o.ACT_GELU_TANH):
        a = o.act_mul(h, kind).astype(np.float64)
        diff = a[0] - a[1]
        assert np.all(np.abs(diff - g) <= _ulp32(a[0]) + _ulp32(a[1]) + 1e-45), kind


def pin_act_hand(o):
    """Gate/up order and hand values: silu(0) * u = 0, silu(g) -> g for large g,
    silu(g) -> 0 for very negative g, silu(ln 3) = (3/4) ln 3, and the up half
    multiplies (a gate of 0 zeroes the output whatever the up value)."""
    h = np.array([[0.0, 50.0, -200.0, np.log(3.0), 5.0, 0.0, 2.0, 1.0,
                   7.0, 2.0, 3.0, 4.0, 0.0, 9.0, 1.0, -3.0]], dtype=np.float32)
    a = o.act_mul(h, o.ACT_SILU)[0]
    assert a[0] == 0.0                                   # gate 0, up 7
    assert a[1] == np.float32(100.0)                     # 50 * sigmoid(50) rounds to 50; times up 2
    assert a[2] == 0.0 and np.signbit(a[2])              # -200 / (1 + e^200) = -0 (times up 3)
    ln3 = np.float64(np.float32(np.log(3.0)))
    assert abs(float(a[3]) - 4.0 * ln3 / (1.0 + 1.0 / 3.0 * np.exp(np.log(3.0) - ln3))) < 1e-6
    assert a[4] == 0.0                                   # up 0
    assert a[5] == 0.0                                   # gate 0, up 9
    assert abs(float(a[6]) - 2.0 / (1.0 + np.exp(-2.0))) < 1e-6
    assert abs(float(a[7]) + 3.0 / (1.0 + np.exp(-1.0))) < 1e-6


def pin_act_quantize_numpy(o):
    """act_mul_quantize_q8_1 is the fp32 Q8_1 replay applied to act_mul's output,
    one row of I/32 blocks per row of h."""
    h = _act_inputs(12, rows=6, n_inter=128)
    h[2, :128] = 0.0                                      # a row of zero blocks
    for kind in (o.ACT_SILU, o.ACT_GELU_TANH):
        blk = o.act_mul_quantize_q8_1(h, kind)
        assert blk.shape == (6, 4, 36)
        d, s, q = _q8_numpy_fp32(o.act_mul(h, kind))
        b = blk.reshape(-1, 36)
        assert np.array_equal(b[:, 0:2].copy().view(np.uint16)[:, 0], d.view(np.uint16))
        assert np.array_equal(b[:, 2:4].copy().view(np.uint16)[:, 0], s.view(np.uint16))
        assert np.array_equal(b[:, 4:].view(np.int8).astype(np.int64), q)
        assert not blk[2].any()


# ------------------------------------------------- other GGUF weight types
def numpy_decode_gguf(wtype, w):
    """Independent vectorised decode of the 32-weight GGUF types [..., nb, bytes]
    -> (levels int64 [..., nb, 32], d fp64 [..., nb], offset fp64 [..., nb])."""
    w = np.ascontiguousarray(w)
    d = w[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    zero = np.zeros_like(d)
    if wtype == "q8_0":
        return w[..., 2:34].copy().view(np.int8).astype(np.int64), d, zero
    has_m = wtype in ("q4_1", "q5_1")
    m = w[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64) if has_m else zero
    if wtype == "q4_1":
        qs = w[..., 4:20].astype(np.int64)
        return np.concatenate([qs & 15, qs >> 4], axis=-1), d, m
    h0 = 4 if has_m else 2
    qh = w[..., h0:h0 + 4].copy().view("<u4")[..., 0].astype(np.int64)
    qs = w[..., h0 + 4:h0 + 20].astype(np.int64)
    nib = np.concatenate([qs & 15, qs >> 4], axis=-1)
    bits = (qh[..., None] >> np.arange(32)) & 1
    lev = nib | (bits << 4)
    return (lev - 16 if wtype == "q5_0" else lev), d, m


def _gguf_random(wtype, E=3, N=5, K=96, seed=0):
    from bit_quantized_moe_quantize_gb300 import synth
    return synth.make_weights_gguf(synth.custom_workload(E, 2, K, N, seed), wtype)


def pin_gguf_hand(o):
    """Hand-assembled blocks of each type, decoded and dotted by hand."""
    a = q8_block(0x3C00, 0x0000, [1] * 32)                  # d_a = 1, q_a = 1, s = 0 (stored)
    # Q8_0: d = 1, codes -128, 127, 0, ..., 5
    b = np.zeros(34, np.uint8)
    b[0], b[1] = 0x00, 0x3C
    q = np.zeros(32, np.int8)
    q[:3] = [-128, 127, 0]
    q[31] = 5
    b[2:] = q.view(np.uint8)
    assert o.dequantize_gguf("q8_0", b[None]).tolist() == q.astype(float).tolist()
    assert o.gguf_block_dot("q8_0", b, a) == 4
    # Q4_1: d = 0.5, m = -2; low nibble j, high nibble 15 - j -> w_j = j/2 - 2, w_{j+16} = (15-j)/2 - 2
    b = np.zeros(20, np.uint8)
    b[0:2] = [0x00, 0x38]
    b[2:4] = [0x00, 0xC0]
    b[4:] = [j | ((15 - j) << 4) for j in range(16)]
    want = [j / 2 - 2 for j in range(16)] + [(15 - j) / 2 - 2 for j in range(16)]
    assert o.dequantize_gguf("q4_1", b[None]).tolist() == want
    assert o.gguf_block_dot("q4_1", b, a) == 2 * sum(range(16))        # levels, not values
    # Q5_0: d = 1, all nibbles 0, qh bits 1 and 16 set -> levels 0 at i = 1, 16, else -16
    b = np.zeros(22, np.uint8)
    b[0:2] = [0x00, 0x3C]
    b[2:6] = [0x02, 0x00, 0x01, 0x00]
    lev = [-16] * 32
    lev[1] = lev[16] = 0
    assert o.dequantize_gguf("q5_0", b[None]).tolist() == [float(v) for v in lev]
    assert o.gguf_block_dot("q5_0", b, a) == -16 * 30
    # Q5_1: d = 0.25, m = 1; nibbles 15 everywhere, qh = 0x80000000 -> level 31 at i = 31, else 15
    b = np.zeros(24, np.uint8)
    b[0:2] = [0x00, 0x34]
    b[2:4] = [0x00, 0x3C]
    b[4:8] = [0x00, 0x00, 0x00, 0x80]
    b[8:] = 0xFF
    want = [15 * 0.25 + 1] * 31 + [31 * 0.25 + 1]
    assert o.dequantize_gguf("q5_1", b[None]).tolist() == want
    assert o.gguf_block_dot("q5_1", b, a) == 15 * 31 + 31


def pin_gguf_numpy_decode(o):
    for wtype in ("q4_1", "q5_0", "q5_1", "q8_0"):
        w = _gguf_random(wtype, seed=3)
        lev, d, m = numpy_decode_gguf(wtype, w)
        want = lev * d[..., None] + m[..., None]
        got = o.dequantize_gguf(wtype, w)
        assert np.array_equal(got, want.reshape(got.shape)), wtype


def pin_gguf_moe_numpy(o):
    """The matmul of each type against a numpy restatement: per block
    d_w d_a sum(q_w q_a) + m d_a sum(q_a) with the exact code sum, in fp64;
    and against the plain dot of the dequantized weights and activations,
    which that is term for term (fp64 rounding only)."""
    from bit_quantized_moe_quantize_gb300 import synth
    rng = np.random.default_rng(4)
    E, k, K, N, T = 4, 2, 128, 6, 5
    x = rng.standard_normal((T, K)).astype(np.float16)
    act = o.quantize_q8_1(x)
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    qa = act[..., 4:].view(np.int8).astype(np.int64)
    da = act[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    suma = qa.sum(axis=-1).astype(np.float64)                    # [T, nb]
    xa = numpy_decode_q8_1(act)
    for wtype in ("q4_1", "q5_0", "q5_1", "q8_0"):
        w = _gguf_random(wtype, E=E, N=N, K=K, seed=5)
        lev, d, m = numpy_decode_gguf(wtype, w)                  # [E, N, nb, 32], [E, N, nb]
        got = o.moe_gguf(wtype, w, act, ids).astype(np.float64)
        wv = (lev * d[..., None] + m[..., None]).reshape(E, N, K)
        for t in range(T):
            for j in range(k):
                e = ids[t, j]
                dots = np.einsum("rbi,bi->rb", lev[e], qa[t])
                want = (d[e] * da[t] * dots + m[e] * da[t] * suma[t]).sum(axis=1)
                assert np.allclose(got[t, j], want, rtol=1e-6, atol=1e-9), wtype
                plain = wv[e] @ xa[t]
                assert np.allclose(want, plain, rtol=1e-12, atol=1e-12), wtype


def pin_gguf_q4_0_is_the_q4_0_matmul(o):
    w, x, ids = tiny_case(seed=9)
    act = o.quantize_q8_1(x)
    assert np.array_equal(o.moe_gguf("q4_0", w, act, ids), o.moe(w, act, ids))


# -------------------------------------------------------------- K-quants
def numpy_decode_kquant(wtype, w):
    """Independent vectorised decode of Q4_K / Q5_K super-blocks [..., nsb, bytes]
    -> fp64 [..., nsb * 256]."""
    w = np.ascontiguousarray(w)
    d = w[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = w[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    sc12 = w[..., 4:16].astype(np.int64)
    lo_sc, lo_m = sc12[..., 0:4] & 63, sc12[..., 4:8] & 63
    hi_sc = (sc12[..., 8:12] & 15) | ((sc12[..., 0:4] >> 6) << 4)
    hi_m = (sc12[..., 8:12] >> 4) | ((sc12[..., 4:8] >> 6) << 4)
    sc = np.concatenate([lo_sc, hi_sc], axis=-1)                 # [..., 8]
    m = np.concatenate([lo_m, hi_m], axis=-1)
    q0 = 48 if wtype == "q5_k" else 16
    qs = w[..., q0:q0 + 128].astype(np.int64).reshape(*w.shape[:-1], 4, 32)
    lev = np.stack([qs & 15, qs >> 4], axis=-2).reshape(*w.shape[:-1], 8, 32)   # sub-block j = 2 c + half
    if wtype == "q5_k":
        qh = w[..., 16:48].astype(np.int64)                       # [..., 32]
        bits = (qh[..., None, :] >> np.arange(8)[:, None]) & 1    # [..., 8, 32]
        lev = lev | (bits << 4)
    vals = d[..., None, None] * sc[..., None] * lev - (dmin[..., None] * m)[..., None]
    return vals.reshape(*w.shape[:-2], w.shape[-2] * 256)


def _kq_scales_bytes(sc, m):
    """Pack eight 6-bit (scale, min) pairs by hand into the 12 scale bytes."""
    b = [0] * 12
    for j in range(4):
        b[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        b[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        b[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return b


def pin_kquant_hand(o):
    """A hand-packed Q4_K and Q5_K super-block: every sub-block's scale and min
    (the low four through byte j, the high four split over nibbles and top bits),
    nibble halves and 5th bits."""
    sc = [1, 2, 3, 4, 33, 34, 35, 50]
    m = [5, 6, 7, 8, 17, 18, 40, 63]
    for wtype, size in (("q4_k", 144), ("q5_k", 176)):
        b = np.zeros(size, np.uint8)
        b[0:2] = [0x00, 0x3C]                 # d = 1
        b[2:4] = [0x00, 0x38]                 # dmin = 0.5
        b[4:16] = _kq_scales_bytes(sc, m)
        q0 = 48 if wtype == "q5_k" else 16
        lev_lo = np.arange(32) % 16
        lev_hi = (np.arange(32) * 7) % 16
        for c in range(4):
            b[q0 + 32 * c:q0 + 32 * c + 32] = lev_lo | (lev_hi << 4)
        if wtype == "q5_k":
            b[16:48] = 0b10100101             # 5th bit set in sub-blocks 0, 2, 5, 7
        got = o.dequantize_gguf(wtype, b[None]).reshape(8, 32)
        for j in range(8):
            lev = (lev_lo if j % 2 == 0 else lev_hi).copy()
            if wtype == "q5_k" and j in (0, 2, 5, 7):
                lev += 16
            assert np.array_equal(got[j], 1.0 * sc[j] * lev - 0.5 * m[j]), (wtype, j)


def pin_kquant_numpy_decode(o):
    for wtype in ("q4_k", "q5_k"):
        w = _gguf_random(wtype, K=512, seed=6)
        assert np.array_equal(o.dequantize_gguf(wtype, w), numpy_decode_kquant(wtype, w)), wtype


def pin_kquant_moe_numpy(o):
    """Each K-quant matmul against the plain dequantized dot in fp64 (its min
    term uses the exact d_a * sum(q_a), so the two agree to rounding)."""
    rng = np.random.default_rng(8)
    E, k, K, N, T = 3, 2, 512, 5, 4
    act = o.quantize_q8_1(rng.standard_normal((T, K)).astype(np.float16))
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    xa = numpy_decode_q8_1(act)
    for wtype in ("q4_k", "q5_k"):
        w = _gguf_random(wtype, E=E, N=N, K=K, seed=9)
        wv = numpy_decode_kquant(wtype, w).reshape(E, N, K)
        got = o.moe_gguf(wtype, w, act, ids).astype(np.float64)
        for t in range(T):
            for j in range(k):
                want = wv[ids[t, j]] @ xa[t]
                scale = np.abs(wv[ids[t, j]]) @ np.abs(xa[t])
                assert np.all(np.abs(got[t, j] - want) <= 1e-6 * scale + 1e-12), wtype


def pin_kquant_unit_scales_are_q4_1(o):
    """A Q4_K super-block whose sub-block scales and mins are all 1 holds eight
    Q4_1 blocks with d' = d and m' = -dmin (nibbles re-laid in Q4_1 order)."""
    rng = np.random.default_rng(10)
    b = np.zeros(144, np.uint8)
    b[0:2] = np.array([0.0625], np.float16).view(np.uint8)
    b[2:4] = np.array([0.375], np.float16).view(np.uint8)
    b[4:16] = _kq_scales_bytes([1] * 8, [1] * 8)
    b[16:] = rng.integers(0, 256, 128, dtype=np.uint8)
    q41 = np.zeros((8, 20), np.uint8)
    for j in range(8):
        lev = (b[16 + 32 * (j // 2):16 + 32 * (j // 2) + 32] >> (4 * (j % 2))) & 15
        q41[j, 0:2] = b[0:2]
        q41[j, 2:4] = np.array([-0.375], np.float16).view(np.uint8)
        q41[j, 4:] = lev[:16] | (lev[16:] << 4)
    assert np.array_equal(o.dequantize_gguf("q4_k", b[None]), o.dequantize_gguf("q4_1", q41))


def numpy_decode_q6k(w):
    """Independent vectorised decode of Q6_K super-blocks [..., nsb, 210] -> fp64 [..., nsb * 256]."""
    w = np.ascontiguousarray(w)
    lead = w.shape[:-1]
    d = w[..., 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
    sc = w[..., 192:208].copy().view(np.int8).astype(np.float64)           # [..., 16]
    ql = w[..., 0:128].astype(np.int64).reshape(*lead, 2, 2, 32)            # half, k % 2, l
    qh = w[..., 128:192].astype(np.int64).reshape(*lead, 2, 32)             # half, l
    out = np.empty((*lead, 2, 4, 32), dtype=np.float64)
    for k in range(4):
        lo4 = (ql[..., k % 2, :] >> (4 * (k // 2))) & 15
        hi2 = (qh >> (2 * k)) & 3
        q = (lo4 | (hi2 << 4)) - 32                                          # [..., 2, 32]
        s_lo = sc[..., [2 * k, 8 + 2 * k]]                                   # [..., 2]
        s_hi = sc[..., [2 * k + 1, 8 + 2 * k + 1]]
        scale = np.concatenate([np.repeat(s_lo[..., None], 16, -1), np.repeat(s_hi[..., None], 16, -1)], -1)
        out[..., k, :] = d[..., None, None] * scale * q
    return out.reshape(*w.shape[:-2], w.shape[-2] * 256)


def pin_q6k_hand(o):
    """A hand-built Q6_K super-block: level = low nibble | 2 high bits << 4, - 32,
    one int8 scale per 16 weights (negative ones included), d stored last."""
    b = np.zeros(210, np.uint8)
    b[208:210] = [0x00, 0x3C]                                    # d = 1
    scales = np.array([1, -2, 3, 4, 5, 6, -7, 8, 9, 10, 11, 12, 13, -14, 15, 127], np.int8)
    b[192:208] = scales.view(np.uint8)
    l = np.arange(32)
    b[0:32] = (l % 16) | (((l + 3) % 16) << 4)                    # half 0, k = 0 low / k = 2 high
    b[32:64] = (l % 7) | ((l % 5) << 4)                           # half 0, k = 1 low / k = 3 high
    b[128:160] = 0b11100100                                       # 2-bit parts 0, 1, 2, 3 for k = 0..3
    got = o.dequantize_gguf("q6_k", b[None]).reshape(8, 32)
    lo4 = {0: l % 16, 1: l % 7, 2: (l + 3) % 16, 3: l % 5}
    for k in range(4):
        q = (lo4[k] | (k << 4)) - 32
        want = np.where(l < 16, scales[2 * k], scales[2 * k + 1]).astype(np.float64) * q
        assert np.array_equal(got[k], want), k
    # half 1 is all zero bytes: level -32 everywhere, scales 8..15
    for k in range(4):
        want = np.where(l < 16, scales[8 + 2 * k], scales[8 + 2 * k + 1]).astype(np.float64) * -32
        assert np.array_equal(got[4 + k], want), 4 + k


def pin_q6k_numpy(o):
    """Decode against the numpy decoder; the matmul against the plain dequantized dot."""
    w = _gguf_random("q6_k", K=512, seed=11)
    assert np.array_equal(o.dequantize_gguf("q6_k", w), numpy_decode_q6k(w))
    rng = np.random.default_rng(12)
    E, k, K, N, T = 3, 2, 512, 5, 4
    act = o.quantize_q8_1(rng.standard_normal((T, K)).astype(np.float16))
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    xa = numpy_decode_q8_1(act)
    w = _gguf_random("q6_k", E=E, N=N, K=K, seed=13)
    wv = numpy_decode_q6k(w).reshape(E, N, K)
    got = o.moe_gguf("q6_k", w, act, ids).astype(np.float64)
    for t in range(T):
        for j in range(k):
            want = wv[ids[t, j]] @ xa[t]
            scale = np.abs(wv[ids[t, j]]) @ np.abs(xa[t])
            assert np.all(np.abs(got[t, j] - want) <= 1e-6 * scale + 1e-12)


# ------------------------------------------------------------- SoA repack
def pin_repack_q4_0_soa(o):
    """The repack is the block bytes sliced: nibble bytes 2..17 in block order,
    then the fp16 at bytes 0..1 of each block; a hand block checks the order."""
    w, _, _ = tiny_case(seed=12)
    qs, d = o.repack_q4_0_soa(w)
    flat = w.reshape(-1, 18)
    assert np.array_equal(qs, flat[:, 2:])
    assert np.array_equal(d.view(np.uint16), flat[:, 0:2].copy().view(np.uint16)[:, 0])
    blk = q4_block(0x3C01, list(range(16)) + list(range(15, -1, -1)))
    qs, d = o.repack_q4_0_soa(np.stack([blk, blk[::-1].copy()]))
    assert d.view(np.uint16).tolist() == [0x3C01, int(blk[17]) | (int(blk[16]) << 8)]
    assert qs[0].tolist() == [j | ((15 - j) << 4) for j in range(16)]


def numpy_decode_q2k_q3k(wtype, w):
    """Independent vectorised decode of Q2_K / Q3_K super-blocks -> fp64 [..., nsb * 256]."""
    w = np.ascontiguousarray(w)
    lead = w.shape[:-1]
    q0 = 16 if wtype == "q2_k" else 32
    codes = w[..., q0:q0 + 64].astype(np.int64).reshape(*lead, 2, 32)           # half, l
    shifts = 2 * np.arange(4)
    lev = (codes[..., None, :] >> shifts[:, None]) & 3                          # half, k, l
    if wtype == "q2_k":
        sc = w[..., 0:16].astype(np.int64)
        scale, mn = (sc & 15).astype(np.float64), (sc >> 4).astype(np.float64)
        d = w[..., 80:82].copy().view(np.float16)[..., 0].astype(np.float64)
        dmin = w[..., 82:84].copy().view(np.float16)[..., 0].astype(np.float64)
    else:
        hm = w[..., 0:32].astype(np.int64)                                       # l
        jj = np.arange(8).reshape(2, 4)                                          # sub-block index per (half, k)
        hbit = (hm[..., None, None, :] >> jj[:, :, None]) & 1
        lev = (lev | (hbit << 2)) - 4
        b = w[..., 96:108].astype(np.int64)
        g = np.arange(16)
        low4 = np.where(g < 8, b[..., g % 8] & 15, b[..., g % 8] >> 4)
        top2 = (b[..., 8 + g % 4] >> (2 * (g // 4))) & 3
        scale = ((low4 | (top2 << 4)) - 32).astype(np.float64)
        mn = np.zeros_like(scale)
        d = w[..., 108:110].copy().view(np.float16)[..., 0].astype(np.float64)
        dmin = np.zeros_like(d)
    grp = np.arange(16).reshape(2, 4, 2)                                        # scale group per (half, k, l >= 16)
    sel = np.repeat(grp, 16, axis=-1)                                           # half, k, 32
    out = np.empty((*lead, 2, 4, 32))
    for h in range(2):
        for k in range(4):
            gl, gh = sel[h, k, 0], sel[h, k, 16]
            sc_v = np.concatenate([np.repeat(scale[..., gl, None], 16, -1), np.repeat(scale[..., gh, None], 16, -1)], -1)
            mn_v = np.concatenate([np.repeat(mn[..., gl, None], 16, -1), np.repeat(mn[..., gh, None], 16, -1)], -1)
            out[..., h, k, :] = d[..., None] * sc_v * lev[..., h, k, :] - dmin[..., None] * mn_v
    return out.reshape(*w.shape[:-2], w.shape[-2] * 256)


def pin_q2k_q3k_hand(o):
    """Hand-built Q2_K and Q3_K super-blocks: code shifts, scale/min nibbles,
    the third bit from hmask, the 6-bit scale packing (low nibbles of bytes
    0..7 for groups 0..7, high nibbles for 8..15, top bits from bytes 8..11)."""
    l = np.arange(32)
    codes = ((l % 4) | (((l + 1) % 4) << 2) | (((l + 2) % 4) << 4) | (((l + 3) % 4) << 6)).astype(np.uint8)
    # Q2_K: d = 1, dmin = 0.5; group g has scale g % 16 and min (g * 3) % 16
    b = np.zeros(84, np.uint8)
    b[0:16] = [(g % 16) | (((g * 3) % 16) << 4) for g in range(16)]
    b[16:48] = codes
    b[48:80] = codes[::-1]
    b[80:82] = [0x00, 0x3C]
    b[82:84] = [0x00, 0x38]
    got = o.dequantize_gguf("q2_k", b[None]).reshape(8, 32)
    for j in range(8):
        h, k = divmod(j, 4)
        src = codes if h == 0 else codes[::-1]
        q = (src.astype(np.int64) >> (2 * k)) & 3
        g = np.where(l < 16, 2 * j, 2 * j + 1)
        assert np.array_equal(got[j], (g % 16) * q - 0.5 * ((g * 3) % 16)), ("q2_k", j)
    # Q3_K: d = 1; scales (6-bit) 0..15 -> values 5 g - 32 + ... chosen as v_g = (7 g + 3) % 64
    v = [(7 * g + 3) % 64 for g in range(16)]
    sc = [0] * 12
    for g in range(16):
        sc[g % 8] |= (v[g] & 15) << (0 if g < 8 else 4)
        sc[8 + g % 4] |= (v[g] >> 4) << (2 * (g // 4))
    b = np.zeros(110, np.uint8)
    b[0:32] = (l * 37) % 256                          # hmask
    b[32:64] = codes
    b[64:96] = codes[::-1]
    b[96:108] = sc
    b[108:110] = [0x00, 0x3C]
    got = o.dequantize_gguf("q3_k", b[None]).reshape(8, 32)
    hm = (l * 37) % 256
    for j in range(8):
        h, k = divmod(j, 4)
        src = codes if h == 0 else codes[::-1]
        q = ((src.astype(np.int64) >> (2 * k)) & 3) | (((hm >> j) & 1) << 2)
        g = np.where(l < 16, 2 * j, 2 * j + 1)
        assert np.array_equal(got[j], (np.array(v)[g] - 32) * (q - 4)), ("q3_k", j)


def pin_q2k_q3k_numpy(o):
    """Decode against the numpy decoder; the matmul against the plain dequantized dot."""
    rng = np.random.default_rng(14)
    E, k, K, N, T = 3, 2, 512, 5, 4
    act = o.quantize_q8_1(rng.standard_normal((T, K)).astype(np.float16))
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    xa = numpy_decode_q8_1(act)
    for wtype in ("q2_k", "q3_k"):
        w = _gguf_random(wtype, E=E, N=N, K=K, seed=15)
        wv = numpy_decode_q2k_q3k(wtype, w)
        assert np.array_equal(o.dequantize_gguf(wtype, w), wv), wtype
        wv = wv.reshape(E, N, K)
        got = o.moe_gguf(wtype, w, act, ids).astype(np.float64)
        for t in range(T):
            for j in range(k):
                want = wv[ids[t, j]] @ xa[t]
                scale = np.abs(wv[ids[t, j]]) @ np.abs(xa[t])
                assert np.all(np.abs(got[t, j] - want) <= 1e-6 * scale + 1e-12), wtype


ALL_PINS = [
    pin_fp16, pin_q4_0_hand, pin_q4_0_nearest_level, pin_q4_0_matches_generator, pin_q4_0_dequant,
    pin_q8_1_hand, pin_q8_1_numpy, pin_q8_1_error_bound, pin_route, pin_block_dot_hand,
    pin_moe_closed_form_vs_bruteforce, pin_moe_numpy_einsum, pin_moe_block_dots,
    pin_moe_split_invariance, pin_moe_bad_ids, pin_moe_slots_numpy_einsum, pin_moe_slots_replicated_rows,
    pin_moe_ep_shards_sum_to_full, pin_act_library, pin_act_tail_accuracy, pin_act_gelu_vs_erf, pin_act_odd_identity, pin_act_hand,
    pin_act_quantize_numpy, pin_gguf_hand, pin_gguf_numpy_decode, pin_gguf_moe_numpy,
    pin_gguf_q4_0_is_the_q4_0_matmul, pin_kquant_hand, pin_kquant_numpy_decode, pin_kquant_moe_numpy,
    pin_kquant_unit_scales_are_q4_1, pin_q6k_hand, pin_q6k_numpy, pin_repack_q4_0_soa, pin_q2k_q3k_hand,
    pin_q2k_q3k_numpy,
]
