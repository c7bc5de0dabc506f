"""Helpers for the GPU parity tests: device copies, seeded cases, tolerances.

Tolerance (floating outputs of the routed matmul), per element and overall:
    |gpu - oracle| <= 1e-3 * ||w_row|| * ||x||          (max error)
    ||gpu - oracle||_2 / ||oracle||_2 <= 1e-4            (relative L2)
with ||w_row|| the L2 norm of the dequantized Q4_0 weight row and ||x|| that
of the dequantized Q8_1 activation row of the slot's token.  Integer results
(Q8_1 bytes, counts, offsets, permutation, per-block dots) must be identical.
"""

from __future__ import annotations

import functools

import numpy as np

MAX_ERR_FACTOR = 1e-3
REL_L2 = 1e-4


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


@functools.lru_cache(maxsize=None)
def case(name: str, tokens: int):
    from bit_quantized_moe_quantize_gb300 import synth
    return synth.make_case(name, tokens)


@functools.lru_cache(maxsize=None)
def weights_of(name: str):
    from bit_quantized_moe_quantize_gb300 import synth
    return synth.make_weights(synth.WORKLOADS[name])


def row_norms_w(oracle, weights, e, r):
    """L2 norms of dequantized weight rows (e[i], r[i])."""
    E, N, nb, _ = weights.shape
    out = np.empty(len(e))
    for i, (ee, rr) in enumerate(zip(e, r)):
        out[i] = np.linalg.norm(oracle.dequantize_q4_0(weights[ee, rr]))
    return out


def act_norms(oracle, act):
    return np.linalg.norm(oracle.dequantize_q8_1(act), axis=-1)


def check_close(gpu, ref, wnorm, xnorm, what=""):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    bound = MAX_ERR_FACTOR * np.asarray(wnorm).reshape(-1) * np.asarray(xnorm).reshape(-1)
    err = np.abs(gpu - ref)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, f"{what}: {bad.size} elements over the max-error bound, first {bad[:5]}, " \
                          f"err {err[bad[:5]]}, bound {bound[bad[:5]]}"
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(gpu - ref) / denom if denom > 0 else np.linalg.norm(gpu - ref)
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3e} > {REL_L2}"
    return rel


def full_norms(oracle, weights, act, ids):
    """Per-output-element (w_row norm, x norm) for the whole [T, k, N] output."""
    E, N, nb, _ = weights.shape
    wn = np.linalg.norm(oracle.dequantize_q4_0(weights.reshape(E * N, nb, 18)), axis=-1).reshape(E, N)
    xn = act_norms(oracle, act)                        # [T]
    idc = np.clip(ids, 0, E - 1)
    return wn[idc], np.broadcast_to(xn[:, None, None], (*ids.shape, N))


def full_norms_slots(oracle, weights, act_slots, ids):
    """As full_norms, with one activation row per slot (act_slots [T*k, nb, 36])."""
    E, N, nb, _ = weights.shape
    wn = np.linalg.norm(oracle.dequantize_q4_0(weights.reshape(E * N, nb, 18)), axis=-1).reshape(E, N)
    xn = act_norms(oracle, act_slots).reshape(ids.shape)   # [T, k]
    idc = np.clip(ids, 0, E - 1)
    return wn[idc], np.broadcast_to(xn[:, :, None], (*ids.shape, N))
