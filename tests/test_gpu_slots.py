"""GPU parity of ft_moe_q4_0_q8_1_slots: the routed matmul with one Q8_1
activation row per routed slot (the second expert layer's input, the first
layer's output after SiLU*up; nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6).

Both paths against the oracle's per-slot matmul within the matmul tolerance,
and, with every slot given its token's row, bit for bit against the per-token
entry point on the same path."""

import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def path():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_quantized_moe_quantize_gb300 as ft
    from bit_quantized_moe_quantize_gb300 import build
    build.build()
    ft.load()
    prev = ft.set_path("auto")
    yield ft
    ft.set_path(prev)


def _slots_case(E, k, K, N, T, seed):
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.custom_workload(E, k, K, N, seed)
    w = synth.make_weights(wl)
    x_slots = synth.make_activations(wl, T * k)       # one fp16 row per slot
    ids = synth.make_topk_ids(wl, T)
    return w, x_slots, ids


# tiny GEMV tiles; 32-wide and 128-wide tensor-core tiles; ragged rows and K stages
CASES = [(8, 2, 256, 128, 16, 70), (5, 2, 512, 200, 77, 71), (8, 2, 512, 256, 1000, 72), (3, 3, 768, 130, 300, 73)]


@pytest.mark.parametrize("E,k,K,N,T,seed", CASES)
@pytest.mark.parametrize("path_name", ["gemv", "gemm"])
def test_slots_match_oracle(path, oracle, E, k, K, N, T, seed, path_name):
    w, x_slots, ids = _slots_case(E, k, K, N, T, seed)
    act_slots = oracle.quantize_q8_1(x_slots)
    ref = oracle.moe_slots(w, act_slots, ids)
    path.set_path(path_name)
    got = G.host(path.moe_q4_0_q8_1_slots(G.dev(w), G.dev(act_slots), G.dev(ids)))
    wn, xn = G.full_norms_slots(oracle, w, act_slots, ids)
    G.check_close(got, ref, wn, xn, f"slots {E},{k},{K},{N},{T}/{path_name}")


@pytest.mark.parametrize("E,k,K,N,T,seed", CASES)
@pytest.mark.parametrize("path_name", ["gemv", "gemm"])
def test_slots_with_token_rows_equal_per_token(path, oracle, E, k, K, N, T, seed, path_name):
    w, x, ids = _slots_case(E, k, K, N, T, seed)
    act = oracle.quantize_q8_1(x[:T])
    act_slots = np.repeat(act, k, axis=0)
    path.set_path(path_name)
    a = G.host(path.moe_q4_0_q8_1(G.dev(w), G.dev(act), G.dev(ids)))
    b = G.host(path.moe_q4_0_q8_1_slots(G.dev(w), G.dev(act_slots), G.dev(ids)))
    assert np.array_equal(a, b)


def test_slots_full_size_sampled(path, oracle):
    """Prefill-shaped batch (E=128, k=8, K=2816, N=1408, T=2048 -> 16384 slots,
    the tensor-core path): 3000 sampled outputs against the oracle."""
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.WORKLOADS["prefill"]
    w = G.weights_of("prefill")
    T, k = 2048, wl.top_k
    x_slots = synth.make_activations(wl, T * k)
    ids = synth.make_topk_ids(wl, T)
    path.set_path("auto")
    act_d = path.quantize_q8_1(G.dev(x_slots))
    out = G.host(path.moe_q4_0_q8_1_slots(G.dev(w), act_d, G.dev(ids))).reshape(T * k, wl.nrows)
    act_slots = G.host(act_d)
    rng = np.random.default_rng(5)
    s = rng.integers(0, T * k, 3000)
    r = rng.integers(0, wl.nrows, 3000)
    # oracle per-slot values, one by one: the per-token sampler on a one-slot-per-token view
    ids_flat = ids.reshape(-1, 1)
    ref = oracle.moe_sample(w, act_slots, ids_flat, s, r)
    wn = G.row_norms_w(oracle, w, ids_flat[s, 0], r)
    xn = G.act_norms(oracle, act_slots[s])
    G.check_close(out[s, r], ref, wn, xn, "slots prefill T=2048 sampled")
