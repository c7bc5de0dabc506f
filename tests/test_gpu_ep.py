"""GPU parity of ft_moe_q4_0_q8_1_ep: the routed matmul on one
expert-parallel shard (global expert ids remapped by the shard's first
expert, other slots masked: nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 8).

Each shard against the oracle's shard matmul within the matmul tolerance on
both paths; the shards of a partition summed against the full matmul; a shard
holding every expert bit for bit against the regular entry point; and the
error flag raised for ids no shard owns, never for ids another shard owns."""

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


def _case(E, k, K, N, T, seed):
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.custom_workload(E, k, K, N, seed)
    return synth.make_weights(wl), synth.make_activations(wl, T), synth.make_topk_ids(wl, T)


# (shape, shard bounds): GEMV-sized and tensor-core-sized batches, ragged rows
CASES = [((8, 2, 256, 128, 16, 80), (0, 3, 8)), ((8, 2, 512, 256, 1000, 81), (0, 5, 8)),
         ((6, 3, 768, 130, 300, 82), (0, 2, 4, 6))]


@pytest.mark.parametrize("shape,bounds", CASES)
@pytest.mark.parametrize("path_name", ["gemv", "gemm"])
def test_shards_match_oracle_and_sum_to_full(path, oracle, shape, bounds, path_name):
    E, k, K, N, T, seed = shape
    w, x, ids = _case(*shape)
    act = oracle.quantize_q8_1(x)
    path.set_path(path_name)
    wn, xn = G.full_norms(oracle, w, act, ids)
    total = np.zeros((T, k, N), dtype=np.float64)
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        got = G.host(path.moe_q4_0_q8_1_ep(G.dev(w[lo:hi]), G.dev(act), G.dev(ids), E, lo))
        ref = oracle.moe_ep(w[lo:hi], act, ids, E, lo)
        local = (ids >= lo) & (ids < hi)
        assert not got[~local].any()                          # other shards' slots are zero rows
        G.check_close(got, ref, wn, xn, f"shard [{lo},{hi}) {shape}/{path_name}")
        total += got
    G.check_close(total, oracle.moe(w, act, ids), wn, xn, f"sum of shards {shape}/{path_name}")
    assert path.read_device_error() == 0


@pytest.mark.parametrize("path_name", ["gemv", "gemm"])
def test_shard_with_every_expert_is_the_full_matmul(path, oracle, path_name):
    w, x, ids = _case(8, 2, 512, 256, 300, 83)
    act = oracle.quantize_q8_1(x)
    path.set_path(path_name)
    a = G.host(path.moe_q4_0_q8_1(G.dev(w), G.dev(act), G.dev(ids)))
    b = G.host(path.moe_q4_0_q8_1_ep(G.dev(w), G.dev(act), G.dev(ids), 8, 0))
    assert np.array_equal(a, b)


def test_error_flag_only_for_ids_no_shard_owns(path, oracle):
    w, x, ids = _case(8, 2, 256, 128, 16, 84)
    act = oracle.quantize_q8_1(x)
    path.set_path("auto")
    path.read_device_error()
    path.moe_q4_0_q8_1_ep(G.dev(w[2:5]), G.dev(act), G.dev(ids), 8, 2)    # most ids belong to other shards
    assert path.read_device_error() == 0
    bad = ids.copy()
    bad[3, 1] = 8                                                          # no shard owns expert 8
    out = G.host(path.moe_q4_0_q8_1_ep(G.dev(w[2:5]), G.dev(act), G.dev(bad), 8, 2))
    assert path.read_device_error() & path.FT_DEVERR_BAD_EXPERT_ID
    assert not out[3, 1].any()


def test_rejects_a_shard_outside_the_experts(path):
    from bit_quantized_moe_quantize_gb300 import FtError
    w, x, ids = _case(8, 2, 256, 128, 4, 85)
    act = np.zeros((4, 8, 36), np.uint8)
    with pytest.raises(FtError) as ei:
        path.moe_q4_0_q8_1_ep(G.dev(w[5:8]), G.dev(act), G.dev(ids), 8, 6)   # [6, 9) is not inside [0, 8)
    assert ei.value.status == 1
