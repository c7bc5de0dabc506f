"""GPU parity of ft_moe_gguf_q8_1: the routed matmul with expert weights of the
other GGUF types (Q4_1, Q5_0, Q5_1, Q8_0 with 32-weight blocks; the K-quants
Q2_K, Q3_K, Q4_K, Q5_K, Q6_K with 256-weight super-blocks; the per-type launchers of
moe_vec.cuh on FreeToken PR #185, "Notes").

Against the oracle's matmul of the same type within the matmul tolerance
(max |err| <= 1e-3 ||w_row|| ||x||, relative L2 <= 1e-4, ||w_row|| of the
dequantized weight row); Q4_0 through the same entry point bit for bit equal
to ft_moe_q4_0_q8_1; bad ids; rows not 16-byte aligned; a full-size decode
step of the 8-expert 14336 x 4096 layer; Q4_K on the tensor cores; the
mma.sync decode tiles of Q4_1, Q8_0 and Q4_K, bit for bit against the dp4a
row kernel where it leaves K unsplit; the shapes the path rejects."""

import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu

TYPES = ["q4_1", "q5_0", "q5_1", "q8_0", "q2_k", "q3_k", "q4_k", "q5_k", "q6_k"]
KQ = ("q2_k", "q3_k", "q4_k", "q5_k", "q6_k")


@pytest.fixture(scope="module")
def ft():
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


def _case(wtype, E, k, K, N, T, seed, routing="uniform"):
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.custom_workload(E, k, K, N, seed, routing=routing)
    return synth.make_weights_gguf(wl, wtype), synth.make_activations(wl, T), synth.make_topk_ids(wl, T)


def _check(ft, oracle, wtype, w, x, ids, what):
    act = oracle.quantize_q8_1(x)
    ref = oracle.moe_gguf(wtype, w, act, ids)
    got = G.host(ft.moe_gguf_q8_1(wtype, G.dev(w), G.dev(act), G.dev(ids)))
    E, N, nb, bb = w.shape
    wn = np.linalg.norm(oracle.dequantize_gguf(wtype, w.reshape(E * N, nb, bb)), axis=-1).reshape(E, N)
    xn = G.act_norms(oracle, act)
    idc = np.clip(ids, 0, E - 1)
    G.check_close(got, ref, wn[idc], np.broadcast_to(xn[:, None, None], (*ids.shape, N)), what)
    return got, ref


# (E, k, K, N, T): tiny; 3 blocks per row (rows of 60-102 bytes, not 16-byte
# aligned: 2-byte copies instead of bulk copies, block-per-lane kernel);
# 8-slot tiles; a top-8 decode step with Zipf routing; rows of 1280 weights
# and a ragged row count (row-per-lane kernel with 2- and 4-slot tiles and
# the K range split); the block-per-lane kernel on 800-weight rows
CASES = [(8, 2, 256, 128, 16, 90, "uniform"), (5, 2, 96, 50, 77, 91, "uniform"),
         (8, 2, 512, 256, 1000, 92, "uniform"), (128, 8, 2048, 768, 8, 93, "zipf"),
         (16, 2, 1280, 200, 24, 98, "uniform"), (4, 2, 1280, 72, 7, 99, "uniform"),
         (6, 2, 800, 100, 20, 100, "uniform")]


@pytest.mark.parametrize("wtype", TYPES)
@pytest.mark.parametrize("E,k,K,N,T,seed,routing", CASES)
def test_gguf_matches_oracle(ft, oracle, wtype, E, k, K, N, T, seed, routing):
    if wtype in KQ and K % 256:
        K = 256                         # the K-quants' super-blocks need whole 256-column rows
    w, x, ids = _case(wtype, E, k, K, N, T, seed, routing)
    _check(ft, oracle, wtype, w, x, ids, f"{wtype} {E},{k},{K},{N},{T}")


@pytest.mark.parametrize("wtype", TYPES)
def test_gguf_full_size_decode(ft, oracle, wtype):
    """One token of the 8-expert top-2 layer with 14336 rows of 4096 columns,
    every output against the oracle."""
    w, x, ids = _case(wtype, 8, 2, 4096, 14336, 1, 94)
    _check(ft, oracle, wtype, w, x, ids, f"{wtype} full-size decode")


def test_gguf_q4_0_is_the_q4_0_entry(ft, oracle):
    import torch
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.custom_workload(8, 2, 512, 256, 95)
    w, x, ids = synth.make_weights(wl), synth.make_activations(wl, 300), synth.make_topk_ids(wl, 300)
    act = G.dev(oracle.quantize_q8_1(x))
    dw, di = G.dev(w), G.dev(ids)
    a = ft.moe_gguf_q8_1("q4_0", dw, act, di)
    b = ft.moe_q4_0_q8_1(dw, act, di)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("wtype", ["q5_1", "q8_0"])
def test_gguf_bad_ids_zero_rows(ft, oracle, wtype):
    w, x, ids = _case(wtype, 8, 2, 256, 128, 40, 96)
    ids = ids.copy()
    ids[2, 0] = -3
    ids[9, 1] = 8
    ft.read_device_error()
    got, ref = _check(ft, oracle, wtype, w, x, ids, f"{wtype} bad ids")
    assert not got[2, 0].any() and not got[9, 1].any()
    assert ft.read_device_error() & ft.FT_DEVERR_BAD_EXPERT_ID


# Q4_K on the tensor-core path: (E, k, K, N, T, seed, routing) - 32-wide slot
# tiles, 128-wide tiles with ragged slot counts and a ragged row count, Zipf
# routing with empty experts, and a prefill-sized batch that the host sends to
# the tensor cores by itself
Q4K_GEMM = [(8, 2, 512, 256, 100, 101, "uniform"), (16, 4, 1024, 200, 700, 102, "uniform"),
            (128, 8, 2048, 768, 64, 103, "zipf"), (6, 2, 768, 136, 333, 104, "uniform")]


@pytest.mark.parametrize("E,k,K,N,T,seed,routing", Q4K_GEMM)
def test_q4_k_on_the_tensor_cores(ft, oracle, E, k, K, N, T, seed, routing):
    w, x, ids = _case("q4_k", E, k, K, N, T, seed, routing)
    prev = ft.set_path("gemm")
    try:
        got, ref = _check(ft, oracle, "q4_k", w, x, ids, f"q4_k gemm {E},{k},{K},{N},{T}")
    finally:
        ft.set_path(prev)
    assert ft.read_device_error() == 0


def test_q4_k_tensor_cores_full_size(ft, oracle):
    """The 128-expert top-8 prefill layer (1408 x 2816) at 2048 tokens with Q4_K
    weights: the host picks the tensor cores; every output of 16 seeded tokens
    against the oracle's matmul of the same type on those tokens."""
    from bit_quantized_moe_quantize_gb300 import synth
    E, k, K, N, T = 128, 8, 2816, 1408, 2048
    wl = synth.custom_workload(E, k, K, N, 105)
    w, x, ids = synth.make_weights_gguf(wl, "q4_k"), synth.make_activations(wl, T), synth.make_topk_ids(wl, T)
    assert ft.selected_path(T, k, E, N, K) == ft.FT_PATH_GEMM
    act = oracle.quantize_q8_1(x)
    got = G.host(ft.moe_gguf_q8_1("q4_k", G.dev(w), G.dev(act), G.dev(ids)))
    assert ft.read_device_error() == 0
    toks = np.sort(np.random.default_rng(106).choice(T, 16, replace=False))
    ref = oracle.moe_gguf("q4_k", w, act[toks], ids[toks])
    wn = np.linalg.norm(oracle.dequantize_gguf("q4_k", w.reshape(E * N, -1, 144)), axis=-1).reshape(E, N)
    xn = G.act_norms(oracle, act[toks])
    G.check_close(got[toks], ref, wn[ids[toks]], np.broadcast_to(xn[:, None, None], (16, k, N)), "q4_k gemm full size")


# Q4_K decode tiles on mma.sync (more than 4 slots per expert on average):
# (E, k, K, N, T, seed) and whether the dp4a row kernel leaves K unsplit there
# (one super-block per row), so that the two agree bit for bit
Q4K_MMA = [(8, 2, 256, 77, 20, 110, True), (6, 3, 256, 1000, 13, 111, True), (16, 4, 2048, 520, 30, 112, False),
           (4, 4, 768, 300, 7, 113, False), (3, 2, 512, 1000, 11, 114, False)]


@pytest.mark.parametrize("E,k,K,N,T,seed,same", Q4K_MMA)
def test_q4_k_mma_tiles(ft, oracle, E, k, K, N, T, seed, same):
    w, x, ids = _case("q4_k", E, k, K, N, T, seed)
    ids = ids.copy()
    ids[T // 2, 0] = E                                    # a bad id: zero row, flag
    assert 4.0 < T * k / E <= 16.0
    ft.read_device_error()
    a, ref = _check(ft, oracle, "q4_k", w, x, ids, f"q4_k mma {E},{k},{K},{N},{T}")
    assert not a[T // 2, 0].any()
    assert ft.read_device_error() & ft.FT_DEVERR_BAD_EXPERT_ID
    act = G.dev(oracle.quantize_q8_1(x))
    prev = ft.set_path("gemv_dp4a")
    try:
        b = G.host(ft.moe_gguf_q8_1("q4_k", G.dev(w), act, G.dev(ids)))
    finally:
        ft.set_path(prev)
    ft.read_device_error()
    if same:
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("wtype", ["q4_1", "q8_0"])
@pytest.mark.parametrize("E,k,K,N,T,seed,same", Q4K_MMA)
def test_32_weight_types_mma_tiles(ft, oracle, wtype, E, k, K, N, T, seed, same):
    """Q4_1 and Q8_0 on the mma.sync tiles: against the oracle, a bad id, and
    bit for bit against the dp4a row kernel where it leaves K unsplit."""
    w, x, ids = _case(wtype, E, k, K, N, T, seed)
    ids = ids.copy()
    ids[T // 2, 0] = -1
    ft.read_device_error()
    a, ref = _check(ft, oracle, wtype, w, x, ids, f"{wtype} mma {E},{k},{K},{N},{T}")
    assert not a[T // 2, 0].any()
    assert ft.read_device_error() & ft.FT_DEVERR_BAD_EXPERT_ID
    act = G.dev(oracle.quantize_q8_1(x))
    prev = ft.set_path("gemv_dp4a")
    try:
        b = G.host(ft.moe_gguf_q8_1(wtype, G.dev(w), act, G.dev(ids)))
    finally:
        ft.set_path(prev)
    ft.read_device_error()
    if same:
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("wtype", ["q4_1", "q8_0"])
def test_32_weight_types_mma_full_size(ft, oracle, wtype):
    """The 8-expert top-2 layer (14336 x 4096) at 32 tokens: the mma.sync tiles
    equal the dp4a row kernel bit for bit, and two tokens match the oracle."""
    w, x, ids = _case(wtype, 8, 2, 4096, 14336, 32, 116)
    act = oracle.quantize_q8_1(x)
    a = G.host(ft.moe_gguf_q8_1(wtype, G.dev(w), G.dev(act), G.dev(ids)))
    prev = ft.set_path("gemv_dp4a")
    try:
        b = G.host(ft.moe_gguf_q8_1(wtype, G.dev(w), G.dev(act), G.dev(ids)))
    finally:
        ft.set_path(prev)
    assert ft.read_device_error() == 0
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    toks = np.array([5, 30])
    ref = oracle.moe_gguf(wtype, w, act[toks], ids[toks])
    E, N = 8, 14336
    bb = w.shape[-1]
    wn = np.linalg.norm(oracle.dequantize_gguf(wtype, w.reshape(E * N, -1, bb)), axis=-1).reshape(E, N)
    xn = G.act_norms(oracle, act[toks])
    G.check_close(a[toks], ref, wn[ids[toks]], np.broadcast_to(xn[:, None, None], (2, 2, N)), f"{wtype} mma full size")


def test_q4_k_mma_full_size(ft, oracle):
    """The 8-expert top-2 layer (14336 x 4096) with Q4_K weights at 32 tokens:
    the mma.sync tiles equal the dp4a row kernel bit for bit (K unsplit at this
    size), and every output of two tokens matches the oracle."""
    w, x, ids = _case("q4_k", 8, 2, 4096, 14336, 32, 115)
    act = oracle.quantize_q8_1(x)
    a = G.host(ft.moe_gguf_q8_1("q4_k", G.dev(w), G.dev(act), G.dev(ids)))
    prev = ft.set_path("gemv_dp4a")
    try:
        b = G.host(ft.moe_gguf_q8_1("q4_k", G.dev(w), G.dev(act), G.dev(ids)))
    finally:
        ft.set_path(prev)
    assert ft.read_device_error() == 0
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    toks = np.array([3, 29])
    ref = oracle.moe_gguf("q4_k", w, act[toks], ids[toks])
    E, N = 8, 14336
    wn = np.linalg.norm(oracle.dequantize_gguf("q4_k", w.reshape(E * N, -1, 144)), axis=-1).reshape(E, N)
    xn = G.act_norms(oracle, act[toks])
    G.check_close(a[toks], ref, wn[ids[toks]], np.broadcast_to(xn[:, None, None], (2, 2, N)), "q4_k mma full size")


def test_gguf_rejects_what_the_path_cannot_run(ft, oracle):
    import torch
    w, x, ids = _case("q8_0", 8, 2, 256, 128, 4, 97)
    act = G.dev(oracle.quantize_q8_1(x))
    dw, di = G.dev(w), G.dev(ids)
    prev = ft.set_path("gemm")
    try:
        with pytest.raises(ft.FtError, match="Q4_0 and Q4_K weights only"):
            ft.moe_gguf_q8_1("q8_0", dw, act, di)
    finally:
        ft.set_path(prev)
    # rows of 32736 Q8_0 columns (not a whole number of 256-weight runs, so the
    # block-per-lane kernel): one ring stage of 8 rows does not fit in shared memory
    big = torch.zeros((2, 8, 1023, 34), dtype=torch.uint8, device="cuda")
    xb = torch.zeros((1, 1023, 36), dtype=torch.uint8, device="cuda")
    ib = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(ft.FtError, match="shared memory"):
        ft.moe_gguf_q8_1("q8_0", big, xb, ib)
