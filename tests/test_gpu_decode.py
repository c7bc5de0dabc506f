"""GPU parity of ft_moe_q4_0_fp16, the hot path from fp16 activations.

A decode-sized batch (at most 512 slots and 1024 experts, ncols % 256 == 0,
x 16-byte aligned, at most 4 slots per expert on average) runs as ONE launch
in which every CTA routes the slots and quantizes its rows itself; the result
must equal ft_quantize_q8_1 followed by ft_moe_q4_0_q8_1 bit for bit (same
GEMV plan, same arithmetic), and match the oracle within the matmul
tolerance.  Outside those limits (among them batches whose tiles run on the
mma.sync kernel) the entry point quantizes into workspace and takes the usual
path: still bit-equal to the two calls.  Bad ids give zero rows and the
device error flag on both forms.
"""

import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu


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


def _custom(E, k, K, N, T, seed, routing="uniform"):
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.custom_workload(E, k, K, N, seed, routing=routing)
    return synth.make_weights(wl), synth.make_activations(wl, T), synth.make_topk_ids(wl, T)


def _launches(ft, fn):
    ft.profile_enable(4)
    fn()
    p = ft.profile_read()
    ft.profile_enable(0)
    return p["launches"]


def _two_calls(ft, w, x, ids):
    return ft.moe_q4_0_q8_1(w, ft.quantize_q8_1(x), ids)


# (E, k, K, N, T, seed, routing): one token of the 8-expert layer (G = 1,
# K-split), 16 tokens over 1024 columns (4-slot tiles), the 128-expert top-8
# layer at 1, 8 and 64 tokens (64 x 8 = 512 slots: the limit), a ragged small
# layer, 1024 experts (the limit)
ONE_LAUNCH = [
    (8, 2, 4096, 14336, 1, 4, "uniform"),
    (8, 2, 1024, 14336, 16, 4, "uniform"),
    (128, 8, 2048, 768, 1, 3, "zipf"),
    (128, 8, 2048, 768, 8, 3, "zipf"),
    (128, 8, 2048, 768, 64, 3, "zipf"),
    (5, 2, 512, 200, 10, 40, "uniform"),
    (1024, 4, 256, 64, 40, 41, "uniform"),
]


@pytest.mark.parametrize("E,k,K,N,T,seed,routing", ONE_LAUNCH)
def test_one_launch_equals_quantize_then_matmul(ft, oracle, E, k, K, N, T, seed, routing):
    import torch
    w, x, ids = _custom(E, k, K, N, T, seed, routing)
    dw, dx, di = G.dev(w), G.dev(x), G.dev(ids)
    assert ft.selected_path(T, k, E, N, K) == ft.FT_PATH_GEMV
    out = ft.moe_q4_0_fp16(dw, dx, di)
    ref2 = _two_calls(ft, dw, dx, di)
    torch.cuda.synchronize()
    assert torch.equal(out, ref2), "one launch differs from quantize + matmul"
    assert _launches(ft, lambda: ft.moe_q4_0_fp16(dw, dx, di, out=out)) == 1
    assert ft.read_device_error() == 0
    # against the oracle: every output for the small cases, sampled for the big ones
    act = oracle.quantize_q8_1(x)
    if T * k * N <= 200_000:
        ref = oracle.moe(w, act, ids)
        wn, xn = G.full_norms(oracle, w, act, ids)
        G.check_close(G.host(out), ref, wn, xn, f"one launch {E},{k},{K},{N},{T}")
    else:
        rng = np.random.default_rng(seed)
        S = T * k
        slots = rng.integers(0, S, 3000)
        rows = rng.integers(0, N, 3000)
        ref = oracle.moe_sample(w, act, ids, slots, rows)
        got = G.host(out).reshape(S, N)[slots, rows]
        e = ids.reshape(-1)[slots]
        wn = G.row_norms_w(oracle, w, e, rows)
        xn = G.act_norms(oracle, act)[slots // k]
        G.check_close(got, ref, wn, xn, f"one launch sample {E},{k},{K},{N},{T}")


@pytest.mark.parametrize("misaligned", [False, True])
def test_bad_ids_zero_rows(ft, oracle, misaligned):
    """Both forms (one launch; x 8-byte aligned only: quantize + route +
    matmul): rows of bad slots are zero, the flag is raised, the rest match."""
    import torch
    w, x, ids = _custom(16, 2, 1024, 300, 24, 42)
    ids = ids.copy()
    ids[0, 0] = -1
    ids[7, 1] = 16
    ids[23, 1] = 1 << 20
    dw, di = G.dev(w), G.dev(ids)
    if misaligned:
        buf = torch.zeros(x.size + 4, dtype=torch.float16, device="cuda")
        dx = buf[4:].view(x.shape)
        dx.copy_(G.dev(x))
    else:
        dx = G.dev(x)
    ft.read_device_error()
    out = torch.full((24, 2, 300), 7.0, dtype=torch.float32, device="cuda")
    n = _launches(ft, lambda: ft.moe_q4_0_fp16(dw, dx, di, out=out))
    assert n == (1 if not misaligned else 3)
    assert ft.read_device_error() == ft.FT_DEVERR_BAD_EXPERT_ID
    got = G.host(out)
    for t, j in ((0, 0), (7, 1), (23, 1)):
        assert not got[t, j].any()
    ref2 = _two_calls(ft, dw, dx, di)
    torch.cuda.synchronize()
    ft.read_device_error()
    assert torch.equal(out, ref2)
    act = oracle.quantize_q8_1(x)
    ref = oracle.moe(w, act, ids)
    wn, xn = G.full_norms(oracle, w, act, ids)
    G.check_close(got, ref, wn, xn, "bad ids")


@pytest.mark.parametrize("E,k,K,N,T,path", [
    (128, 8, 2816, 1408, 2048, "auto"),      # prefill: quantize into workspace, tensor cores
    (8, 2, 256, 128, 300, "gemv"),           # 600 slots: past the one-launch limit
    (8, 2, 800, 100, 9, "auto"),             # ncols % 256 != 0: block-per-lane GEMV
    (8, 2, 4096, 14336, 32, "auto"),         # 8-slot tiles of 4096 columns: mma.sync tiles
    (8, 2, 1024, 14336, 32, "auto"),         # 8-slot tiles of 1024 columns: mma.sync tiles
    (2000, 2, 256, 64, 4, "auto"),           # more experts than the one-launch limit
    (8, 2, 512, 256, 16, "gemm"),            # forced tensor cores
])
def test_other_batches_equal_quantize_then_matmul(ft, E, k, K, N, T, path):
    import torch
    w, x, ids = _custom(E, k, K, N, T, 43)
    dw, dx, di = G.dev(w), G.dev(x), G.dev(ids)
    ft.set_path(path)
    try:
        out = ft.moe_q4_0_fp16(dw, dx, di)
        ref2 = _two_calls(ft, dw, dx, di)
        torch.cuda.synchronize()
        assert torch.equal(out, ref2)
        assert _launches(ft, lambda: ft.moe_q4_0_fp16(dw, dx, di, out=out)) >= 2
        assert ft.read_device_error() == 0
    finally:
        ft.set_path("auto")


def test_one_launch_replays_in_a_cuda_graph(ft):
    """Captured once, replayed with new inputs copied into the same buffers."""
    import torch
    w, x, ids = _custom(8, 2, 4096, 14336, 1, 44)
    _, x2, ids2 = _custom(8, 2, 4096, 14336, 1, 45)
    dw, dx, di = G.dev(w), G.dev(x), G.dev(ids)
    out = torch.empty((1, 2, 14336), dtype=torch.float32, device="cuda")
    ft.reserve(1, 2, 8, 14336, 4096)
    ft.moe_q4_0_fp16(dw, dx, di, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ft.moe_q4_0_fp16(dw, dx, di, out=out)
    torch.cuda.current_stream().wait_stream(s)
    dx.copy_(G.dev(x2))
    di.copy_(G.dev(ids2))
    g.replay()
    torch.cuda.synchronize()
    ref = _two_calls(ft, dw, dx, di)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
