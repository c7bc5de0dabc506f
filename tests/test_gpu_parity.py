"""CUDA path vs the CPU oracle, through the C ABI (GPU only).

Integer work is compared bit for bit: Q8_1 bytes, counts, offsets, the
permutation, and the per-block integer dots of both matmul paths.  Floating
outputs are compared element by element within the tolerance stated in
gpu_util.  Sizes run from the tiny layer (several tiles and ragged tails) to
the full prefill / Qwen3 / Mixtral shapes, where outputs are sampled and the
oracle computes each sampled element on its own.
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
    ft.set_path("auto")
    return ft


@pytest.fixture
def path(ft):
    prev = ft.set_path("auto")
    yield ft
    ft.set_path(prev)


# ------------------------------------------------------------------ quantizer
@pytest.mark.parametrize("T,K,seed", [(1, 32, 0), (16, 256, 1), (7, 2816, 2), (33, 4096, 3), (0, 64, 4)])
def test_quantize_bit_exact(ft, oracle, T, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K)).astype(np.float16)
    if T > 3:
        x[1] = 0                                   # amax == 0 blocks
        x[2, :32] = np.float16(3e-6)               # d lands in fp16 subnormals
        x[3] *= np.float16(40)                     # large values
    got = G.host(ft.quantize_q8_1(G.dev(x)))
    want = oracle.quantize_q8_1(x)
    assert np.array_equal(got, want)


def _near_tie_rows():
    """Every fp16 value in [-m, m] for several block maxima m, 31 per block plus
    m itself: x / d lands on or next to half integers over and over."""
    blocks = []
    for m in (12.7, 1.0, 127.0, 0.3, 5e-3, 3e4):
        m16 = np.float16(m)
        allv = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)
        allv = allv[(allv > 0) & (allv <= m16)]
        allv = np.concatenate([allv, -allv])
        n = len(allv) // 31 * 31
        b = allv[:n].reshape(-1, 31)
        blocks.append(np.concatenate([b, np.full((len(b), 1), m16, dtype=np.float16)], axis=1))
    v = np.concatenate(blocks)
    v = v[: len(v) // 8 * 8]
    return v.reshape(-1, 256)


@pytest.mark.parametrize("copies", [1, 12], ids=["lane_groups", "block_per_thread"])
def test_quantize_near_ties_bit_exact(ft, oracle, copies):
    """The reciprocal-multiply quotient must round like the IEEE division on
    every near tie; one copy (6992 blocks) runs the small-batch kernel, twelve
    copies (past two 256-thread CTAs per SM of blocks) the one-thread-per-block
    kernel."""
    x = np.concatenate([_near_tie_rows()] * copies)
    got = G.host(ft.quantize_q8_1(G.dev(x)))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


def test_quantize_unaligned_input(ft, oracle):
    """x only 8-byte aligned on a batch big enough for the one-thread-per-block
    kernel: its 16-byte loads are not used, same bytes."""
    import torch
    x = np.random.default_rng(7).standard_normal((4096, 1024)).astype(np.float16)
    buf = torch.empty(x.size + 4, dtype=torch.float16, device="cuda")
    dx = buf[4:].view(4096, 1024)
    dx.copy_(torch.from_numpy(x))
    assert dx.data_ptr() % 16 == 8
    got = G.host(ft.quantize_q8_1(dx))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


@pytest.mark.parametrize("name,T", [("mixtral_8x7b", 32768), ("prefill", 8191)])
def test_quantize_bit_exact_full_size(ft, oracle, name, T):
    x = G.case(name, T)["x"] if name != "mixtral_8x7b" else _mixtral_x(T)
    got = G.host(ft.quantize_q8_1(G.dev(x)))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


def _mixtral_x(T):
    from bit_quantized_moe_quantize_gb300 import synth
    return synth.make_activations(synth.WORKLOADS["mixtral_8x7b"], T)


# --------------------------------------------------------------------- router
ROUTE_CASES = [("tiny", 16), ("launch_limit", 8192), ("launch_limit", 16384), ("prefill", 8191),
               ("qwen3_30b_a3b", 1), ("qwen3_30b_a3b", 64), ("qwen3_30b_a3b", 8192), ("mixtral_8x7b", 32768)]


@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_route_bit_exact(ft, oracle, name, T):
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.WORKLOADS[name]
    ids = synth.make_topk_ids(wl, T)
    c, o, p = ft.route_offsets(G.dev(ids), wl.n_experts)
    rc, ro, rp, bad = oracle.route(ids, wl.n_experts)
    assert bad == 0
    assert np.array_equal(G.host(c), rc)
    assert np.array_equal(G.host(o), ro)
    assert np.array_equal(G.host(p), rp)


def test_route_edge_cases(ft, oracle):
    rng = np.random.default_rng(9)
    for T, k, E in [(1, 1, 1), (3, 2, 2), (1000, 4, 3000), (300, 1, 7), (4096, 8, 8)]:
        ids = rng.integers(0, E, (T, k)).astype(np.int32)
        ids[0] = 0
        c, o, p = ft.route_offsets(G.dev(ids), E)
        rc, ro, rp, _ = oracle.route(ids, E)
        assert np.array_equal(G.host(c), rc) and np.array_equal(G.host(o), ro) and np.array_equal(G.host(p), rp)
    ids = np.full((513, 3), 5, dtype=np.int32)     # all slots on one expert
    c, o, p = ft.route_offsets(G.dev(ids), 6)
    assert np.array_equal(G.host(p), np.arange(513 * 3))
    assert G.host(c).tolist() == [0, 0, 0, 0, 0, 1539]


def test_route_bad_ids_flag(ft, oracle):
    import torch
    ids = np.array([[0, 1], [-1, 2], [3, 9], [2, 2]], dtype=np.int32)
    ft.read_device_error()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    c, o, p = ft.route_offsets(G.dev(ids), 4, dev_err=err)
    rc, ro, rp, bad = oracle.route(ids, 4)
    assert bad == 2
    assert np.array_equal(G.host(p), rp) and np.array_equal(G.host(o), ro)
    assert int(err.item()) & ft.FT_DEVERR_BAD_EXPERT_ID


# ------------------------------------------------------------- matmul, small
def _run(ft, weights, act, ids, path_name):
    ft.set_path(path_name)
    out = ft.moe_q4_0_q8_1(G.dev(weights), G.dev(act), G.dev(ids))
    return G.host(out)


def _dots(ft, weights, act, ids, path_name):
    ft.set_path(path_name)
    return G.host(ft.block_dots(G.dev(weights), G.dev(act), G.dev(ids)))


SMALL = [("tiny", 16)]


@pytest.mark.parametrize("path_name", ["gemv", "gemm"])
def test_tiny_layer_full_compare(path, oracle, path_name):
    c = G.case("tiny", 16)
    act = oracle.quantize_q8_1(c["x"])
    ref = oracle.moe_sample(c["weights"], act, c["topk_ids"],
                            np.repeat(np.arange(32), 128), np.tile(np.arange(128), 32)).reshape(16, 2, 128)
    got = _run(path, c["weights"], act, c["topk_ids"], path_name)
    wn, xn = G.full_norms(oracle, c["weights"], act, c["topk_ids"])
    G.check_close(got, ref, wn, xn, f"tiny/{path_name}")


@pytest.mark.parametrize("path_name", ["gemv", "gemm"])
def test_block_dots_bit_exact(path, oracle, path_name):
    c = G.case("tiny", 16)
    act = oracle.quantize_q8_1(c["x"])
    got = _dots(path, c["weights"], act, c["topk_ids"], path_name)
    assert np.array_equal(got, oracle.moe_block_dots(c["weights"], act, c["topk_ids"]))


def _custom(E, k, K, N, T, seed, routing="uniform", zero_rows=False):
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.custom_workload(E, k, K, N, seed, routing=routing)
    w = synth.make_weights(wl)
    x = synth.make_activations(wl, T)
    ids = synth.make_topk_ids(wl, T)
    if zero_rows:
        x[::5] = 0                                        # amax == 0 activation blocks
        w[:, ::7, ::3] = np.frombuffer(bytes([0, 0] + [0x88] * 16), np.uint8)   # d == 0 weight blocks
    return w, x, ids


RAGGED = [
    # E, k, K, N, T, seed: ragged rows (N % 128), ragged slot tiles, several K stages
    (5, 2, 512, 200, 77, 11),
    (3, 3, 768, 130, 300, 12),
    (16, 4, 256, 64, 129, 13),
    (2, 1, 4096, 260, 400, 14),
]


@pytest.mark.parametrize("E,k,K,N,T,seed", RAGGED)
@pytest.mark.parametrize("path_name", ["gemv", "gemv_dp4a", "gemm"])
def test_ragged_full_compare(path, oracle, E, k, K, N, T, seed, path_name):
    w, x, ids = _custom(E, k, K, N, T, seed, zero_rows=True)
    act = oracle.quantize_q8_1(x)
    ref = oracle.moe(w, act, ids).astype(np.float64)
    got = _run(path, w, act, ids, path_name)
    wn, xn = G.full_norms(oracle, w, act, ids)
    G.check_close(got, ref, wn, xn, f"ragged {E},{k},{K},{N},{T}/{path_name}")


# the first two take the 32-wide tensor-core tiles (few slots per expert), the
# last two the 128-wide tiles (many slots per expert)
@pytest.mark.parametrize("E,k,K,N,T,seed", [(5, 2, 512, 200, 77, 11), (16, 4, 256, 64, 129, 13),
                                            (3, 3, 768, 130, 300, 12), (2, 1, 4096, 260, 400, 14)])
@pytest.mark.parametrize("path_name", ["gemv", "gemv_dp4a", "gemm"])
def test_ragged_block_dots(path, oracle, E, k, K, N, T, seed, path_name):
    w, x, ids = _custom(E, k, K, N, T, seed, zero_rows=True)
    act = oracle.quantize_q8_1(x)
    assert np.array_equal(_dots(path, w, act, ids, path_name), oracle.moe_block_dots(w, act, ids))


@pytest.mark.parametrize("K", [96, 288, 800])
def test_gemv_odd_row_lengths(path, oracle, K):
    """ncols not a multiple of 256: rows are not 16-byte aligned (GEMV plain-load path)."""
    w, x, ids = _custom(4, 2, K, 40, 9, 20 + K)
    act = oracle.quantize_q8_1(x)
    assert path.selected_path(9, 2, 4, 40, K) == path.FT_PATH_GEMV
    got = _run(path, w, act, ids, "auto")
    wn, xn = G.full_norms(oracle, w, act, ids)
    G.check_close(got, oracle.moe(w, act, ids), wn, xn, f"K={K}")
    assert np.array_equal(_dots(path, w, act, ids, "auto"), oracle.moe_block_dots(w, act, ids))


# 8-slot GEMV tiles on the mma.sync kernel ("gemv"; "gemv_dp4a" keeps them on
# the dp4a row kernel): exact block dots, outputs within the tolerance of the
# oracle; ragged row counts (not a multiple of 32 rows per warp), one and
# several boxes per row, experts with a second, partial tile, a bad id.  Both
# kernels form the same integer block dots and scale them in the same order,
# so where the dp4a kernel does not split K (one box per row, K = 256, or
# enough row groups: the full Mixtral-shaped layer) they agree bit for bit.
MMA_CASES = [
    # E, k, K, N, T, seed, bit-identical to the dp4a kernel: 5..8 slots per expert on average
    (8, 2, 4096, 14336 // 8, 32, 70, False),
    (8, 2, 256, 77, 20, 71, True),
    (4, 4, 768, 300, 7, 72, False),
    (16, 4, 2048, 520, 30, 73, False),
    (3, 2, 512, 1000, 11, 74, False),
    (6, 3, 256, 4000, 13, 75, True),
]


@pytest.mark.parametrize("E,k,K,N,T,seed,same", MMA_CASES)
def test_gemv_mma_tiles(path, oracle, E, k, K, N, T, seed, same):
    w, x, ids = _custom(E, k, K, N, T, seed, zero_rows=True)
    ids = ids.copy()
    ids[T // 2, 0] = E                                    # a bad id: zero row, flag
    act = oracle.quantize_q8_1(x)
    mean = T * k / E
    assert 4.0 < mean <= 8.0
    path.read_device_error()
    a = _run(path, w, act, ids, "gemv")
    assert path.read_device_error() & path.FT_DEVERR_BAD_EXPERT_ID
    assert not a[T // 2, 0].any()
    ref = oracle.moe(w, act, ids)
    wn, xn = G.full_norms(oracle, w, act, ids)
    G.check_close(a, ref, wn, xn, f"mma {E},{k},{K},{N},{T}")
    assert np.array_equal(_dots(path, w, act, ids, "gemv"), oracle.moe_block_dots(w, act, ids))
    b = _run(path, w, act, ids, "gemv_dp4a")
    if same:
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    else:
        G.check_close(a, b, wn, xn, f"mma vs dp4a {E},{k},{K},{N},{T}")


@pytest.mark.parametrize("wtype", ["q4_0", "q4_k"])
def test_gemv_mma_one_slot_group_long_rows(path, oracle, wtype):
    """Rows of 14336 weights (the Mixtral-shaped second layer, 4096 rows): the
    staged 16-slot activation tile does not fit, so the tiles hold one group
    of 8 slots (experts with more get a second tile) and 56 boxes per row;
    sampled outputs of every slot against the oracle, a bad id."""
    from bit_quantized_moe_quantize_gb300 import synth
    E, k, K, N, T = 8, 2, 14336, 4096, 30
    wl = synth.custom_workload(E, k, K, N, 120)
    w = synth.make_weights(wl) if wtype == "q4_0" else synth.make_weights_gguf(wl, wtype)
    x, ids = synth.make_activations(wl, T), synth.make_topk_ids(wl, T).copy()
    ids[7, 1] = -1
    act = oracle.quantize_q8_1(x)
    path.set_path("auto")
    path.read_device_error()
    if wtype == "q4_0":
        got = G.host(path.moe_q4_0_q8_1(G.dev(w), G.dev(act), G.dev(ids)))
    else:
        got = G.host(path.moe_gguf_q8_1(wtype, G.dev(w), G.dev(act), G.dev(ids)))
    assert path.read_device_error() & path.FT_DEVERR_BAD_EXPERT_ID
    assert not got[7, 1].any()
    S = T * k
    rng = np.random.default_rng(121)
    slots = np.repeat(np.arange(S), 40)
    rows = rng.integers(0, N, slots.size)
    keep = ids.reshape(-1)[slots] >= 0
    slots, rows = slots[keep], rows[keep]
    flat = ids.reshape(-1)
    if wtype == "q4_0":
        ref = oracle.moe_sample(w, act, ids, slots, rows)
        wn = G.row_norms_w(oracle, w, flat[slots], rows)
    else:
        toks = np.unique(slots // k)[:3]
        sel = np.isin(slots // k, toks)
        slots, rows = slots[sel], rows[sel]
        full = oracle.moe_gguf(wtype, w, act[toks], ids[toks]).reshape(len(toks) * k, N)
        pos = {t: i for i, t in enumerate(toks)}
        ref = full[[pos[s // k] * k + s % k for s in slots], rows]
        deq = oracle.dequantize_gguf(wtype, w[flat[slots], rows])
        wn = np.linalg.norm(deq, axis=-1)
    xn = G.act_norms(oracle, act)[slots // k]
    G.check_close(got.reshape(S, N)[slots, rows], ref, wn, xn, f"{wtype} long rows")


@pytest.mark.parametrize("T", [24, 32])
def test_gemv_mma_full_size_matches_dp4a(path, oracle, T):
    """The Mixtral-shaped layer at 6 and 8 slots per expert: the mma.sync tiles
    and the dp4a row kernel (unsplit K at this size) give the same bits, and
    sampled outputs match the oracle."""
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.WORKLOADS["mixtral_8x7b"]
    w = G.weights_of("mixtral_8x7b")
    x = synth.make_activations(wl, T)
    ids = synth.make_topk_ids(wl, T)
    act = oracle.quantize_q8_1(x)
    a = _run(path, w, act, ids, "gemv")
    b = _run(path, w, act, ids, "gemv_dp4a")
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    S, N = T * wl.top_k, wl.nrows
    rng = np.random.default_rng(2000 + T)
    slots, rows = rng.integers(0, S, 2000), rng.integers(0, N, 2000)
    ref = oracle.moe_sample(w, act, ids, slots, rows)
    wn = G.row_norms_w(oracle, w, ids.reshape(-1)[slots], rows)
    xn = G.act_norms(oracle, act)[slots // wl.top_k]
    G.check_close(a.reshape(S, N)[slots, rows], ref, wn, xn, f"mixtral T={T}")


def test_gemm_rejects_unaligned_k(path):
    from bit_quantized_moe_quantize_gb300 import FtError
    w, x, ids = _custom(4, 2, 288, 40, 9, 31)
    path.set_path("gemm")
    with pytest.raises(FtError) as ei:
        path.moe_q4_0_q8_1(G.dev(w), G.dev(np.zeros((9, 9, 36), np.uint8)), G.dev(ids))
    assert ei.value.status == 1


def test_bad_ids_zero_rows_and_flag(path, oracle):
    w, x, ids = _custom(4, 2, 256, 128, 6, 40)
    ids = ids.copy()
    ids[1, 0] = -1
    ids[4, 1] = 4
    act = oracle.quantize_q8_1(x)
    ref = oracle.moe(w, act, ids)
    for p in ("gemv", "gemv_dp4a", "gemm"):
        path.read_device_error()
        out = G.dev(np.full((6, 2, 128), np.nan, np.float32))
        path.set_path(p)
        path.moe_q4_0_q8_1(G.dev(w), G.dev(act), G.dev(ids), out=out)
        got = G.host(out)
        assert not got[1, 0].any() and not got[4, 1].any()
        assert np.isfinite(got).all()
        wn, xn = G.full_norms(oracle, w, act, ids)
        G.check_close(got, ref, wn, xn, f"bad ids/{p}")
        assert path.read_device_error() & path.FT_DEVERR_BAD_EXPERT_ID


def test_empty_batch_is_noop(ft):
    import torch
    w = torch.zeros((4, 8, 8, 18), dtype=torch.uint8, device="cuda")
    out = ft.moe_q4_0_q8_1(w, torch.zeros((0, 8, 36), dtype=torch.uint8, device="cuda"),
                           torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    assert out.shape == (0, 2, 8)


# ------------------------------------------------- launch limit (grid.z cap)
@pytest.mark.parametrize("T", [8192, 16384])
@pytest.mark.parametrize("path_name", ["gemv", "gemm"])
def test_launch_limit_matches_oracle_and_halves(path, oracle, T, path_name):
    """tokens * top_k = 65536 / 131072 slots: one launch equals the oracle and the
    concatenation of its two halves (each under the old 65535 grid.z cap)."""
    c = G.case("launch_limit", T)
    act = oracle.quantize_q8_1(c["x"])
    ids = c["topk_ids"]
    got = _run(path, c["weights"], act, ids, path_name)
    ref = oracle.moe(c["weights"], act, ids)
    wn, xn = G.full_norms(oracle, c["weights"], act, ids)
    G.check_close(got, ref, wn, xn, f"launch_limit T={T}/{path_name}")
    h = T // 2
    a = _run(path, c["weights"], act[:h], ids[:h], path_name)
    b = _run(path, c["weights"], act[h:], ids[h:], path_name)
    assert np.array_equal(got, np.concatenate([a, b]))


def test_slot_count_just_below_and_above_cap(path, oracle):
    """tokens * top_k = 65535 (k = 5, T = 13107) and 65536 both launch and match."""
    for T, k in [(13107, 5), (16384, 4)]:
        w, x, ids = _custom(8, k, 256, 128, T, 50 + k)
        act = oracle.quantize_q8_1(x)
        ref = oracle.moe(w, act, ids)
        wn, xn = G.full_norms(oracle, w, act, ids)
        for p in ("gemv", "gemm"):
            G.check_close(_run(path, w, act, ids, p), ref, wn, xn, f"T*k={T * k}/{p}")


def test_gemv_and_gemm_agree(path, oracle):
    c = G.case("launch_limit", 8192)
    act = oracle.quantize_q8_1(c["x"])
    a = _run(path, c["weights"], act, c["topk_ids"], "gemv")
    b = _run(path, c["weights"], act, c["topk_ids"], "gemm")
    wn, xn = G.full_norms(oracle, c["weights"], act, c["topk_ids"])
    G.check_close(a, b, wn, xn, "gemv vs gemm")


def test_deterministic(path, oracle):
    c = G.case("tiny", 16)
    act = oracle.quantize_q8_1(c["x"])
    for p in ("gemv", "gemm"):
        r1 = _run(path, c["weights"], act, c["topk_ids"], p)
        r2 = _run(path, c["weights"], act, c["topk_ids"], p)
        assert np.array_equal(r1, r2)


@pytest.mark.parametrize("T", [150, 1000])
def test_graph_capture_replay(path, oracle, T):
    """Quantize + route + matmul captured in a CUDA graph and replayed give the
    eager result bit for bit (no allocation or host sync inside).  T = 150
    (37.5 slots per expert) takes the 32-wide tensor-core tiles, T = 1000 the
    128-wide ones."""
    import torch
    w, x, ids = _custom(8, 2, 512, 256, T, 60)
    dw, dx, di = G.dev(w), G.dev(x), G.dev(ids)
    for p in ("gemv", "gemm"):
        path.set_path(p)
        path.reserve(T, 2, 8, 256, 512)
        act = torch.empty((T, 16, 36), dtype=torch.uint8, device="cuda")
        out = torch.empty((T, 2, 256), dtype=torch.float32, device="cuda")
        path.quantize_q8_1(dx, out=act)
        path.moe_q4_0_q8_1(dw, act, di, out=out)
        eager = G.host(out).copy()
        out.zero_()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                path.quantize_q8_1(dx, out=act)
                path.moe_q4_0_q8_1(dw, act, di, out=out)
        torch.cuda.current_stream().wait_stream(s)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(G.host(out), eager)


# ------------------------------------------------- full sizes, sampled outputs
FULL = [("prefill", 2048), ("prefill", 4096), ("prefill", 8191), ("qwen3_30b_a3b", 1), ("qwen3_30b_a3b", 8),
        ("qwen3_30b_a3b", 64), ("qwen3_30b_a3b", 512), ("qwen3_30b_a3b", 8192), ("mixtral_8x7b", 1),
        ("mixtral_8x7b", 32), ("mixtral_8x7b", 32768)]


@pytest.mark.parametrize("name,T", FULL)
def test_full_size_sampled(path, oracle, name, T):
    """The launch configuration the benchmark times (auto path), on the full
    workload; 3000 sampled outputs (plus every row of a few slots) against the
    oracle element by element, and global invariants over the whole output."""
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.WORKLOADS[name]
    w = G.weights_of(name)
    x = synth.make_activations(wl, T)
    ids = synth.make_topk_ids(wl, T)
    path.set_path("auto")
    dx = G.dev(x)
    act_d = path.quantize_q8_1(dx)
    out = G.host(path.moe_q4_0_q8_1(G.dev(w), act_d, G.dev(ids)))
    act = G.host(act_d)
    assert np.array_equal(act, oracle.quantize_q8_1(x))
    S, N = T * wl.top_k, wl.nrows
    rng = np.random.default_rng(1000 + T)
    n = 3000
    slots = rng.integers(0, S, n)
    rows = rng.integers(0, N, n)
    whole = rng.choice(S, size=min(S, 3), replace=False)
    slots = np.concatenate([slots, np.repeat(whole, N)])
    rows = np.concatenate([rows, np.tile(np.arange(N), len(whole))])
    ref = oracle.moe_sample(w, act, ids, slots, rows)
    got = out.reshape(S, N)[slots, rows]
    flat = ids.reshape(-1)
    wn = G.row_norms_w(oracle, w, flat[slots], rows)
    xn = G.act_norms(oracle, act)[slots // wl.top_k]
    G.check_close(got, ref, wn, xn, f"{name} T={T}")
    assert np.isfinite(out).all()
