"""Failure paths and memory guards, on the GPU, in forms that fault nothing.

* A bounded in-kernel wait that gives up: ft_debug_wait_timeout launches a
  kernel that holds TMEM and waits on an mbarrier nothing arrives on, with a
  limit of a few milliseconds.  It must return, raise FT_DEVERR_WAIT_TIMEOUT
  in the device error word, and leave the context usable: the next routed
  matmuls (both paths) run clean and match the oracle.
* Canaries around the caller's output: the matmul writes exactly the
  [tokens, top_k, nrows] elements it owns, on both paths and on ragged
  shapes; guard elements on either side keep their bit pattern.
* The guard block after the library's workspace keeps its pattern through
  every call (ft_moe_read_device_error reports FT_DEVERR_WORKSPACE_GUARD
  otherwise).
"""

import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu

GUARD = 4099                       # guard elements on each side of the output
SENTINEL = np.uint32(0x7FA5A5A5)   # a NaN bit pattern no kernel writes


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


def _guarded_out(shape):
    """A device buffer with GUARD sentinel floats before and after a contiguous
    view of `shape`; returns (whole buffer, view)."""
    import torch
    n = int(np.prod(shape))
    buf = torch.from_numpy(np.full(n + 2 * GUARD, SENTINEL, np.uint32).view(np.float32)).cuda()
    return buf, buf[GUARD:GUARD + n].view(*shape)


def _guards_intact(buf):
    b = G.host(buf).view(np.uint32)
    return bool((b[:GUARD] == SENTINEL).all() and (b[-GUARD:] == SENTINEL).all())


def test_wait_timeout_returns_and_context_stays_usable(ft, oracle):
    ft.read_device_error()                                  # start from a clear word
    ft.debug_wait_timeout(2_000_000)                        # 2 ms
    assert ft.read_device_error() == ft.FT_DEVERR_WAIT_TIMEOUT
    ft.debug_wait_timeout(1_000)                            # the shortest limit accepted
    assert ft.read_device_error() == ft.FT_DEVERR_WAIT_TIMEOUT
    c = G.case("tiny", 16)
    act = oracle.quantize_q8_1(c["x"])
    ref = oracle.moe(c["weights"], act, c["topk_ids"])
    wn, xn = G.full_norms(oracle, c["weights"], act, c["topk_ids"])
    for p in ("gemv", "gemm"):
        ft.set_path(p)
        got = G.host(ft.moe_q4_0_q8_1(G.dev(c["weights"]), G.dev(act), G.dev(c["topk_ids"])))
        G.check_close(got, ref, wn, xn, f"after timeout/{p}")
        assert ft.read_device_error() == 0


def test_wait_timeout_rejects_bad_limits(ft):
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(ft.FtError) as ei:
            ft.debug_wait_timeout(bad)
        assert ei.value.status == 1


CANARY_CASES = [
    # E, k, K, N, T, seed: both tile widths, ragged rows and slot tiles, K = 96 (GEMV only)
    (4, 2, 256, 128, 16, 21),
    (5, 2, 512, 200, 77, 22),
    (16, 4, 1024, 384, 300, 23),
    (8, 2, 96, 64, 9, 24),
]


@pytest.mark.parametrize("E,k,K,N,T,seed", CANARY_CASES)
def test_output_canaries_and_workspace_guard(ft, oracle, E, k, K, N, T, seed):
    w, x, ids = _custom(E, k, K, N, T, seed)
    act = oracle.quantize_q8_1(x)
    ref = oracle.moe(w, act, ids)
    wn, xn = G.full_norms(oracle, w, act, ids)
    ft.read_device_error()
    paths = ("gemv", "gemm") if K % 256 == 0 else ("gemv",)
    for p in paths:
        ft.set_path(p)
        buf, out = _guarded_out((T, k, N))
        ft.moe_q4_0_q8_1(G.dev(w), G.dev(act), G.dev(ids), out=out)
        assert _guards_intact(buf), f"{p}: the matmul wrote outside its output"
        G.check_close(G.host(out), ref, wn, xn, f"canary/{p}")
        assert ft.read_device_error() == 0, f"{p}: device flag or workspace guard"
        buf, dots = _guarded_out((T * k, N, K // 32))
        import torch
        dots_i = dots.view(torch.int32)
        ft.block_dots(G.dev(w), G.dev(act), G.dev(ids), out=dots_i)
        assert _guards_intact(buf), f"{p}: the block-dot dump wrote outside its output"
        assert np.array_equal(G.host(dots_i), oracle.moe_block_dots(w, act, ids))
        assert ft.read_device_error() == 0


def test_workspace_guard_after_the_largest_calls(ft, oracle):
    """The prefill batch fills the tensor-core path's workspace to its end
    (routed activation copy last); the guard after it must hold."""
    c = G.case("prefill", 8191)
    ft.set_path("gemm")
    x = G.dev(c["x"])
    act = ft.quantize_q8_1(x)
    out = ft.moe_q4_0_q8_1(G.dev(c["weights"]), act, G.dev(c["topk_ids"]))
    assert ft.read_device_error() == 0
    del out
