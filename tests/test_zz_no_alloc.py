"""ft_moe_route_offsets_noalloc: the router for callers that may not allocate
device memory (a serving runtime whose memory planner owns the whole GPU, a
plugin inside another framework's allocator, a loop that cannot take
cudaMalloc's implicit synchronization).  Its histogram scratch is a fixed
array inside the library, so the check here is that it returns exactly what
the allocating entry point ft_moe_route_offsets returns, on two calls in a
row that share that array, and that it turns away problems too large for it.

The file name makes pytest collect it last; it builds and loads the library
itself, so it also passes alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_quantize_gb300 import _lib, build
    build.build()
    return _lib.load()


def _route_noalloc(lib, ids, n_experts):
    import torch
    T, k = ids.shape
    counts = torch.full((n_experts,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((n_experts + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.ft_moe_route_offsets_noalloc(
        ctypes.c_void_p(ids.data_ptr()), T, k, n_experts, ctypes.c_void_p(counts.data_ptr()),
        ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(perm.data_ptr()), ctypes.c_void_p(err.data_ptr()),
        stream)
    assert st == 0, lib.ft_last_error().decode()
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy(), int(err.item())


def _route_alloc(ids, n_experts):
    import bit_quantized_moe_quantize_gb300 as ft
    c, o, p = ft.route_offsets(ids, n_experts)
    return c.cpu().numpy(), o.cpu().numpy(), p.cpu().numpy()


def test_matches_allocating_router_on_two_calls(lib):
    import torch
    from bit_quantized_moe_quantize_gb300 import synth
    # first call: a big prefill batch (65528 slots, 128 experts) fills most of
    # the shared scratch; second call: a skewed smaller batch that must not see
    # anything left over from the first
    cases = [(synth.WORKLOADS["prefill"], 8191), (synth.WORKLOADS["qwen3_30b_a3b"], 512)]
    for wl, T in cases:
        ids = torch.from_numpy(synth.make_topk_ids(wl, T)).cuda()
        c, o, p, err = _route_noalloc(lib, ids, wl.n_experts)
        rc, ro, rp = _route_alloc(ids, wl.n_experts)
        assert np.array_equal(c, rc)
        assert np.array_equal(o, ro)
        assert np.array_equal(p, rp)
        assert err == 0


def test_rejects_problems_larger_than_the_scratch(lib):
    vp = ctypes.c_void_p
    # 2^20 slots over 4096 experts would need 4096 * 4096 words
    st = lib.ft_moe_route_offsets_noalloc(vp(0x1000), 1 << 17, 8, 4096, vp(0x2000), vp(0x3000), vp(0x4000),
                                          vp(0), vp(0))
    assert st == 2
    assert "scratch" in lib.ft_last_error().decode()
