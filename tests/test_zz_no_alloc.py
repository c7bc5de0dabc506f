"""ft_moe_route_offsets_noalloc: the router for callers that may not allocate
device memory (a serving runtime whose memory planner owns the whole GPU, a
plugin inside another framework's allocator, a loop that cannot take
cudaMalloc's implicit synchronization).  Its histogram scratch is a fixed
array inside the library, so the checks here are:

* its counts, offsets and permutation equal the CPU oracle's bit for bit and
  those of the allocating entry point ft_moe_route_offsets;
* two calls in a row share the array: the second one (a different expert
  count, more than 32 chunks of 256 slots, so the three-kernel route that
  keeps its histogram in the array runs) sees nothing left from the first,
  and a batch that needs exactly the array's 2^18 words runs;
* bad expert ids are left out of the routing, with or without an error word
  (without one the flag goes to the array's own tail word);
* a problem one chunk larger than the array is turned away with
  FT_ERR_SIZE before anything runs.

The file name makes pytest collect it last; it builds and loads the library
itself, so it also passes alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SCRATCH_WORDS = 1 << 18
CHUNK = 256


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_quantize_gb300 import _lib, build
    build.build()
    return _lib.load()


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.get()


def _route_noalloc(lib, ids, n_experts, with_err=True):
    import torch
    T, k = ids.shape
    counts = torch.full((n_experts,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((n_experts + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.ft_moe_route_offsets_noalloc(
        ctypes.c_void_p(ids.data_ptr()), T, k, n_experts, ctypes.c_void_p(counts.data_ptr()),
        ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(perm.data_ptr()),
        ctypes.c_void_p(err.data_ptr() if with_err else 0), stream)
    assert st == 0, lib.ft_last_error().decode()
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy(), int(err.item())


def _route_alloc(ids, n_experts):
    import bit_quantized_moe_quantize_gb300 as ft
    c, o, p = ft.route_offsets(ids, n_experts)
    return c.cpu().numpy(), o.cpu().numpy(), p.cpu().numpy()


def _uniform_ids(T, k, E, seed):
    rng = np.random.default_rng(seed)
    return np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)


def _check(lib, orc, ids_np, E, with_err=True):
    import torch
    ids = torch.from_numpy(ids_np).cuda()
    c, o, p, err = _route_noalloc(lib, ids, E, with_err)
    oc, oo, op, obad = orc.route(ids_np, E)
    assert np.array_equal(c, oc)
    assert np.array_equal(o, oo)
    assert np.array_equal(p, op)
    rc, ro, rp = _route_alloc(ids, E)
    assert np.array_equal(c, rc) and np.array_equal(o, ro) and np.array_equal(p, rp)
    import bit_quantized_moe_quantize_gb300 as ft
    ft.read_device_error()          # the allocating router flags bad ids in the library's own word
    return err, obad


def test_matches_the_oracle_on_two_calls_in_a_row(lib, orc):
    from bit_quantized_moe_quantize_gb300 import synth
    # first call: the prefill batch (65528 slots, 128 experts: 256 chunks, an
    # eighth of the array); second call: 8192 tokens of top-8 over 1024
    # experts, 65536 slots = 256 chunks x 1024 experts = exactly the array's
    # 2^18 words, so the second histogram covers and overwrites the first
    wl = synth.WORKLOADS["prefill"]
    err, bad = _check(lib, orc, synth.make_topk_ids(wl, 8191), wl.n_experts)
    assert err == 0 and bad == 0
    ids = _uniform_ids(8192, 8, 1024, 5)
    assert (ids.size + CHUNK - 1) // CHUNK * 1024 == SCRATCH_WORDS
    err, bad = _check(lib, orc, ids, 1024)
    assert err == 0 and bad == 0


def test_skewed_batch_after_a_full_one(lib, orc):
    from bit_quantized_moe_quantize_gb300 import synth
    wl = synth.WORKLOADS["qwen3_30b_a3b"]
    err, bad = _check(lib, orc, synth.make_topk_ids(wl, 8192), wl.n_experts)   # Zipf, 256 chunks
    assert err == 0 and bad == 0
    err, bad = _check(lib, orc, synth.make_topk_ids(wl, 512), wl.n_experts)    # one-launch route
    assert err == 0 and bad == 0


@pytest.mark.parametrize("with_err", [True, False])
def test_bad_ids_left_out(lib, orc, with_err):
    ids = _uniform_ids(3000, 4, 64, 6)
    ids[5, 1] = -1
    ids[77, 0] = 64
    ids[2999, 3] = 1 << 30
    err, bad = _check(lib, orc, ids, 64, with_err)
    assert bad == 3
    if with_err:
        assert err == 1                                  # FT_DEVERR_BAD_EXPERT_ID
    else:
        assert err == 0                                  # the caller's word was not passed


def test_rejects_problems_larger_than_the_scratch(lib):
    vp = ctypes.c_void_p
    # 65537 slots over 1024 experts: 257 chunks x 1024 words, one chunk over
    st = lib.ft_moe_route_offsets_noalloc(vp(0x1000), 65537, 1, 1024, vp(0x2000), vp(0x3000), vp(0x4000),
                                          vp(0), vp(0))
    assert st == 2
    assert "scratch" in lib.ft_last_error().decode()
    # 2^20 slots over 4096 experts: far over
    st = lib.ft_moe_route_offsets_noalloc(vp(0x1000), 1 << 17, 8, 4096, vp(0x2000), vp(0x3000), vp(0x4000),
                                          vp(0), vp(0))
    assert st == 2
