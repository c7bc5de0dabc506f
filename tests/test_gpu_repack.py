"""GPU parity of ft_repack_q4_0_soa, the one-time structure-of-arrays export
of Q4_0 weights (nibble bytes, then fp16 scales): bit for bit against the
oracle's repack, on a small layer, on weights only 2-byte aligned, on an odd
block count, and on the full 128-expert 1408 x 2816 prefill layer."""

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
    return ft


def _check(ft, oracle, w, dw=None):
    qs, d = ft.repack_q4_0_soa(G.dev(w) if dw is None else dw)
    rq, rd = oracle.repack_q4_0_soa(w)
    assert np.array_equal(G.host(qs), rq)
    assert np.array_equal(G.host(d).view(np.uint16), rd.view(np.uint16))


def test_repack_small(ft, oracle):
    _check(ft, oracle, G.weights_of("tiny"))


def test_repack_odd_count_and_2_byte_alignment(ft, oracle):
    import torch
    w = G.weights_of("tiny").reshape(-1, 18)[:1001]              # 1001 blocks
    buf = torch.empty(w.size + 2, dtype=torch.uint8, device="cuda")
    dw = buf[2:].view(1001, 18)
    dw.copy_(torch.from_numpy(np.ascontiguousarray(w)))
    assert dw.data_ptr() % 4 == 2
    _check(ft, oracle, w, dw)


def test_repack_full_prefill_layer(ft, oracle):
    _check(ft, oracle, G.weights_of("prefill"))
