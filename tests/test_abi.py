"""The C-ABI library loads on a host without a GPU, exports every symbol
include/ft_moe.h declares, and rejects bad arguments on the host before any
CUDA call (CPU only: nothing here launches a kernel)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_moe_quantize_gb300 import _lib, build
    build.build()
    return _lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "ft_moe.h")).read()
    return re.findall(r"FT_API\s+[\w\s\*]+?\b(ft_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(header_functions())
    for required in ("ft_quantize_q8_1", "ft_moe_route_offsets", "ft_moe_q4_0_q8_1"):
        assert required in names


def test_exports_every_declared_symbol(lib):
    from bit_quantized_moe_quantize_gb300 import _lib
    names = header_functions()
    assert names
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib.EXPORTS)


def test_library_is_native_and_current(lib):
    from bit_quantized_moe_quantize_gb300 import build
    assert build.is_current()
    assert lib.ft_abi_version() == 1
    with open(build.LIB, "rb") as f:
        assert f.read(4) == b"\x7fELF"


def test_no_load_time_cuda_dependency():
    """The library links the CUDA runtime statically and reaches the driver
    lazily, so it loads on machines without a GPU driver."""
    from bit_quantized_moe_quantize_gb300 import build
    ctypes.CDLL(build.LIB)   # would raise if libcuda.so.1 were a load-time need


def _err(lib):
    return lib.ft_last_error().decode()


def test_quantize_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    assert lib.ft_quantize_q8_1(vp(0), vp(0), -1, 32, vp(0)) == 1
    assert lib.ft_quantize_q8_1(vp(0), vp(0), 4, 33, vp(0)) == 1
    assert "multiple of 32" in _err(lib)
    assert lib.ft_quantize_q8_1(vp(0), vp(0), 4, 0, vp(0)) == 1
    assert lib.ft_quantize_q8_1(vp(0), vp(0), 0, 64, vp(0)) == 0          # empty batch: no-op
    assert lib.ft_quantize_q8_1(vp(0), vp(0), 4, 64, vp(0)) == 1          # null pointers
    assert lib.ft_quantize_q8_1(vp(0x1002), vp(0x2000), 4, 64, vp(0)) == 3   # misaligned x
    assert lib.ft_quantize_q8_1(vp(0), vp(0), 1 << 62, 64, vp(0)) == 2    # size overflow


def test_route_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.ft_moe_route_offsets
    assert f(vp(0), 4, 0, 8, vp(0), vp(0), vp(0), vp(0), vp(0)) == 1      # top_k 0
    assert f(vp(0), 4, 9, 8, vp(0), vp(0), vp(0), vp(0), vp(0)) == 1      # top_k > E
    assert f(vp(0), 4, 2, 0, vp(0), vp(0), vp(0), vp(0), vp(0)) == 1      # no experts
    assert f(vp(0), 4, 2, 5000, vp(0), vp(0), vp(0), vp(0), vp(0)) == 1   # > FT_MAX_EXPERTS
    assert f(vp(0), 1 << 30, 8, 8, vp(0), vp(0), vp(0), vp(0), vp(0)) == 2   # slots >= 2^31
    assert "2^31" in _err(lib)
    assert f(vp(0), 4, 2, 8, vp(0), vp(0), vp(0), vp(0), vp(0)) == 1      # null pointers
    assert f(vp(0x1001), 4, 2, 8, vp(0x2000), vp(0x3000), vp(0x4000), vp(0), vp(0)) == 3


def test_matmul_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.ft_moe_q4_0_q8_1
    W, A, I, O = vp(0x10000), vp(0x20000), vp(0x30000), vp(0x40000)
    assert f(W, A, I, O, 4, 2, 8, 128, 100, vp(0)) == 1        # ncols % 32
    assert f(W, A, I, O, 4, 2, 8, 0, 256, vp(0)) == 1          # nrows
    assert f(W, A, I, O, 4, 2, 8, 128, 1 << 20, vp(0)) == 2    # ncols over the limit
    assert f(W, A, I, O, 4, 2, 4096, 1 << 20, 256, vp(0)) == 2  # E*N >= 2^31
    assert f(W, A, I, O, 0, 2, 8, 128, 256, vp(0)) == 0        # no slots: no-op
    assert f(vp(0), A, I, O, 4, 2, 8, 128, 256, vp(0)) == 1    # null weights
    assert f(W, A, I, vp(0), 4, 2, 8, 128, 256, vp(0)) == 1    # null out
    assert f(vp(0x10008), A, I, O, 4, 2, 8, 128, 256, vp(0)) == 3   # weights not 16-byte aligned
    assert f(W, A, vp(0x30002), O, 4, 2, 8, 128, 256, vp(0)) == 3   # ids misaligned
    d = lib.ft_moe_block_dots
    assert d(W, A, I, vp(0), 4, 2, 8, 128, 256, vp(0)) == 1
    assert d(W, A, I, O, 1 << 20, 8, 8, 4096, 4096, vp(0)) == 2     # dots > 2^31 elements


def test_workspace_and_path_selection(lib):
    ws = lib.ft_moe_workspace_bytes
    small = ws(16, 2, 8, 128, 256)
    big = ws(8192, 8, 128, 1408, 2816)
    assert 0 < small < big
    assert big >= 8192 * 8 * 4              # holds the permutation
    assert ws(16, 2, 8, 128, 100) == 0      # invalid shape
    prev = lib.ft_moe_set_path(0)
    try:
        sel = lib.ft_moe_selected_path
        assert sel(1, 8, 128, 768, 2048) == 1            # decode: GEMV
        assert sel(8191, 8, 128, 1408, 2816) == 2        # prefill: tensor cores
        assert sel(8191, 8, 128, 1408, 2816 + 32) == 1   # ncols % 256 != 0: GEMV only
        # 32 routed slots per expert: the GEMV's 16-slot mma.sync tiles; 48: tensor cores
        assert sel(512, 8, 128, 768, 2048) == 1 and sel(768, 8, 128, 768, 2048) == 2
        gsel = lib.ft_moe_gguf_selected_path
        assert gsel(12, 8191, 8, 128, 1408, 2816) == 2   # Q4_K: tensor cores
        assert gsel(14, 8191, 8, 128, 1408, 2816) == 1   # Q6_K: GEMV only
        assert gsel(12, 512, 8, 128, 768, 2048) == 1     # Q4_K, 32 slots per expert: mma.sync tiles
        assert gsel(99, 1, 8, 128, 768, 2048) == -1      # unknown type
        assert gsel(12, 1, 8, 128, 768, 2816 + 32) == -1  # not whole super-blocks
        assert lib.ft_moe_set_path(3) == 0               # the GEMV path on the dp4a kernels, forced
        assert sel(512, 8, 128, 768, 2048) == 1 and sel(8191, 8, 128, 1408, 2816) == 1
        assert lib.ft_moe_set_path(2) == 3
        assert sel(1, 8, 128, 768, 2048) == 2
        assert lib.ft_moe_set_path(7) == -1
        assert sel(1, 8, 128, 768, 100) == -1
    finally:
        lib.ft_moe_set_path(prev if prev >= 0 else 0)


def test_last_error_is_per_call(lib):
    vp = ctypes.c_void_p
    assert lib.ft_quantize_q8_1(vp(0), vp(0), 4, 33, vp(0)) == 1
    assert _err(lib)
    assert lib.ft_quantize_q8_1(vp(0), vp(0), 0, 64, vp(0)) == 0
    assert _err(lib) == ""


def test_product_path_never_imports_the_oracle():
    """The CUDA binding and the benchmark's GPU leg must not reach the oracle."""
    pkg = os.path.join(ROOT, "bit_quantized_moe_quantize_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn
    for fn in os.listdir(os.path.join(pkg, "csrc")):
        src = open(os.path.join(pkg, "csrc", fn)).read()
        assert "ft_oracle" not in src and "oracle_" not in src, fn


def test_activation_and_ffn_reject_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.ft_act_mul_quantize_q8_1
    H, A = vp(0x10000), vp(0x20000)
    assert f(H, A, -1, 64, 0, vp(0)) == 1                     # rows < 0
    assert f(H, A, 4, 48, 0, vp(0)) == 1                      # n_inter % 32
    assert f(H, A, 4, 64, 2, vp(0)) == 1                      # unknown activation
    assert "act_kind" in _err(lib)
    assert f(H, A, 0, 64, 1, vp(0)) == 0                      # no rows: no-op
    assert f(vp(0), A, 4, 64, 0, vp(0)) == 1                  # null h
    assert f(vp(0x10008), A, 4, 64, 0, vp(0)) == 3            # h not 16-byte aligned
    assert f(H, vp(0x20002), 4, 64, 0, vp(0)) == 3            # act not 4-byte aligned
    assert f(H, A, 1 << 60, 64, 0, vp(0)) == 2                # size overflow
    g = lib.ft_moe_ffn_q4_0_q8_1
    W1, W2, X, I, Hh, M, O = (vp(0x10000 * i) for i in range(1, 8))
    assert g(W1, W2, X, I, Hh, M, O, 4, 2, 8, 256, 100, 0, vp(0)) == 1  # n_inter % 32
    assert g(W1, W2, X, I, Hh, M, O, 4, 2, 8, 250, 128, 0, vp(0)) == 1  # hidden % 32
    assert g(W1, W2, X, I, Hh, M, O, 4, 2, 8, 256, 128, 5, vp(0)) == 1  # unknown activation
    assert g(W1, W2, X, I, Hh, M, O, 0, 2, 8, 256, 128, 0, vp(0)) == 0  # no slots: no-op
    assert g(W1, W2, X, I, Hh, vp(0), O, 4, 2, 8, 256, 128, 0, vp(0)) == 1   # null act_mid
    assert g(W1, W2, X, I, vp(0), M, vp(0), 4, 2, 8, 256, 128, 0, vp(0)) == 1  # null out (h NULL: fused)
    assert g(W1, W2, X, I, vp(0x50008), M, O, 4, 2, 8, 256, 128, 0, vp(0)) == 3   # h misaligned
    assert g(W1, W2, X, I, Hh, vp(0x60004), O, 4, 2, 8, 256, 128, 0, vp(0)) == 3  # act_mid misaligned


def test_fused_layer1_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.ft_moe_q4_0_q8_1_act
    W, X, I, M = (vp(0x10000 * i) for i in range(1, 5))
    assert f(W, X, I, M, 4, 2, 8, 100, 256, 0, vp(0)) == 1       # n_inter % 32
    assert f(W, X, I, M, 4, 2, 8, 0, 256, 0, vp(0)) == 1         # n_inter = 0
    assert f(W, X, I, M, 4, 2, 8, 128, 250, 0, vp(0)) == 1       # hidden % 32
    assert f(W, X, I, M, 4, 2, 8, 128, 256, 7, vp(0)) == 1       # unknown activation
    assert "act_kind" in _err(lib)
    assert f(W, X, I, M, 4, 9, 8, 128, 256, 0, vp(0)) == 1       # top_k > n_experts
    assert f(W, X, I, M, 0, 2, 8, 128, 256, 0, vp(0)) == 0       # no slots: no-op
    assert f(W, X, I, vp(0), 4, 2, 8, 128, 256, 0, vp(0)) == 1   # null act_mid
    assert f(vp(0x10008), X, I, M, 4, 2, 8, 128, 256, 0, vp(0)) == 3   # w13 misaligned
    assert f(W, X, I, vp(0x40002), 4, 2, 8, 128, 256, 0, vp(0)) == 3   # act_mid not 4-byte aligned
    assert f(W, X, I, M, 1 << 40, 8, 8, 128, 256, 0, vp(0)) == 2       # tokens * top_k >= 2^31
    r = lib.ft_moe_ffn_reserve
    assert r(16, 2, 8, 256, 0) == 1                                # n_inter = 0
    assert r(16, 2, 8, 250, 128) == 1                              # hidden % 32
    assert r(16, 9, 8, 256, 128) == 1                              # top_k > n_experts


def test_gguf_matmul_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.ft_moe_gguf_q8_1
    W, A, I, O = vp(0x10000), vp(0x20000), vp(0x30000), vp(0x40000)
    assert f(5, W, A, I, O, 4, 2, 8, 128, 256, vp(0)) == 1       # unknown type
    assert "weight type" in _err(lib)
    assert f(0, W, A, I, O, 4, 2, 8, 128, 256, vp(0)) == 1       # unknown type
    assert f(8, W, A, I, O, 4, 2, 8, 128, 100, vp(0)) == 1       # ncols % 32
    assert f(3, W, A, I, O, 0, 2, 8, 128, 256, vp(0)) == 0       # no slots: no-op
    assert f(6, W, A, I, vp(0), 4, 2, 8, 128, 256, vp(0)) == 1   # null out
    assert f(7, vp(0x10008), A, I, O, 4, 2, 8, 128, 256, vp(0)) == 3   # weights misaligned
    assert f(12, W, A, I, O, 4, 2, 8, 128, 160, vp(0)) == 1      # Q4_K: ncols % 256
    assert "ncols % 256" in _err(lib)
    assert f(13, W, A, I, O, 4, 2, 8, 128, 288, vp(0)) == 1      # Q5_K: ncols % 256


def test_repack_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.ft_repack_q4_0_soa
    W, Q, D = vp(0x10000), vp(0x20000), vp(0x30000)
    assert f(W, Q, D, -1, vp(0)) == 1                          # n_blocks < 0
    assert f(W, Q, D, 0, vp(0)) == 0                           # no blocks: no-op
    assert f(vp(0), Q, D, 4, vp(0)) == 1                       # null weights
    assert f(W, vp(0x20008), D, 4, vp(0)) == 3                 # qs not 16-byte aligned
    assert f(vp(0x10001), Q, D, 4, vp(0)) == 3                 # weights odd
    assert f(W, Q, D, 1 << 62, vp(0)) == 2                     # size overflow


def test_debug_stream_read_rejects_bad_arguments_on_the_host(lib):
    vp = ctypes.c_void_p
    f = lib.ft_debug_stream_read
    assert f(vp(0x10000), 100, vp(0)) == 1          # not a multiple of 16
    assert f(vp(0x10000), -16, vp(0)) == 1          # negative
    assert f(vp(0x10000), 0, vp(0)) == 0            # nothing to read: no-op
    assert f(vp(0), 64, vp(0)) == 1                 # null buffer
    assert f(vp(0x10008), 64, vp(0)) == 3           # not 16-byte aligned


def test_debug_wait_timeout_rejects_bad_limits_on_the_host(lib):
    vp = ctypes.c_void_p
    for bad in (0, 999, 2_000_000_000):
        assert lib.ft_debug_wait_timeout(bad, vp(0)) == 1
    assert "limit_ns" in _err(lib)


@pytest.mark.parametrize("value,code", [("gemv", 1), ("gemm", 2), ("gemv_dp4a", 3), ("auto", 0), ("bogus", 0)])
def test_path_environment_variable(lib, value, code):
    """FT_MOE_PATH sets the initial path setting (read once, at the first
    use, in a fresh process): ft_moe_set_path returns it as the previous one."""
    import subprocess
    import sys
    prog = ("import ctypes, sys; from bit_quantized_moe_quantize_gb300 import _lib; "
            "L = _lib.load(); sys.stdout.write(str(L.ft_moe_set_path(0)))")
    env = dict(os.environ, FT_MOE_PATH=value)
    got = subprocess.run([sys.executable, "-c", prog], env=env, cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert got.returncode == 0, got.stderr
    assert got.stdout.strip() == str(code)
