"""Values the pages print, stored under tests/golden/ with their citations:
the batch sizes at the 65535 grid.z launch cap, and the T4 kernel-time table
the benchmark quotes as context.  CPU only."""

import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [line.rstrip("\n").split("\t") for line in f if line.strip() and not line.startswith("#")]


def test_launch_limit_batches():
    """Each printed batch: slots = tokens * top_k, on the stated side of 65535,
    and the library's host checks accept it (tokens * top_k < 2^31; no size
    product is bounded by a grid dimension)."""
    from bit_quantized_moe_quantize_gb300 import _lib, build
    build.build()
    L = _lib.load()
    rows = _rows("launch_limits.tsv")
    assert len(rows) == 5
    for tokens, top_k, slots, past, source in rows:
        t, k, s = int(tokens), int(top_k), int(slots)
        assert t * k == s, source
        assert (s > 65535) == (past == "yes"), source
        # the prefill layer's shape (N 1408, K 2816) with enough experts for top_k
        assert L.ft_moe_workspace_bytes(t, k, max(8, k), 1408, 2816) > 0, source


def test_t4_table_is_what_the_benchmark_quotes():
    import bench
    rows = _rows("t4_moe_vec_timings.tsv")
    assert [int(r[0]) for r in rows] == [2048, 4096, 8191]
    for tokens, _m1, _m2, p1, _p2 in rows:
        # bench.py's context figure: routed tokens/s of the patched kernel's first run
        assert bench.PAGES_T4_TOKENS_PER_S[("prefill", int(tokens))] == int(tokens) / (float(p1) / 1000.0)
