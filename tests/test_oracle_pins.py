"""The CPU oracle against its pins, and mutated oracles against the same pins.

CPU only.  The mutation half copies ``oracle/ft_oracle.c``, plants one
plausible mistake in the copy, builds it in a temporary directory and runs
every pin on it in a fresh process: at least one pin must fail.  The committed
oracle is never modified.
"""

import multiprocessing as mp
import os
import shutil

import numpy as np
import pytest

import pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle, pin):
    pin(oracle)


def test_workload_quantized_through_oracle(oracle):
    """The tiny-layer workload goes through the oracle end to end; the result is
    finite, has the documented shape and its zero pattern matches the routing."""
    from bit_quantized_moe_quantize_gb300 import synth
    case = synth.make_case("tiny", 16)
    act = oracle.quantize_q8_1(case["x"])
    y = oracle.moe(case["weights"], act, case["topk_ids"])
    assert y.shape == (16, 2, 128) and np.isfinite(y).all()
    assert np.abs(y).max() > 0


MUTANTS = {
    "q4_nibble_order_quantizer": ("(q[j] | (q[j + 16] << 4))", "(q[j + 16] | (q[j] << 4))"),
    "q4_nibble_order_decode": ("return i < 16 ? (qs[i] & 0x0f) : (qs[i - 16] >> 4);",
                               "return i < 16 ? (qs[i] >> 4) : (qs[i - 16] & 0x0f);"),
    "q4_offset_7": ("(q4_0_nibble(w_block, i) - 8)", "(q4_0_nibble(w_block, i) - 7)"),
    "q4_scale_sign": ("float d = m / -8.0f;", "float d = m / 8.0f;"),
    "token_index_mod": ("int64_t t = s / top_k;", "int64_t t = s % top_k;"),
    "q8_truncate": ("q = (int)roundf(x[i] / d);", "q = (int)(x[i] / d);"),
    "q8_scale_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "q8_s_from_fp16_d": ("float s = d * (float)sum;",
                         "float s = (float)oracle_half_to_double(oracle_float_to_half(d)) * (float)sum;"),
    "dot_drops_act_scale": ("y += dw * da * (double)oracle_block_dot(wb, ab);",
                            "y += dw * (double)oracle_block_dot(wb, ab);"),
    "route_unstable": ("perm[offsets[e] + cursor[e]] = (int32_t)s;",
                       "perm[offsets[e] + counts[e] - 1 - cursor[e]] = (int32_t)s;"),
    "fp16_truncates": ("double q = nearbyint(m * 2048.0);", "double q = floor(m * 2048.0);"),
    "silu_sign": ("return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    "gelu_drops_cubic": ("(g + 0.044715 * g * g * g)", "(g)"),
    "gelu_drops_factor_2": ("return g / (1.0 + exp(-2.0 * y));", "return g / (1.0 + exp(-y));"),
    "gelu_tanh_form": ("return g / (1.0 + exp(-2.0 * y));", "return 0.5 * g * (1.0 + tanh(y));"),
    "gate_up_swapped": ("(act_fn((double)hr[i], kind) * (double)hr[n_inter + i])",
                        "(act_fn((double)hr[n_inter + i], kind) * (double)hr[i])"),
    "act_kind_swapped": ("if (kind == ORACLE_ACT_SILU)", "if (kind != ORACLE_ACT_SILU)"),
    "q5_high_bit_index": ("hi5 = (int)((qh >> i) & 1u);", "hi5 = (int)((qh >> (i % 16)) & 1u);"),
    "q5_0_offset_15": ("(type == ORACLE_GGUF_Q5_0 ? 16 : 0)", "(type == ORACLE_GGUF_Q5_0 ? 15 : 0)"),
    "gguf_offset_term_dropped": (" +\n                         gguf_offset(wb, type) * da * (double)suma;", ";"),
    "gguf_offset_uses_stored_s": ("gguf_offset(wb, type) * da * (double)suma;",
                                  "gguf_offset(wb, type) * oracle_half_to_double(rd16(ab + 2));"),
    "q8_0_unsigned": ("return (int)(int8_t)blk[2 + i];", "return (int)blk[2 + i];"),
    "q4_1_m_read_as_d": ("return oracle_half_to_double(rd16(blk + 2));", "return oracle_half_to_double(rd16(blk));"),
    "q4_1_nibble_order": ("return i < 16 ? (blk[4 + i] & 0x0f) : (blk[4 + i - 16] >> 4);",
                          "return i < 16 ? (blk[4 + i] >> 4) : (blk[4 + i - 16] & 0x0f);"),
    "kquant_scale_high_bits": ("*sc = (sc12[j + 4] & 0x0f) | ((sc12[j - 4] >> 6) << 4);",
                               "*sc = (sc12[j + 4] & 0x0f) | ((sc12[j] >> 6) << 4);"),
    "kquant_min_sign": ("- dmn * da * (double)suma;", "+ dmn * da * (double)suma;"),
    "kquant_nibble_half": ("lev[l] = (j % 2 == 0) ? (qs[l] & 0x0f) : (qs[l] >> 4);",
                           "lev[l] = (j % 2 == 0) ? (qs[l] >> 4) : (qs[l] & 0x0f);"),
    "q5k_bit_index": ("lev[l] |= ((sb[16 + l] >> j) & 1) << 4;", "lev[l] |= ((sb[16 + l] >> (j / 2)) & 1) << 4;"),
    "q6k_offset_31": ("lev[l] = (lo4 | (hi2 << 4)) - 32;", "lev[l] = (lo4 | (hi2 << 4)) - 31;"),
    "q6k_high_bits": ("const int hi2 = (sb[128 + 32 * h + l] >> (2 * k)) & 3;",
                      "const int hi2 = (sb[128 + 32 * h + l] >> k) & 3;"),
    "q6k_scale_group": ("if (l < 16) dlo_i += lev[l] * (int32_t)(int8_t)ab6[4 + l];",
                        "if (l < 15) dlo_i += lev[l] * (int32_t)(int8_t)ab6[4 + l];"),
    "repack_skips_wrong_bytes": ("memcpy(qs + b * 16, blocks + b * Q4_0_BYTES + 2, 16);",
                                 "memcpy(qs + b * 16, blocks + b * Q4_0_BYTES + 1, 16);"),
    "q3k_third_bit_index": ("v = (v | (((sb[l] >> j) & 1) << 2)) - 4;", "v = (v | (((sb[l] >> k) & 1) << 2)) - 4;"),
    "q3k_scale_top_bits": ("const int top2 = (sc[8 + g % 4] >> (2 * (g / 4))) & 3;",
                           "const int top2 = (sc[8 + g / 4] >> (2 * (g % 4))) & 3;"),
    "q2k_min_from_scale": ("*m_lo = dmin * (sb[2 * j] >> 4);", "*m_lo = dmin * (sb[2 * j] & 0x0f);"),
    "q2k_group_split": ("if (l < 16) {\n                                dot_lo", "if (l < 8) {\n                                dot_lo"),
    "bad_id_not_zeroed": ("    if (e < 0 || e >= n_experts)\n        return 0.0;\n",
                          "    if (e < 0 || e >= n_experts)\n        e = 0;\n"),
}


def _run_pins_on(so_path, q):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle as oracle_pkg
    import pins as pins_mod
    o = oracle_pkg.Oracle(so_path)
    failed = []
    for pin in pins_mod.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
        except Exception as exc:  # a mutant that misbehaves otherwise also counts as caught
            failed.append(f"{pin.__name__}:{type(exc).__name__}")
    q.put(failed)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    import oracle as oracle_pkg
    src = os.path.join(ROOT, "oracle", "ft_oracle.c")
    text = open(src).read()
    old, new = MUTANTS[name]
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    mut = tmp_path / "ft_oracle.c"
    mut.write_text(text.replace(old, new))
    shutil.copy(os.path.join(ROOT, "oracle", "ft_oracle.h"), tmp_path / "ft_oracle.h")
    so = oracle_pkg.build(src=str(mut), out_dir=str(tmp_path))
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_run_pins_on, args=(so, q))
    p.start()
    p.join(300)
    if p.is_alive():
        p.kill()
        pytest.fail(f"mutant {name} hung")
    failed = q.get() if p.exitcode == 0 else [f"crashed({p.exitcode})"]
    assert failed, f"mutant {name} passed every pin"
