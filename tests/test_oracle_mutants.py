"""The oracle's pins catch plausible mistakes.

Each case plants one slip in a copy of the oracle's C source (on the CPU,
never in the CUDA library), builds it, and runs the pin suite against it. At
least one pin must fail for every mutant; an uncaught mutant means the pins
leave that part of the oracle unchecked. Every mutant keeps all memory
accesses in bounds.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import synth
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "ds4moe_oracle.c")

MUTANTS = {
    "scale_min_nibbles_swapped": [("int sc = scales[j] & 15;", "int sc = scales[j] >> 4;"),
                                  ("int m = scales[j] >> 4;", "int m = scales[j] & 15;")],
    "codes_msb_first": [("(qs[i / 4] >> (2 * (i % 4))) & 3", "(qs[i / 4] >> (6 - 2 * (i % 4))) & 3")],
    "d_dmin_swapped": [("oracle_f16(le16(blk + 80))", "oracle_f16(le16(blk + 82x))"),
                       ("oracle_f16(le16(blk + 82))", "oracle_f16(le16(blk + 80))"),
                       ("blk + 82x", "blk + 82")],
    "min_added": [("w[i] = d * sc * q - dmin * m;", "w[i] = d * sc * q + dmin * m;")],
    "min_dropped": [("w[i] = d * sc * q - dmin * m;", "w[i] = d * sc * q;")],
    "block_order_reversed": [("oracle_dequant_q2(row + b * Q2_BYTES, w + b * 256);",
                              "oracle_dequant_q2(row + b * Q2_BYTES, w + (k / 256 - 1 - b) * 256);")],
    "q8_unsigned": [("w[i] = d * (double)(int8_t)blk[2 + i];", "w[i] = d * (double)blk[2 + i];")],
    "f16_exponent_bias": [("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);")],
    "bf16_no_hidden_bit": [("v = ldexp((double)(128 + m), e - 134);", "v = ldexp((double)m, e - 134);")],
    "silu_sign": [("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));")],
    "sigmoid_is_exp": [("return 1.0 / (1.0 + exp(-z));", "return exp(z);")],
    "router_transposed": [("L += xt[h] * (double)router_w[(int64_t)e * H + h];",
                           "L += xt[h] * (double)router_w[(int64_t)h * E + e];")],
    "ties_prefer_higher_index": [("return (a->e > b->e) - (a->e < b->e);", "return (a->e < b->e) - (a->e > b->e);")],
    "nan_ranked_first": [("if (a_nan != b_nan) return a_nan - b_nan;", "if (a_nan != b_nan) return b_nan - a_nan;")],
    "ascending_selection": [("if (a->sel > b->sel) return -1;", "if (a->sel > b->sel) return 1;"),
                            ("if (a->sel < b->sel) return 1;", "if (a->sel < b->sel) return -1;")],
    "bias_in_weights": [("total += score[order[k].e];", "total += (double)order[k].sel;"),
                        ("weights[(int64_t)t * K + k] = total > 0.0 ? score[order[k].e] / total : 1.0 / K;",
                         "weights[(int64_t)t * K + k] = total > 0.0 ? (double)order[k].sel / total : 1.0 / K;")],
    "no_renormalisation": [("score[order[k].e] / total : 1.0 / K;", "score[order[k].e] : 1.0 / K;")],
    "gate_up_exchanged": [("h[i] = oracle_silu(g) * u;\n        }\n#pragma omp for schedule(static)\n"
                           "        for (int j = 0; j < H; j++) {\n            oracle_dequant_q2_row",
                           "h[i] = oracle_silu(u) * g;\n        }\n#pragma omp for schedule(static)\n"
                           "        for (int j = 0; j < H; j++) {\n            oracle_dequant_q2_row")],
    "routing_weight_dropped": [("acc[j0 + i] += wk * (s1[i] * s2[i] * ye[j0 + i]);",
                                "acc[j0 + i] += (s1[i] * s2[i] * ye[j0 + i]);")],
    "gain_nibble_high_first": [("s[i] = 1.0 + X * oracle_e2m1((uint8_t)((blk[i / 2] >> (4 * (i % 2))) & 15));",
                                "s[i] = 1.0 + X * oracle_e2m1((uint8_t)((blk[i / 2] >> (4 - 4 * (i % 2))) & 15));")],
    "gain_stores_s_not_s_minus_1": [("s[i] = 1.0 + X * oracle_e2m1", "s[i] = X * oracle_e2m1")],
    "gain_tables_added": [("s1[i] * s2[i] * ye[j0 + i]", "(s1[i] + s2[i] - 1.0) * ye[j0 + i]")],
    "gain_second_table_ignored": [("s1[i] * s2[i] * ye[j0 + i]", "s1[i] * ye[j0 + i]")],
    "gain_indexed_by_slot": [("gain1 + ((int64_t)e * (H / 32)", "gain1 + ((int64_t)k * (H / 32)")],
    "e2m1_exponent_bias": [("ldexp(1.0 + 0.5 * man, ex - 1)", "ldexp(1.0 + 0.5 * man, ex - 2)")],
    "e2m1_no_subnormal": [("ex == 0 ? 0.5 * man :", "ex == 0 ? 0.0 :")],
    "e8m0_bias": [("ldexp(1.0, (int)x - 127)", "ldexp(1.0, (int)x - 128)")],
    "mx4_nibble_high_first": [("w[i] = X * oracle_e2m1((uint8_t)((blk[i / 2] >> (4 * (i % 2))) & 15));",
                               "w[i] = X * oracle_e2m1((uint8_t)((blk[i / 2] >> (4 - 4 * (i % 2))) & 15));")],
    "mx4_scale_ignored": [("w[i] = X * oracle_e2m1((uint8_t)", "w[i] = 1.0 * oracle_e2m1((uint8_t)")],
    "q8_truncates": [("q[b * 32 + i] = (int8_t)nearbyintf(r);", "q[b * 32 + i] = (int8_t)r;")],
    "q8_scale_128": [("const float db = amax / 127.0f;", "const float db = amax / 128.0f;")],
    "mx4_act_scale_off_by_one": [("sb = (e - 1) - 2 + 127;", "sb = (e - 1) - 1 + 127;")],
    "mx4_act_ties_to_odd": [("(dist == bd && c % 2 == 0)", "(dist == bd && c % 2 == 1)")],
    "mx4_act_sign_dropped": [("return (uint8_t)(best | (signbit(r) ? 8 : 0));", "return (uint8_t)best;")],
    "x_not_quantised": [("quantise_act(act, xt, H, a);", "quantise_act(ACT_EXACT, xt, H, a);")],
    "h_not_quantised": [("quantise_act(act, h, I, hq);", "quantise_act(ACT_EXACT, h, I, hq);")],
    "h_quantised_in_double": [("        f[i] = (float)v[i];", "        f[i] = (float)(v[i] * (1.0 + 1e-7));")],
    "vq_index_msb_first": [("v |= ((stream[bit / 8] >> (bit % 8)) & 1) << i;",
                            "v |= ((stream[bit / 8] >> (7 - bit % 8)) & 1) << i;")],
    "vq_plane_ignored": [("v |= ((plane[k / 8] >> (k % 8)) & 1) << 12;", "v |= 0;")],
    "vq_plane_bit_low": [("v |= ((plane[k / 8] >> (k % 8)) & 1) << 12;", "v ^= ((plane[k / 8] >> (k % 8)) & 1);")],
    "vq_row_gain_ignored": [("const double g = oracle_f16(gains[r]);", "const double g = 1.0;")],
    "e4m3_exponent_bias": [("ldexp(8.0 + man, ex - 10)", "ldexp(8.0 + man, ex - 11)")],
    "e4m3_subnormal_scale": [("ldexp((double)man, -9)", "ldexp((double)man, -10)")],
    "vq_codeword_reversed": [("w[8 * j + i] = g * oracle_e4m3(codebook[8 * n + i]);",
                              "w[8 * j + i] = g * oracle_e4m3(codebook[8 * n + 7 - i]);")],
    "vq_groups_reversed_in_row": [("oracle_vq_index(stream, plane, r * (k / 8) + j)",
                                   "oracle_vq_index(stream, plane, r * (k / 8) + (k / 8 - 1 - j))")],
    "vq_expert_stream_offset_dropped": [("m->stream + e * (n * 12 / 8)", "m->stream + 0 * (n * 12 / 8)")],
    "vq_expert_gains_offset_dropped": [("m->gains + e * rows", "m->gains")],
    "shared_dropped": [("acc[j] += ye[j];\n        }", "acc[j] += 0.0 * ye[j];\n        }")],
    "shared_weighted": [("acc[j] += ye[j];\n        }", "acc[j] += weights[(int64_t)t * K] * ye[j];\n        }")],
    "down_uses_gate_activation": [("ye[j] = dot(w, h, I);", "ye[j] = dot(w, xt, I);")],
}


def _pin_functions(tiny):
    """(name, callable) for every pin in the pin suite."""
    out = []
    for name in dir(pins):
        if not name.startswith("test_"):
            continue
        fn = getattr(pins, name)
        if name in ("test_q2_golden_blocks",):
            out += [(f"{name}[{c}]", (lambda c=c, fn=fn: fn(c))) for c in pins.Q2_CLOSED]
        elif name in ("test_q8_golden_blocks",):
            out += [(f"{name}[{c}]", (lambda c=c, fn=fn: fn(c))) for c in pins.Q8_CLOSED]
        elif name == "test_vq_layer_matches_dense_numpy":
            out += [(f"{name}[{b}]", (lambda b=b, fn=fn: fn(b))) for b in (12, 13)]
        elif fn.__code__.co_argcount == 1:
            out.append((name, (lambda fn=fn: fn(tiny))))
        else:
            out.append((name, fn))
    return out


@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    return wl.shape, synth.make_layer(wl.shape, wl.layer_seeds[0]), synth.make_tokens("tiny")


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


def _build_mutant(src, subs, path):
    for old, new in subs:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new, 1)
    cpath = path + ".c"
    with open(cpath, "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
                           "-o", path, cpath, "-lm"])


def test_unmutated_oracle_passes_every_pin(tiny):
    for name, fn in _pin_functions(tiny):
        fn()


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant, tiny, workdir):
    src = open(SRC).read()
    lib = os.path.join(workdir, f"lib_{mutant}.so")
    _build_mutant(src, MUTANTS[mutant], lib)
    failed = []
    with oracle.using_library(lib), np.errstate(all="ignore"):
        for name, fn in _pin_functions(tiny):
            try:
                fn()
            except (AssertionError, ValueError):
                failed.append(name)
                break
    assert failed, f"no pin catches mutant {mutant}"
