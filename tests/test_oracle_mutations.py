"""Planted mistakes in the oracle must be caught by its pins.

Each case copies tl_oracle.c, plants one plausible mistake (a wrong index, a
flipped sign, a dropped term, a wrong rounding), compiles the copy with the
same flags on the CPU, swaps it in, and runs the pins of test_oracle.py; at
least one pin must fail.  Every planted mistake keeps memory accesses in
bounds, so a mutant fails by value, never by crashing the test process.
"""
import os
import subprocess

import pytest

from oracle import build as obuild
from oracle import oracle as omod
from tests import test_oracle as T

MUTATIONS = {
    "lane_index": ("int lane = 4 * g + t;", "int lane = 4 * t + g;"),
    "word_index": ("int j = 2 * u + h;", "int j = 2 * h + u;"),
    "hi_lo_columns": ("*lo_bit = 2 * s + 16 * e;", "*lo_bit = 2 * s + 16 * (1 - e);"),
    "step_order": ("*lo_bit = 2 * s + 16 * e;", "*lo_bit = 2 * (7 - s) + 16 * e;"),
    "sign_map": ("return 1 - f;", "return f - 1;"),
    "padding_fill": ("P[i] = 0x55555555u;", "P[i] = 0u;"),
    "dropped_term": ("acc += (double)w[k] * (double)bf16_to_float(X[n * K + k]);",
                     "if (k) acc += (double)w[k] * (double)bf16_to_float(X[n * K + k]);"),
    "transposed_x": ("(double)bf16_to_float(X[n * K + k])", "(double)bf16_to_float(X[k * N + n])"),
    "wrong_scale_row": ("Y[n * M + m] = (float)(acc * (double)scale[m]);",
                        "Y[n * M + m] = (float)(acc * (double)scale[0]);"),
    "scale_rounded_early": ("Y[n * M + m] = (float)(acc * (double)scale[m]);",
                            "Y[n * M + m] = (float)acc * scale[m];"),
    "zero_point_sign": ("acc - (int64_t)z[n] * (int64_t)rowsum[m]",
                        "acc + (int64_t)z[n] * (int64_t)rowsum[m]"),
    "epilogue_drops_s": ("float t = (float)corrected * s[n];", "float t = (float)corrected;"),
    "zero_point_truncated": ("z = -128 - (int32_t)rintf(lo / s);", "z = -128 - (int32_t)(lo / s);"),
    "quant_step_256": ("s = (hi - lo) / 255.0f;", "s = (hi - lo) / 256.0f;"),
    "quant_clamp_low": ("if (r < -128.0f) r = -128.0f;", "if (r < -127.0f) r = -127.0f;"),
    "sym_divisor": ("s = (a == 0.0f) ? 1.0f : a / 127.0f;", "s = (a == 0.0f) ? 1.0f : a / 128.0f;"),
    "rowsum_dropped": ("for (int64_t k = 0; k < K; ++k) acc += oracle_weight(P, m, k, Kp, NULL);",
                       "for (int64_t k = 1; k < K; ++k) acc += oracle_weight(P, m, k, Kp, NULL);"),
    "quant_ties_away_asym": ("float r = rintf(bf16_to_float(x[k]) / s) + (float)z;",
                             "float r = roundf(bf16_to_float(x[k]) / s) + (float)z;"),
    "quant_ties_away_sym": ("float r = rintf(bf16_to_float(x[k]) / s);",
                            "float r = roundf(bf16_to_float(x[k]) / s);"),
    "quant_range_without_zero": ("float lo = 0.0f, hi = 0.0f;", "float lo = 1e30f, hi = -1e30f;"),
    "head_argmax_last_of_ties": ("if (best_i < 0 || y > best_y) {", "if (best_i < 0 || y >= best_y) {"),
    "head_zero_point_sign": ("int64_t corrected = acc - (int64_t)z[n] * rs;",
                             "int64_t corrected = acc + (int64_t)z[n] * rs;"),
    "head_rowsum_dropped": ("rs += (int64_t)H[v * D + d];", "rs += 0;"),
    "head_transposed": ("acc += (int64_t)H[v * D + d] * (int64_t)Q[n * D + d];",
                        "acc += (int64_t)H[d * V + v % D] * (int64_t)Q[n * D + d];"),
    "embed_scale_row": ("float y = (float)E[t * D + d] * scale[t];",
                        "float y = (float)E[t * D + d] * scale[0];"),
    "rmsnorm_without_eps": ("double r = 1.0 / sqrt(ss / (double)K + eps);",
                            "double r = 1.0 / sqrt(ss / (double)K);"),
    "swiglu_sign": ("H[i] = g / (1.0 + exp(-g)) * u;", "H[i] = g / (1.0 + exp(g)) * u;"),
    "absmean_ties_away": ("T[m * K + k] = (int8_t)rint(r);", "T[m * K + k] = (int8_t)round(r);"),
    "absmean_no_clamp": ("if (r > 1.0) r = 1.0;", "if (r > 2.0) r = 2.0;"),
    "blockscale_wrong_block": ("y += (double)bscale[m * KB + b] * s;", "y += (double)bscale[m * KB] * s;"),
    "int_acc_dropped_term": ("for (int64_t k = 0; k < K; ++k) acc += (int64_t)w[k] * (int64_t)Q[n * K + k];",
                             "for (int64_t k = 0; k + 1 < K; ++k) acc += (int64_t)w[k] * (int64_t)Q[n * K + k];"),
}


def _pins():
    """(name, callable) for every pin, with the oracle module bound."""
    o = omod
    return [
        ("layout", lambda: T.test_layout_hand_derived_positions(o)),
        ("roundtrip", lambda: [T.test_pack_unpack_roundtrip(o, M, K) for M, K in T.SHAPES]),
        ("rowsum", lambda: [T.test_rowsum_three_ways(o, M, K) for M, K in T.SHAPES]),
        ("brute_a", lambda: [T.test_linear_a_matches_dense_bruteforce(o, M, K, N)
                             for M, K in T.SHAPES for N in (1, 3)]),
        ("closed_a", lambda: T.test_linear_a_closed_forms(o)),
        ("quant_onehot", lambda: T.test_quant_one_hot_closed_form(o)),
        ("quant_props", lambda: [T.test_quant_properties(o, s) for s in (False, True)]),
        ("quant_ties", lambda: T.test_quant_ties_round_to_even(o)),
        ("quant_range", lambda: T.test_quant_range_includes_zero(o)),
        ("int_sums", lambda: [T.test_linear_b_integer_sums_match_numpy(o, M, K) for M, K in T.SHAPES]),
        ("onehot_b", lambda: T.test_linear_b_one_hot_identity(o)),
        ("b_tracks_a", lambda: [T.test_linear_b_tracks_linear_a_within_quant_error(o, s)
                                for s in (False, True)]),
        ("head_sums", lambda: [T.test_head_integer_sums_and_argmax(o, V, D, N)
                               for V, D, N in ((37, 64, 1), (100, 160, 3), (5, 16, 8))]),
        ("head_ties", lambda: T.test_head_ties_go_to_the_smallest_index(o)),
        ("head_dense", lambda: T.test_head_tracks_the_dense_product(o)),
        ("head_onehot", lambda: T.test_head_one_hot_closed_form(o)),
        ("embed", lambda: T.test_embed_rows_times_scale(o)),
        ("rmsnorm", lambda: T.test_rmsnorm_identities(o)),
        ("swiglu", lambda: T.test_swiglu_identities(o)),
        ("absmean", lambda: T.test_absmean_closed_forms(o)),
        ("blockscale", lambda: [T.test_blockscale_linear_matches_dense(o, M, K, N)
                                for M, K, N in ((16, 128, 1), (37, 300, 3), (5, 1000, 2))]),
    ]


def _compile(tmp_path, name, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib_{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-pthread", "-shared", "-fPIC", str(path), "-o", str(lib), "-lm"])
    return str(lib)


def test_unmutated_oracle_passes_every_pin():
    for name, fn in _pins():
        fn()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    mutated = omod.load(_compile(tmp_path, name, old, new))
    saved = omod.lib()
    omod._lib = mutated
    caught = []
    try:
        for pin, fn in _pins():
            try:
                fn()
            except (AssertionError, ValueError):
                caught.append(pin)
    finally:
        omod._lib = saved
    assert caught, f"no pin caught the planted mistake {name}"
