"""The synthetic workload reproduces the shapes and statistics the pages print."""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth
from tests.conftest import read_golden

G = {k: v for k, v in read_golden("neutrino_shapes.txt")}


def test_8b_parameter_arithmetic():
    s = synth.NEUTRINO_8B
    assert s.total_params() == int(G["params_8b"])
    assert round(s.ternary_weights() / 1e9, 2) == float(G["coded_weights_8b_e9"])
    assert round(s.embedding_params() / 1e9, 2) == float(G["embedding_params_8b_e9"])
    assert round(s.norm_params() / 1e6, 1) == float(G["norm_params_8b_e6"])
    assert 4 * s.layers + 1 == int(G["norm_tensors_8b"])
    assert s.linears == int(G["linears_8b"])
    assert s.kv_bytes_per_token_fp16() == int(G["kv_bytes_per_token_8b"])
    assert s.kv_bytes_per_token_fp16() == int(G["kv_kib_per_token_8b"]) * 1024
    assert round(100 * s.ternary_weights() / s.total_params(), 1) == float(G["coded_param_pct_8b"])


def test_8b_layer_bytes_are_three_bits_per_weight():
    per_layer = synth.NEUTRINO_8B.ternary_weights_per_layer()
    assert per_layer == 192_937_984
    assert per_layer * 3 == int(G["bytes_per_layer_8b"]) * 8


def test_06b_parameter_arithmetic():
    s = synth.NEUTRINO_06B
    assert s.total_params() == int(G["params_06b"])
    assert s.linears == int(G["linears_06b"])
    assert round(100 * s.ternary_weights() / s.total_params(), 1) == float(G["coded_param_pct_06b"])


def test_stack_layout_order_and_shapes():
    lay = synth.stack_layout(synth.NEUTRINO_8B)
    assert len(lay) == 252
    assert lay[:7] == [(0, "q", 4096, 4096), (0, "k", 1024, 4096), (0, "v", 1024, 4096),
                       (0, "o", 4096, 4096), (0, "gate", 12288, 4096),
                       (0, "up", 12288, 4096), (0, "down", 4096, 12288)]
    assert sum(m * k for _, _, m, k in lay) == synth.NEUTRINO_8B.ternary_weights()


def test_zero_fraction_table_matches_pages():
    z = synth.zero_fraction_8b
    lo, hi = float(G["attention_band_lo_pct"]) / 100, float(G["attention_band_hi_pct"]) / 100
    for l in range(36):
        for p in ("q", "k", "v", "o"):
            assert lo <= z(l, p) <= hi
    assert z(0, "down") == pytest.approx(float(G["densest_down_pct"]) / 100, abs=1e-12)
    assert z(2, "down") == pytest.approx(float(G["down_spike_pct"]) / 100, abs=1e-12)
    assert z(3, "gate") == pytest.approx(float(G["gate_spike_pct"]) / 100, abs=1e-12)
    for l in range(5, 36):
        assert z(l, "gate") == z(l, "down") == z(l, "up") == synth.P0_DEFAULT
    # the stack-wide zero share stays close to the published 62.63 %
    tot = sum(m * k * z(l, p) for l, p, m, k in synth.stack_layout(synth.NEUTRINO_8B))
    assert abs(100 * tot / synth.NEUTRINO_8B.ternary_weights() - float(G["zero_pct_8b"])) < 0.5


@pytest.mark.parametrize("p0", [0.626, 0.7247, 0.6059])
def test_ternary_statistics_within_binomial_bounds(p0):
    M, K = 1024, 1024
    W = synth.ternary(M, K, p0, seed=1)
    n = W.size
    zero = (W == 0).mean()
    plus = (W == 1).mean()
    sd = np.sqrt(p0 * (1 - p0) / n)
    assert abs(zero - p0) < 4 * sd + 1.0 / 65536
    half = (1 - p0) / 2
    assert abs(plus - half) < 4 * np.sqrt(half * (1 - half) / n) + 1.0 / 65536
    assert set(np.unique(W)) <= {-1, 0, 1}


def test_generators_are_seeded():
    a = synth.ternary(64, 256, 0.626, 5)
    b = synth.ternary(64, 256, 0.626, 5)
    c = synth.ternary(64, 256, 0.626, 6)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    x = synth.activations(3, 100, 4)
    assert np.array_equal(x, synth.activations(3, 100, 4))
    s = synth.scales(100, 2)
    assert s.dtype == np.float32 and s.min() >= 0.005 and s.max() <= 0.05


def test_outliers_and_unit_rms():
    x = synth.bf16_bits_to_f32(synth.activations(4, 4096, 1, outlier_frac=0.01))
    big = np.abs(x) > 8
    cols = np.flatnonzero(big.any(axis=0))
    assert 20 <= len(cols) <= 41           # ~41 outlier channels, most exceed 8
    xr = synth.bf16_bits_to_f32(synth.activations(4, 4096, 1, unit_rms=True))
    rms = np.sqrt((xr.astype(np.float64) ** 2).mean(axis=1))
    assert np.allclose(rms, 1.0, atol=2e-3)


def test_bf16_rounding_of_inputs():
    v = np.array([1 + 2**-8, 1 + 3 * 2**-8, -0.0, np.inf], dtype=np.float32)
    assert list(synth.to_bf16_bits(v)) == [0x3F80, 0x3F82, 0x8000, 0x7F80]
