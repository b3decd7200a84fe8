"""GPU: RMSNorm + quantisation and SwiGLU + quantisation, through the C ABI,
against the CPU oracle.

The ops are computed in fp32 and rounded once to bf16, so each bf16 output
must be the bf16 nearest the oracle's float64 value or its neighbour (one
unit in the last place: the fp32 result can sit on the other side of a
rounding boundary).  The quantisation is decided on that bf16 row, so Q, s
and z must be bit for bit the oracle's quantiser applied to the GPU's own
bf16 output (and equal to the library's stand-alone quantiser on it).
"""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402
from tests.test_parity_gpu import bf16_tensor  # noqa: E402


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _within_one_ulp(got_bits, ref64):
    """got is the bf16 nearest ref64, or one of its two neighbours."""
    near = synth.to_bf16_bits(ref64.astype(np.float32)).astype(np.int32)
    # compare in the ordered integer image of bf16 (sign-magnitude -> two's complement)
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.all(np.abs(ordered(got_bits) - ordered(near)) <= 1)


def _check_quant(oracle_mod, Y, Q, s, z, symmetric):
    yb = _bits(Y)
    Qr, sr, zr = oracle_mod.quant(yb, symmetric=symmetric)
    assert np.array_equal(Q.cpu().numpy(), Qr)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zr)
    Q2, s2, z2 = tl.tl_quantize_act(Y, symmetric=symmetric)
    assert torch.equal(Q2, Q) and torch.equal(s2.view(torch.int32), s.view(torch.int32))


# one token's row spans a cluster of up to eight CTAs: 1 (K <= 1024) ... 8,
# ragged last slices (1025, 4100) and the largest row (32768)
@pytest.mark.parametrize("N,K", [(1, 4096), (8, 4096), (3, 1024), (2, 333), (1, 12288),
                                 (2, 4100), (1, 32768)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_rmsnorm_quant(oracle_mod, N, K, symmetric):
    X = synth.activations(N, K, seed=K + N, outlier_frac=0.01)
    rng = np.random.default_rng(K)
    gamma = synth.to_bf16_bits(rng.uniform(0.2, 2.0, size=K).astype(np.float32))
    Y, Q, s, z = tl.tl_rmsnorm_quant(bf16_tensor(X), bf16_tensor(gamma), 1e-6,
                                     symmetric=symmetric)
    torch.cuda.synchronize()
    assert _within_one_ulp(_bits(Y), oracle_mod.rmsnorm(X, gamma, 1e-6))
    _check_quant(oracle_mod, Y, Q, s, z, symmetric)
    # the quantised output alone gives the same codes
    _, Q1, s1, _ = tl.tl_rmsnorm_quant(bf16_tensor(X), bf16_tensor(gamma), 1e-6, want_y=False,
                                       symmetric=symmetric)
    assert torch.equal(Q1, Q) and torch.equal(s1.view(torch.int32), s.view(torch.int32))


@pytest.mark.parametrize("N,M", [(1, 12288), (8, 12288), (3, 3072), (2, 777), (1, 1025),
                                 (4, 32768)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_swiglu_quant(oracle_mod, N, M, symmetric):
    rng = np.random.default_rng(M + N)
    G = synth.to_bf16_bits((rng.standard_normal((N, M)) * 3).astype(np.float32))
    U = synth.to_bf16_bits(rng.standard_normal((N, M)).astype(np.float32))
    H, Q, s, z = tl.tl_swiglu_quant(bf16_tensor(G), bf16_tensor(U), symmetric=symmetric)
    torch.cuda.synchronize()
    assert _within_one_ulp(_bits(H), oracle_mod.swiglu(G, U))
    _check_quant(oracle_mod, H, Q, s, z, symmetric)


def test_rmsnorm_of_a_zero_row_and_swiglu_extremes(oracle_mod):
    X = np.zeros((2, 256), dtype=np.uint16)
    X[1] = synth.to_bf16_bits(np.full(256, 1e-20, np.float32))
    gamma = synth.to_bf16_bits(np.ones(256, np.float32))
    Y, Q, s, z = tl.tl_rmsnorm_quant(bf16_tensor(X), bf16_tensor(gamma), 1e-6)
    torch.cuda.synchronize()
    assert not _bits(Y)[0].any() and float(s[0]) == 1.0 and int(z[0]) == 0
    assert _within_one_ulp(_bits(Y), oracle_mod.rmsnorm(X, gamma, 1e-6))
    G = synth.to_bf16_bits(np.float32([[100.0, -100.0, 0.0, 30.0]]))
    U = synth.to_bf16_bits(np.float32([[1.0, 1.0, 5.0, -2.0]]))
    H, *_ = tl.tl_swiglu_quant(bf16_tensor(G), bf16_tensor(U))
    torch.cuda.synchronize()
    assert _within_one_ulp(_bits(H), oracle_mod.swiglu(G, U))
