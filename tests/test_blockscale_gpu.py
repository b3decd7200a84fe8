"""GPU: the block-wise scale variant (one scale per row and 128-column
block, codes from the absmean ternariser) against the CPU oracle, within
the mode-A tolerance of the other parity tests."""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402
from tests.test_parity_gpu import TOL_A, bf16_tensor, rel_err  # noqa: E402


def _weights(oracle_mod, M, K, seed):
    rng = np.random.default_rng(seed)
    Wf = (rng.standard_normal((M, K)) * rng.uniform(0.01, 0.1, size=(M, 1))).astype(np.float32)
    w = tl.BlockScaledWeight.from_float(Wf)
    T, bs = oracle_mod.absmean_ternarize(Wf)
    return w, oracle_mod.pack(T), bs


@pytest.mark.parametrize("M,K", [(2048, 1024), (4096, 4096), (777, 333), (4096, 12288),
                                 (12288, 4096), (16, 128), (5, 1000), (300, 4224)])
@pytest.mark.parametrize("N", [1, 8, 13])
def test_blockscale_against_oracle(oracle_mod, M, K, N):
    w, P, bs = _weights(oracle_mod, M, K, M + K)
    X = synth.activations(N, K, seed=N + K, outlier_frac=0.01)
    Y = tl.tl_linear_blockscale(w, bf16_tensor(X)).cpu().numpy()
    ref = oracle_mod.linear_blockscale(P, bs, M, K, X)
    assert rel_err(Y, ref) <= TOL_A


def test_blockscale_one_signed_activations_and_bf16_output(oracle_mod):
    M, K = 2048, 12288
    w, P, bs = _weights(oracle_mod, M, K, 3)
    X = synth.to_bf16_bits(np.abs(np.random.default_rng(4).standard_normal((8, K))).astype(np.float32))
    ref = oracle_mod.linear_blockscale(P, bs, M, K, X)
    Y = tl.tl_linear_blockscale(w, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A
    Yb = tl.tl_linear_blockscale(w, bf16_tensor(X), out_dtype=tl.TL_OUT_BF16).float().cpu().numpy()
    assert rel_err(Yb, ref) <= TOL_A + 2.0 ** -8


@pytest.mark.parametrize("K", [4096, 1000])
def test_blockscale_unaligned_activations(oracle_mod, K):
    """X starting 2 bytes past a 16-byte boundary (activations read from
    global memory rather than staged): the same sums as the staged path."""
    M, N = 4096, 3
    w, P, bs = _weights(oracle_mod, M, K, K + 1)
    X = synth.activations(N, K, seed=K, outlier_frac=0.01)
    flat = bf16_tensor(np.concatenate([np.zeros(1, np.uint16), X.reshape(-1)]))[1:].view(N, K)
    ref = oracle_mod.linear_blockscale(P, bs, M, K, X)
    Yu = tl.tl_linear_blockscale(w, flat).cpu().numpy()
    assert rel_err(Yu, ref) <= TOL_A
    Ya = tl.tl_linear_blockscale(w, bf16_tensor(X)).cpu().numpy()
    assert np.array_equal(Ya.view(np.uint32), Yu.view(np.uint32))


def test_blockscale_batch_invariance(oracle_mod):
    """A token's result does not depend on the batch it is in (staged rows at
    one token, global reads at eight tokens of K = 12,288)."""
    M, K = 1024, 12288
    w, P, bs = _weights(oracle_mod, M, K, 9)
    X = bf16_tensor(synth.activations(8, K, seed=10, outlier_frac=0.01))
    Y8 = tl.tl_linear_blockscale(w, X).cpu().numpy().view(np.uint32)
    for n in range(8):
        Y1 = tl.tl_linear_blockscale(w, X[n:n + 1].contiguous()).cpu().numpy().view(np.uint32)
        assert np.array_equal(Y8[n], Y1[0]), n
