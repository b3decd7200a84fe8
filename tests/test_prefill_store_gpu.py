"""GPU: prefill-sized launches whose tiles cover the SMs (no K split), where
whole tiles leave by TMA stores when the output rows allow it (16-byte
aligned, a multiple of 16 bytes) and by element stores otherwise.  Mode B
bit for bit against the oracle (fp32, bf16 and raw int32 outputs, both
quantiser variants, a group, ragged token counts), mode A within the
tolerance."""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402
from tests.test_parity_gpu import TOL_A, Mat, bf16_tensor, rel_err  # noqa: E402

K = 512


def _b(oracle_mod, m, X, symmetric):
    Qr, sr, zr = oracle_mod.quant(X, symmetric=symmetric)
    return oracle_mod.linear_b(m.P, m.scale, m.rowsum, m.M, m.K, Qr, sr, zr)


@pytest.mark.parametrize("M", [148 * 128, 148 * 128 + 1])     # TMA stores / element stores
@pytest.mark.parametrize("N", [256, 300])
@pytest.mark.parametrize("symmetric", [False, True])
def test_unsplit_prefill_mode_b_bit_exact(oracle_mod, M, N, symmetric):
    m = Mat(oracle_mod, M, K, seed=M + N)
    X = synth.activations(N, K, seed=N, outlier_frac=0.01)
    accr, Yr = _b(oracle_mod, m, X, symmetric)
    Q, s, z = tl.tl_quantize_act(bf16_tensor(X), symmetric=symmetric)
    ws = tl.make_workspace([[m.dev]], N)
    Y = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, workspace=ws)
    Yb = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, out_dtype=tl.TL_OUT_BF16, workspace=ws)
    acc = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, out_dtype=tl.TL_OUT_I32_RAW, workspace=ws)
    flags = tl.TL_FLAG_SYMMETRIC if symmetric else 0
    Yf = tl.tl_linear(m.dev, bf16_tensor(X), mode=tl.TL_MODE_I8_FUSED, out_dtype=tl.TL_OUT_BF16,
                      workspace=ws, flags=flags)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), accr)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
    rne = oracle_mod.bf16_rne(Yr)
    assert np.array_equal(Yb.cpu().view(torch.int16).numpy().view(np.uint16), rne)
    assert np.array_equal(Yf.cpu().view(torch.int16).numpy().view(np.uint16), rne)


@pytest.mark.parametrize("M", [148 * 128, 148 * 128 + 1])
def test_unsplit_prefill_mode_a(oracle_mod, M):
    N = 300
    m = Mat(oracle_mod, M, K, seed=M)
    X = synth.activations(N, K, seed=5)
    ref = oracle_mod.linear_a(m.P, m.scale, M, K, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A
    Yb = tl.tl_linear(m.dev, bf16_tensor(X), out_dtype=tl.TL_OUT_BF16).float().cpu().numpy()
    assert rel_err(Yb, ref) <= TOL_A + 2.0 ** -8


def test_unsplit_prefill_group(oracle_mod):
    """A gate/up-like pair of 74 row tiles each (one wave of 148 tiles)."""
    N = 256
    mats = [Mat(oracle_mod, 74 * 128, K, seed=60 + i) for i in range(2)]
    X = synth.activations(N, K, seed=61)
    Q, s, z = tl.tl_quantize_act(bf16_tensor(X))
    ys = tl.tl_linear_group([m.dev for m in mats], Q, s, z, mode=tl.TL_MODE_I8,
                            out_dtype=tl.TL_OUT_BF16)
    torch.cuda.synchronize()
    for m, y in zip(mats, ys):
        _, Yr = _b(oracle_mod, m, X, False)
        assert np.array_equal(y.cpu().view(torch.int16).numpy().view(np.uint16), oracle_mod.bf16_rne(Yr))
