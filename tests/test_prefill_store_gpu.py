"""GPU: prefill-sized launches whose tiles cover the SMs (no K split), where
whole tiles leave by TMA stores when the output rows allow it (16-byte
aligned, a multiple of 16 bytes) and by element stores otherwise.  Mode B
bit for bit against the oracle (fp32, bf16 and raw int32 outputs, both
quantiser variants, a group, ragged token counts), mode A within the
tolerance.  And a K-split launch's arrival counters, kept in the
workspace's front bytes."""
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


def test_split_prefill_leaves_the_front_zero(oracle_mod):
    """A K-split launch keeps its per-tile arrival counters in the
    workspace's front bytes (no clearing launch before it): after the call
    they are zero again, and the same workspace then serves a decode call
    and a second split call correctly."""
    M, Kb, N = 1024, 12288, 300
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = tl.prefill_plan([tl.tl_weight(0x1000, 0x2000, 0x3000, M, Kb, tl.TL_LAYOUT_TL2P_V2)], N, sms)
    assert p["S"] > 1
    m = Mat(oracle_mod, M, Kb, seed=91)
    X = synth.activations(N, Kb, seed=92)
    Q, s, z = tl.tl_quantize_act(bf16_tensor(X))
    need = max(tl.tl_workspace_bytes([m.dev], N), tl.tl_workspace_bytes([m.dev], 3))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y1 = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, workspace=ws)
    torch.cuda.synchronize()
    front = 256 + p["tiles"] * 8
    assert int(ws[:front].count_nonzero()) == 0
    _, Yr = _b(oracle_mod, m, X, False)
    assert np.array_equal(y1.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
    # a decode call, then the split call again, on the same workspace
    X1 = synth.activations(3, Kb, seed=93)
    Q1, s1, z1 = tl.tl_quantize_act(bf16_tensor(X1))
    y3 = tl.tl_linear(m.dev, Q1, s1, z1, mode=tl.TL_MODE_I8, workspace=ws)
    y2 = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, workspace=ws)
    torch.cuda.synchronize()
    _, Yr1 = _b(oracle_mod, m, X1, False)
    assert np.array_equal(y3.cpu().numpy().view(np.uint32), Yr1.view(np.uint32))
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
    assert int(ws[:front].count_nonzero()) == 0
