"""GPU: the full 36-layer 8B-shaped stack, in the launch configuration the
benchmark times (a CUDA graph of per-group launches with programmatic
dependent launch), checked against the CPU oracle on sampled rows of every
projection of three layers (the first, a middle one and the last): within
the mode-A tolerance, and bit for bit in mode B (quantiser launches, or the
quantisation fused into the linears).  The same stack run as one chain
launch must give the graph's bits everywhere."""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402
from bit_matvec_ternary_b300.stack import GROUPS, LinearStack, StackWeights  # noqa: E402
from tests.test_parity_gpu import TOL_A, rel_err  # noqa: E402

SHAPE = synth.NEUTRINO_8B
CHECKED = (0, 17, 35)


@pytest.fixture(scope="module")
def weights():
    return StackWeights(SHAPE, keep_host=CHECKED)


def _rows(M, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=48, replace=False)]))


@pytest.mark.parametrize("N,mode", [(1, tl.TL_MODE_BF16), (8, tl.TL_MODE_BF16), (8, tl.TL_MODE_I8),
                                    (1, tl.TL_MODE_I8), (1, tl.TL_MODE_I8_FUSED),
                                    (8, tl.TL_MODE_I8_FUSED)])
def test_full_stack_against_oracle_on_sampled_rows(oracle_mod, weights, N, mode):
    outl = 0.01 if N == 8 else 0.0
    st = LinearStack(SHAPE, N=N, mode=mode, weights=weights, outlier_frac=outl)
    st.capture()
    st.Y_flat.fill_(float("nan"))
    st.graph.replay()
    torch.cuda.synchronize()
    graph_out = st.Y_flat.clone()
    for layer in CHECKED:
        for gi, grp in enumerate(GROUPS):
            xh = st.X[layer][gi].cpu().view(torch.int16).numpy().view(np.uint16)
            for p, y in zip(grp, st.Y[layer][gi]):
                W, scale = weights.host[(layer, p)]
                M, K = W.shape
                rows = _rows(M, 1000 * layer + gi)
                P = oracle_mod.pack(W[rows])
                got = y.cpu().numpy()[:, rows]
                if mode == tl.TL_MODE_BF16:
                    ref = oracle_mod.linear_a(P, scale[rows], rows.size, K, xh)
                    assert rel_err(got, ref) <= TOL_A, (layer, p)
                else:
                    Qr, sr, zr = oracle_mod.quant(xh)
                    rs = oracle_mod.rowsum(P, rows.size, K)
                    _, ref = oracle_mod.linear_b(P, scale[rows], rs, rows.size, K, Qr, sr, zr)
                    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (layer, p)
    # the same stack as one chain launch (mode B's chain for the fused mode:
    # its quantiser steps are its own): the graph's bits
    cs = st if mode != tl.TL_MODE_I8_FUSED else LinearStack(
        SHAPE, N=N, mode=tl.TL_MODE_I8, weights=weights, outlier_frac=outl)
    cs.Y_flat.fill_(float("nan"))
    chain = cs.chain()
    chain.run()
    torch.cuda.synchronize()
    assert chain.status() == 0
    assert torch.equal(cs.Y_flat.view(torch.int32), graph_out.view(torch.int32))
