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


@pytest.mark.parametrize("N,mode", [(1, tl.TL_MODE_BF16), (8, tl.TL_MODE_I8_FUSED)])
def test_host_copy_graph_equals_the_device_graph(oracle_mod, weights, N, mode):
    """The pass with its host copies in the graph (each layer's inputs copied
    in on one stream ahead of it, its outputs out on another after it): the
    pinned host outputs equal the device graph's outputs bit for bit, and new
    host inputs are picked up by the next replay (checked against the oracle
    on sampled rows of the last layer)."""
    st = LinearStack(SHAPE, N=N, mode=mode, out_dtype=tl.TL_OUT_F32, symmetric=False,
                     weights=weights)
    st.capture()
    st.graph.replay()
    torch.cuda.synchronize()
    ref = st.Y_flat.cpu().numpy().view(np.uint32).copy()
    hx = torch.empty(st.X_flat.shape, dtype=st.X_flat.dtype, pin_memory=True)
    hx.copy_(st.X_flat.cpu())
    hy = torch.zeros(st.Y_flat.shape, dtype=st.Y_flat.dtype, pin_memory=True)
    g = st.capture_e2e(hx, hy)
    st.Y_flat.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(hy.numpy().view(np.uint32), ref)
    # new inputs for the last layer's down projection, from the host only
    l = SHAPE.layers - 1
    K = SHAPE.linear_shapes()["down"][1]
    X = synth.activations(N, K, seed=991, outlier_frac=0.01)
    lo = st.x_span[l][1] - N * K
    hx[lo:].copy_(torch.from_numpy(X.view(np.int16).reshape(-1).copy()).view(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    W, scale = weights.host[(l, "down")]
    M = W.shape[0]
    rows = _rows(M, 5)
    Pr = oracle_mod.pack(W[rows])
    y = hy.numpy()[st.y_span[l][1] - N * M:].reshape(N, M)[:, rows]
    if mode == tl.TL_MODE_BF16:
        yr = oracle_mod.linear_a(Pr, scale[rows], len(rows), K, X)
        assert rel_err(y, yr) <= TOL_A
    else:
        Q, s, z = oracle_mod.quant(X)
        _, yr = oracle_mod.linear_b(Pr, scale[rows], oracle_mod.rowsum(Pr, len(rows), K),
                                    len(rows), K, Q, s, z)
        assert np.array_equal(y.view(np.uint32), yr.view(np.uint32))
