"""GPU: chains of linears run by one persistent launch.

A chain must give, bit for bit, what the launch-per-linear path gives for the
same arguments (same work split, same summation order), read each step's
input only after the previous step has written it, leave its workspace's
counters zero after every pass, and report a wait that gives up through its
status word without hanging the launch.
"""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402
from bit_matvec_ternary_b300.stack import GROUPS, LinearStack  # noqa: E402
from tests.test_parity_gpu import TOL_A, Mat, bf16_tensor, rel_err  # noqa: E402

A, B = tl.TL_MODE_BF16, tl.TL_MODE_I8


def _passes_done(chain):
    # the chain counts its completed passes right after the status word
    return int(chain.workspace[256:264].view(torch.int64).item())


def _layer_steps(oracle_mod, N, seed):
    shp = synth.NEUTRINO_8B.linear_shapes()
    mats = {p: Mat(oracle_mod, shp[p][0], shp[p][1], seed=seed + i,
                   p0=synth.zero_fraction(synth.NEUTRINO_8B, 1, p))
            for i, p in enumerate(synth.PROJ_ORDER)}
    steps, xs = [], []
    for gi, grp in enumerate(GROUPS):
        K = shp[grp[0]][1]
        Xh = synth.activations(N, K, seed=seed + 50 + gi, outlier_frac=0.01)
        outs = [torch.empty((N, mats[p].M), dtype=torch.float32, device="cuda") for p in grp]
        steps.append(([mats[p].dev for p in grp], bf16_tensor(Xh), outs))
        xs.append(Xh)
    return mats, steps, xs


@pytest.mark.parametrize("mode", [A, B])
@pytest.mark.parametrize("N", [1, 3, 8])
def test_chain_equals_launch_per_linear(oracle_mod, mode, N):
    """One 8B-shaped layer (q/k/v, o, gate/up, down) as a chain."""
    mats, steps, xs = _layer_steps(oracle_mod, N, seed=700 + N)
    refs = []
    for ws, X, _ in steps:
        if mode == A:
            refs.append(tl.tl_linear_group(ws, X))
        else:
            Q, s, z = tl.tl_quantize_act(X)
            refs.append(tl.tl_linear_group(ws, Q, s, z, mode=B))
    chain = tl.Chain(steps, N, mode)
    for p in range(3):
        for _, _, outs in steps:
            for o in outs:
                o.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        assert chain.status() == 0
        for (_, _, outs), ref in zip(steps, refs):
            for o, r in zip(outs, ref):
                assert torch.equal(o.view(torch.int32), r.view(torch.int32))
        assert _passes_done(chain) == p + 1
    # and one group against the oracle directly
    m = mats["down"]
    Xh = xs[3]
    y = steps[3][2][0].cpu().numpy()
    if mode == A:
        assert rel_err(y, oracle_mod.linear_a_mt(m.P, m.scale, m.M, m.K, Xh)) <= TOL_A
    else:
        Qr, sr, zr = oracle_mod.quant(Xh)
        ref = oracle_mod.linear_b_mt(m.P, m.scale, m.rowsum, m.M, m.K, Qr, sr, zr)
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


# (M, K) of each step; step i + 1 reads step i's bf16 output, so K(i+1) = M(i).
DEPENDENT = [(4096, 4096), (12288, 4096), (4096, 12288), (777, 4096), (1024, 777), (300, 1024)]


@pytest.mark.parametrize("mode", [A, B])
@pytest.mark.parametrize("N", [1, 8])
def test_chain_steps_read_what_the_previous_step_wrote(oracle_mod, mode, N):
    """Each step's input is the previous step's output (bf16), so a step that
    read its input before the previous one had finished writing it would
    differ from the oracle applied to the GPU's own previous output.  The
    shapes cover one-slice and three-slice steps and ragged M and K."""
    mats = [Mat(oracle_mod, M, K, seed=800 + i) for i, (M, K) in enumerate(DEPENDENT)]
    x0 = synth.activations(N, DEPENDENT[0][1], seed=801)
    xs = [bf16_tensor(x0)] + [torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
                              for M, _ in DEPENDENT]
    steps = [([m.dev], xs[i], [xs[i + 1]]) for i, m in enumerate(mats)]
    chain = tl.Chain(steps, N, mode, out_dtype=tl.TL_OUT_BF16)
    for rep in range(2):
        for t in xs[1:]:
            t.zero_()
        chain.run()
        torch.cuda.synchronize()
        assert chain.status() == 0
        for i, m in enumerate(mats):
            xin = xs[i].cpu().view(torch.int16).numpy().view(np.uint16)
            got = xs[i + 1].cpu().view(torch.int16).numpy().view(np.uint16)
            if mode == B:
                Qr, sr, zr = oracle_mod.quant(xin)
                ref = oracle_mod.linear_b_mt(m.P, m.scale, m.rowsum, m.M, m.K, Qr, sr, zr)
                assert np.array_equal(got, oracle_mod.bf16_rne(ref)), (rep, i)
            else:
                ref = oracle_mod.linear_a_mt(m.P, m.scale, m.M, m.K, xin)
                assert rel_err(synth.bf16_bits_to_f32(got), ref) <= TOL_A + 2.0 ** -8, (rep, i)


def test_chain_wait_gives_up_and_reports_it(oracle_mod):
    """A gate that nothing opens: every wait for step 0's inputs gives up
    after its limit, the status word says so, the launch ends by itself, and
    after the caller zero-fills the workspace the same chain runs correctly."""
    mats, steps, _ = _layer_steps(oracle_mod, 1, seed=900)
    refs = [tl.tl_linear_group(ws, X) for ws, X, _ in steps]
    gate = torch.zeros(1, dtype=torch.int32, device="cuda")
    chain = tl.Chain(steps, 1, A, gate=gate, wait_limit=1 << 22)
    chain.run()
    torch.cuda.synchronize()
    assert chain.status() == tl.TL_DEVERR_TIMEOUT
    chain.workspace.zero_()
    gate.fill_(1)
    chain.run()
    torch.cuda.synchronize()
    assert chain.status() == 0
    for (_, _, outs), ref in zip(steps, refs):
        for o, r in zip(outs, ref):
            assert torch.equal(o.view(torch.int32), r.view(torch.int32))


@pytest.mark.parametrize("mode", [A, B])
def test_stack_chain_equals_captured_graph(oracle_mod, mode):
    """Two 8B-shaped layers at eight tokens: the stack as one chain gives
    the same bits as its graph of launch-per-linear calls."""
    shape = synth.NEUTRINO_8B
    st = LinearStack(shape, N=8, mode=mode, layers=2, outlier_frac=0.01)
    st.capture()
    st.graph.replay()
    torch.cuda.synchronize()
    ref = st.Y_flat.clone()
    st.Y_flat.fill_(float("nan"))
    chain = st.chain()
    chain.run()
    torch.cuda.synchronize()
    assert chain.status() == 0
    assert torch.equal(st.Y_flat.view(torch.int32), ref.view(torch.int32))
