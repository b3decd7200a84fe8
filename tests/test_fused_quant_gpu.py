"""GPU parity of TL_MODE_I8_FUSED: the decode kernel quantises each token of
its bf16 X itself.  The result must be bit for bit the oracle's per-token
quantisation followed by the oracle's integer linear (and so what
tl_quantize_act + TL_MODE_I8 gives), for every shape, batch, alignment and
both quantiser variants.
"""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402

F = tl.TL_MODE_I8_FUSED


def bf16_tensor(bits: np.ndarray):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


class Mat:
    def __init__(self, oracle_mod, M, K, seed, W=None):
        self.W = synth.ternary(M, K, 0.626, seed) if W is None else W
        self.scale = synth.scales(M, seed)
        self.M, self.K = M, K
        self.P = oracle_mod.pack(self.W)
        self.rowsum = oracle_mod.rowsum(self.P, M, K)
        self.dev = tl.TernaryWeight.from_int8(self.W, self.scale)


def oracle_y(oracle_mod, m, X, symmetric=False):
    Q, s, z = oracle_mod.quant(X, symmetric=symmetric)
    _, Y = oracle_mod.linear_b(m.P, m.scale, m.rowsum, m.M, m.K, Q, s, z)
    return Y


def fused(m, Xd, symmetric=False, out_dtype=tl.TL_OUT_F32, flags=0):
    flags |= tl.TL_FLAG_SYMMETRIC if symmetric else 0
    Y = tl.tl_linear(m.dev, Xd, mode=F, out_dtype=out_dtype, flags=flags)
    torch.cuda.synchronize()
    return Y


def bits(t):
    return t.cpu().numpy().view(np.uint32)


SHAPES = [(2048, 1024), (1024, 2048), (3072, 1024), (4096, 4096), (1024, 4096), (4096, 12288),
          (5, 37), (17, 129), (100, 1000), (33, 4099), (1, 1), (16, 128), (777, 333)]


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("N", [1, 3, 8])
@pytest.mark.parametrize("symmetric", [False, True])
def test_fused_bit_exact(oracle_mod, M, K, N, symmetric):
    m = Mat(oracle_mod, M, K, seed=5 * M + K)
    X = synth.activations(N, K, seed=3 * N + K, outlier_frac=0.01 if K >= 100 else 0.0)
    Yr = oracle_y(oracle_mod, m, X, symmetric)
    Y = fused(m, bf16_tensor(X), symmetric)
    assert np.array_equal(bits(Y), Yr.view(np.uint32))


@pytest.mark.parametrize("symmetric", [False, True])
def test_fused_equals_two_launch_path(oracle_mod, symmetric):
    m = Mat(oracle_mod, 4096, 4096, seed=1)
    X = bf16_tensor(synth.activations(8, 4096, seed=2, outlier_frac=0.01))
    Q, s, z = tl.tl_quantize_act(X, symmetric=symmetric)
    Y2 = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8)
    Y1 = fused(m, X, symmetric)
    assert np.array_equal(bits(Y1), bits(Y2))


def test_fused_special_tokens(oracle_mod):
    """All-zero, all-negative, all-positive and tie-rounding tokens, and the
    quantiser's extremes against +-1 weights (the largest |acc|)."""
    K = 4096
    M = 64
    W = np.ones((M, K), dtype=np.int8)
    W[1::2] = -1
    W[2::4, ::3] = 0
    m = Mat(oracle_mod, M, K, seed=7, W=W)
    X = synth.activations(8, K, seed=8)
    X[0] = 0
    X[1] = synth.to_bf16_bits(-np.abs(synth.bf16_bits_to_f32(X[1])))
    X[2] = synth.to_bf16_bits(np.abs(synth.bf16_bits_to_f32(X[2])))
    X[3] = 0
    X[3, :6] = synth.to_bf16_bits(np.float32([255.0, 2.5, 0.5, 1.5, 3.5, -4.5]))
    x4 = np.full(K, -1.0, dtype=np.float32)
    x4[0] = 1e-3
    X[4] = synth.to_bf16_bits(x4)
    X[5] = synth.to_bf16_bits(np.full(K, 3.0, dtype=np.float32))   # constant row
    for sym in (False, True):
        Yr = oracle_y(oracle_mod, m, X, sym)
        assert np.array_equal(bits(fused(m, bf16_tensor(X), sym)), Yr.view(np.uint32))


@pytest.mark.parametrize("M,K", [(4096, 4096), (1024, 12288), (777, 333)])
def test_fused_batch_invariance(oracle_mod, M, K):
    m = Mat(oracle_mod, M, K, seed=11)
    X = bf16_tensor(synth.activations(8, K, seed=12, outlier_frac=0.01))
    Y8 = bits(fused(m, X))
    for n in range(8):
        Y1 = bits(fused(m, X[n:n + 1].contiguous()))
        assert np.array_equal(Y8[n], Y1[0]), n


def test_fused_unaligned_rows_use_scalar_loads(oracle_mod):
    """X starting 2 bytes past a 16-byte boundary, and K not a multiple of 8."""
    for K in (4096, 1000, 333):
        m = Mat(oracle_mod, 1024, K, seed=K)
        X = synth.activations(5, K, seed=K + 1, outlier_frac=0.01)
        flat = bf16_tensor(np.concatenate([np.zeros(1, np.uint16), X.reshape(-1)]))[1:].view(5, K)
        Yr = oracle_y(oracle_mod, m, X)
        assert np.array_equal(bits(fused(m, flat)), Yr.view(np.uint32)), K


@pytest.mark.parametrize("N", [9, 20, 300])
def test_fused_batches_above_eight(oracle_mod, N):
    """Chunks of 8 on the decode kernel below 256 tokens; from 256 the
    quantiser's bf16 integers feed the tensor-core kernel."""
    m = Mat(oracle_mod, 1024, 3072, seed=30)
    X = synth.activations(N, 3072, seed=31)
    Yr = oracle_y(oracle_mod, m, X)
    assert np.array_equal(bits(fused(m, bf16_tensor(X))), Yr.view(np.uint32))


def test_fused_group_and_bf16_output(oracle_mod):
    mats = [Mat(oracle_mod, M, 4096, seed=20 + i) for i, M in enumerate((4096, 1024, 1024))]
    X = synth.activations(3, 4096, seed=21)
    ys = tl.tl_linear_group([m.dev for m in mats], bf16_tensor(X), mode=F,
                            out_dtype=tl.TL_OUT_BF16)
    torch.cuda.synchronize()
    for m, y in zip(mats, ys):
        Yr = oracle_y(oracle_mod, m, X)
        got = y.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, oracle_mod.bf16_rne(Yr))


@pytest.mark.parametrize("M,K", [(16, 65536), (64, 49152)])
def test_fused_long_k(oracle_mod, M, K):
    """Many K slices: every CTA of every slice derives the same s and z."""
    m = Mat(oracle_mod, M, K, seed=M + K)
    X = synth.activations(4, K, seed=K, outlier_frac=0.01)
    Yr = oracle_y(oracle_mod, m, X)
    assert np.array_equal(bits(fused(m, bf16_tensor(X))), Yr.view(np.uint32))


def test_fused_pdl_chain_in_a_graph(oracle_mod):
    """Dependent launches (TL_FLAG_PDL): a bf16-output linear feeding a fused
    one, captured in a graph and replayed."""
    m1 = Mat(oracle_mod, 2048, 1024, seed=40)
    m2 = Mat(oracle_mod, 1024, 2048, seed=41)
    X = bf16_tensor(synth.activations(2, 1024, seed=42))
    ws = tl.make_workspace([[m1.dev], [m2.dev]], 2)
    h = torch.empty((2, 2048), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((2, 1024), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tl.tl_linear(m1.dev, X, out=h, out_dtype=tl.TL_OUT_BF16, workspace=ws, stream=s)
        tl.tl_linear(m2.dev, h, out=y, mode=F, workspace=ws, flags=tl.TL_FLAG_PDL, stream=s)
    s.synchronize()
    first = bits(y).copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tl.tl_linear(m1.dev, X, out=h, out_dtype=tl.TL_OUT_BF16, workspace=ws,
                     flags=tl.TL_FLAG_PDL, stream=s)
        tl.tl_linear(m2.dev, h, out=y, mode=F, workspace=ws, flags=tl.TL_FLAG_PDL, stream=s)
    y.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(y), first)
    hb = h.cpu().view(torch.int16).numpy().view(np.uint16)
    Yr = oracle_y(oracle_mod, m2, hb)
    assert np.array_equal(first, Yr.view(np.uint32))


@pytest.mark.parametrize("M,K,N", [(3072, 1024, 512), (1024, 12288, 256), (777, 4096, 300)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_fused_prefill_sizes(oracle_mod, M, K, N, symmetric):
    """Prefill-sized batches (the K-split path at K = 12,288, ragged M and N):
    bit for bit the oracle's quantisation and integer linear, fp32 and bf16
    out, and a group."""
    m = Mat(oracle_mod, M, K, seed=M + K + N)
    X = synth.activations(N, K, seed=N + 3, outlier_frac=0.01)
    Yr = oracle_y(oracle_mod, m, X, symmetric)
    Xd = bf16_tensor(X)
    assert np.array_equal(bits(fused(m, Xd, symmetric)), Yr.view(np.uint32))
    yb = fused(m, Xd, symmetric, out_dtype=tl.TL_OUT_BF16).cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(yb, oracle_mod.bf16_rne(Yr))
    m2 = Mat(oracle_mod, 512, K, seed=7)
    ys = tl.tl_linear_group([m.dev, m2.dev], Xd, mode=F,
                            flags=tl.TL_FLAG_SYMMETRIC if symmetric else 0)
    torch.cuda.synchronize()
    assert np.array_equal(bits(ys[0]), Yr.view(np.uint32))
    assert np.array_equal(bits(ys[1]), oracle_y(oracle_mod, m2, X, symmetric).view(np.uint32))
