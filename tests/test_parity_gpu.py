"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Mode B (int8 activations) must match bit for bit; mode A (bf16 activations,
fp32 sums) within 1e-3 of the oracle, relative to max(|y_ref|, 1e-2 * rms of
the token's outputs).  Every token's result must not depend on the batch.
"""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402

TOL_A = 1e-3


def rel_err(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    den = np.maximum(np.abs(ref), 1e-2 * np.maximum(rms, 1e-30))
    return float(np.max(np.abs(y - ref) / den)) if y.size else 0.0


def bf16_tensor(bits: np.ndarray):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def case(M, K, seed, p0=0.626):
    W = synth.ternary(M, K, p0, seed)
    scale = synth.scales(M, seed)
    return W, scale


class Mat:
    def __init__(self, oracle_mod, M, K, seed, p0=0.626, W=None):
        if W is None:
            W, scale = case(M, K, seed, p0)
        else:
            scale = synth.scales(M, seed)
        self.W, self.scale, self.M, self.K = W, scale, M, K
        self.P = oracle_mod.pack(W)
        self.rowsum = oracle_mod.rowsum(self.P, M, K)
        self.dev = tl.TernaryWeight.from_int8(W, scale)


def oracle_b(oracle_mod, m, X):
    Q, s, z = oracle_mod.quant(X)
    acc, Y = oracle_mod.linear_b(m.P, m.scale, m.rowsum, m.M, m.K, Q, s, z)
    return Q, s, z, acc, Y


def gpu_b(m, X, out_dtype=tl.TL_OUT_F32, symmetric=False):
    Q, s, z = tl.tl_quantize_act(bf16_tensor(X), symmetric=symmetric)
    Y = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return Q, s, z, Y


CONFIG_SHAPES = [(2048, 1024), (1024, 1024), (1024, 2048), (3072, 1024), (1024, 3072),
                 (4096, 4096), (1024, 4096), (4096, 12288)]
RAGGED = [(5, 37), (17, 129), (100, 1000), (33, 4099), (1, 1), (16, 128), (777, 333)]


@pytest.mark.parametrize("M,K", CONFIG_SHAPES + RAGGED)
@pytest.mark.parametrize("N", [1, 8])
def test_mode_a_parity(oracle_mod, M, K, N):
    m = Mat(oracle_mod, M, K, seed=M + 7 * K)
    X = synth.activations(N, K, seed=N + K)
    ref = oracle_mod.linear_a(m.P, m.scale, M, K, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert Y.shape == ref.shape
    assert rel_err(Y, ref) <= TOL_A


@pytest.mark.parametrize("N", [2, 3, 5, 6, 7])
def test_mode_a_parity_other_batches(oracle_mod, N):
    m = Mat(oracle_mod, 2048, 1024, seed=0)
    X = synth.activations(N, 1024, seed=3, outlier_frac=0.01)
    ref = oracle_mod.linear_a(m.P, m.scale, 2048, 1024, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A


@pytest.mark.parametrize("M,K", CONFIG_SHAPES + RAGGED)
@pytest.mark.parametrize("N", [1, 8])
def test_mode_b_bit_exact(oracle_mod, M, K, N):
    m = Mat(oracle_mod, M, K, seed=3 * M + K)
    X = synth.activations(N, K, seed=2 * N + K, outlier_frac=0.01)
    Qr, sr, zr, accr, Yr = oracle_b(oracle_mod, m, X)
    Q, s, z, Y = gpu_b(m, X)
    assert np.array_equal(Q.cpu().numpy(), Qr)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zr)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
    acc = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, out_dtype=tl.TL_OUT_I32_RAW)
    assert np.array_equal(acc.cpu().numpy(), accr)


def test_mode_b_bf16_output_is_rne_of_oracle(oracle_mod):
    m = Mat(oracle_mod, 1024, 4096, seed=5)
    X = synth.activations(8, 4096, seed=5)
    *_, Yr = oracle_b(oracle_mod, m, X)
    *_, Y = gpu_b(m, X, out_dtype=tl.TL_OUT_BF16)
    got = Y.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, oracle_mod.bf16_rne(Yr))


def test_mode_a_bf16_output(oracle_mod):
    m = Mat(oracle_mod, 3072, 1024, seed=6)
    X = synth.activations(4, 1024, seed=6)
    ref = oracle_mod.linear_a(m.P, m.scale, 3072, 1024, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X), out_dtype=tl.TL_OUT_BF16).float().cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A + 2.0 ** -8


@pytest.mark.parametrize("K", [1, 7, 128, 1000, 4096, 12288, 16384, 16392])
@pytest.mark.parametrize("symmetric", [False, True])
def test_quantizer_bit_exact(oracle_mod, K, symmetric):
    X = synth.activations(8, K, seed=K, outlier_frac=0.01 if K >= 100 else 0.0)
    X[3] = 0                                # an all-zero token
    if K > 5:
        X[5, :] = synth.to_bf16_bits(-np.abs(synth.bf16_bits_to_f32(X[5])))  # all <= 0
    if K >= 8:
        # exact ties of x / s (s = 1): the rounding must go to even
        X[6] = 0
        X[6, :6] = synth.to_bf16_bits(np.float32([255.0, 2.5, 0.5, 1.5, 3.5, -4.5]))
        X[7] = 0
        X[7, :7] = synth.to_bf16_bits(np.float32([127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5]))
    Qr, sr, zr = oracle_mod.quant(X, symmetric=symmetric)
    Q, s, z = tl.tl_quantize_act(bf16_tensor(X), symmetric=symmetric)
    torch.cuda.synchronize()
    assert np.array_equal(Q.cpu().numpy(), Qr)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zr)
    # the same rows from a pointer that is not 16-byte aligned (scalar loads)
    flat = bf16_tensor(np.concatenate([np.zeros(1, np.uint16), X.reshape(-1)]))[1:].view(8, K)
    Q2, s2, z2 = tl.tl_quantize_act(flat, symmetric=symmetric)
    torch.cuda.synchronize()
    assert np.array_equal(Q2.cpu().numpy(), Qr)
    assert np.array_equal(s2.cpu().numpy().view(np.uint32), sr.view(np.uint32))


@pytest.mark.parametrize("mode", [tl.TL_MODE_BF16, tl.TL_MODE_I8])
@pytest.mark.parametrize("M,K", [(4096, 4096), (1024, 12288), (777, 333)])
def test_batch_invariance(oracle_mod, mode, M, K):
    """Each token's row at N=8 is bitwise the N=1 result for that token."""
    m = Mat(oracle_mod, M, K, seed=11)
    X = bf16_tensor(synth.activations(8, K, seed=12, outlier_frac=0.01))
    if mode == tl.TL_MODE_BF16:
        Y8 = tl.tl_linear(m.dev, X)
        singles = [tl.tl_linear(m.dev, X[n:n + 1].contiguous()) for n in range(8)]
    else:
        Q, s, z = tl.tl_quantize_act(X)
        Y8 = tl.tl_linear(m.dev, Q, s, z, mode=mode)
        singles = [tl.tl_linear(m.dev, Q[n:n + 1].contiguous(), s[n:n + 1].contiguous(),
                                z[n:n + 1].contiguous(), mode=mode) for n in range(8)]
    torch.cuda.synchronize()
    Y8 = Y8.cpu().numpy().view(np.uint32)
    for n in range(8):
        assert np.array_equal(Y8[n], singles[n].cpu().numpy().view(np.uint32)[0]), n


def test_deterministic_across_runs(oracle_mod):
    m = Mat(oracle_mod, 12288, 4096, seed=13)
    X = bf16_tensor(synth.activations(8, 4096, seed=14))
    a = tl.tl_linear(m.dev, X).cpu().numpy()
    b = tl.tl_linear(m.dev, X).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("mode", [tl.TL_MODE_BF16, tl.TL_MODE_I8])
def test_group_equals_single_calls(oracle_mod, mode):
    mats = [Mat(oracle_mod, M, 4096, seed=20 + i) for i, M in enumerate((4096, 1024, 1024))]
    X = bf16_tensor(synth.activations(3, 4096, seed=21))
    if mode == tl.TL_MODE_I8:
        Q, s, z = tl.tl_quantize_act(X)
        ys = tl.tl_linear_group([m.dev for m in mats], Q, s, z, mode=mode)
        singles = [tl.tl_linear(m.dev, Q, s, z, mode=mode) for m in mats]
    else:
        ys = tl.tl_linear_group([m.dev for m in mats], X)
        singles = [tl.tl_linear(m.dev, X) for m in mats]
    Xh = X.cpu().view(torch.int16).numpy().view(np.uint16)
    for m, y, y1 in zip(mats, ys, singles):
        ref = oracle_mod.linear_a(m.P, m.scale, m.M, m.K, Xh)
        if mode == tl.TL_MODE_BF16:
            assert rel_err(y.cpu().numpy(), ref) <= TOL_A
        else:
            *_, Yr = oracle_b(oracle_mod, m, Xh)
            assert np.array_equal(y.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
            assert np.array_equal(y1.cpu().numpy().view(np.uint32), Yr.view(np.uint32))


@pytest.mark.parametrize("N", [9, 12, 20])
def test_batches_above_eight_run_in_chunks(oracle_mod, N):
    m = Mat(oracle_mod, 1024, 3072, seed=30)
    X = synth.activations(N, 3072, seed=31)
    ref = oracle_mod.linear_a(m.P, m.scale, 1024, 3072, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A
    *_, Yr = oracle_b(oracle_mod, m, X)
    *_, Yb = gpu_b(m, X)
    assert np.array_equal(Yb.cpu().numpy().view(np.uint32), Yr.view(np.uint32))


def test_zero_rows_and_one_hot(oracle_mod):
    M, K = 300, 2048
    W, _ = case(M, K, 40)
    W[17] = 0
    W[299] = 0
    m = Mat(oracle_mod, M, K, seed=40, W=W)
    X = synth.activations(8, K, seed=41)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    ref = oracle_mod.linear_a(m.P, m.scale, M, K, X)
    assert np.all(ref[:, 17] == 0) and np.all(ref[:, 299] == 0)
    assert rel_err(Y, ref) <= TOL_A            # zero rows: within the mode A bound
    *_, Yb = gpu_b(m, X)
    assert np.all(Yb.cpu().numpy()[:, [17, 299]] == 0)   # mode B: exactly zero
    oh = np.zeros((1, K), dtype=np.float32)
    oh[0, 1234] = 3.0
    Y1 = tl.tl_linear(m.dev, bf16_tensor(synth.to_bf16_bits(oh))).cpu().numpy()
    expect = (m.scale.astype(np.float64) * W[:, 1234] * 3.0).astype(np.float32)
    assert np.array_equal(Y1[0], expect)


@pytest.mark.parametrize("sign", [1, -1])
def test_adversarial_extreme_sums_stay_exact(oracle_mod, sign):
    """All weights +-1 and activations at the quantiser's extremes: the
    largest |acc| the path can meet (128 * K) must come out exact."""
    M, K = 64, 12288
    W = np.full((M, K), sign, dtype=np.int8)
    W[1::2] = -sign
    m = Mat(oracle_mod, M, K, seed=50, W=W)
    x = np.full((2, K), -1.0, dtype=np.float32)
    x[:, 0] = 1e-3                          # lo = -1, hi ~ 0: q = -128 except q[0] = 127
    X = synth.to_bf16_bits(x)
    Qr, sr, zr, accr, Yr = oracle_b(oracle_mod, m, X)
    assert np.abs(accr).max() == 128 * (K - 1) - 127
    Q, s, z, Y = gpu_b(m, X)
    acc = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, out_dtype=tl.TL_OUT_I32_RAW)
    assert np.array_equal(acc.cpu().numpy(), accr)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
    ref = oracle_mod.linear_a(m.P, m.scale, M, K, X)
    Ya = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Ya, ref) <= TOL_A


LONG_OR_TALL = [(16, 65536), (64, 49152), (100000, 128), (40, 20000)]


@pytest.mark.parametrize("M,K", LONG_OR_TALL)
def test_long_k_and_tall_shapes(oracle_mod, M, K):
    """Many K slices per row tile, or more CTAs than SMs."""
    m = Mat(oracle_mod, M, K, seed=M % 97 + K)
    X = synth.activations(3, K, seed=K, outlier_frac=0.01)
    ref = oracle_mod.linear_a(m.P, m.scale, M, K, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A
    *_, Yr = oracle_b(oracle_mod, m, X)
    *_, Yb = gpu_b(m, X)
    assert np.array_equal(Yb.cpu().numpy().view(np.uint32), Yr.view(np.uint32))


def _scaled_tokens(K, seed):
    """Tokens whose magnitudes leave [2^-60, 2^61): huge, tiny, one huge
    outlier among ordinary values, and bf16 subnormals among ordinary values."""
    base = synth.bf16_bits_to_f32(synth.activations(5, K, seed=seed))
    x = np.array(base, dtype=np.float64)
    x[0] *= 1e25
    x[1] *= 1e-25
    x[2, K // 3] = 3e20
    x[3, ::7] = 1e-39
    return synth.to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("M,K", [(1024, 4096), (300, 12288), (17, 129)])
@pytest.mark.parametrize("N", [1, 5])
def test_activations_outside_the_fixed_window(oracle_mod, M, K, N):
    m = Mat(oracle_mod, M, K, seed=M + K)
    X = _scaled_tokens(K, seed=M)[:N] if N > 1 else _scaled_tokens(K, seed=M)[1:2]
    ref = oracle_mod.linear_a(m.P, m.scale, M, K, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert np.all(np.isfinite(Y))
    assert rel_err(Y, ref) <= TOL_A


def test_workspace_is_left_zeroed(oracle_mod):
    m = Mat(oracle_mod, 4096, 4096, seed=60)
    X = bf16_tensor(synth.activations(8, 4096, seed=61))
    ws = tl.make_workspace([[m.dev]], 8)
    for _ in range(3):
        tl.tl_linear(m.dev, X, workspace=ws)
    torch.cuda.synchronize()
    nbytes = tl.tl_workspace_bytes([m.dev], 8)
    R = (4096 + 15) // 16
    front = 256 + _round256(8 * R) + _round256(R * 8 * 16 * 8)   # status, counters, exchange slots
    assert int(ws[:front].count_nonzero()) == 0
    assert nbytes <= ws.numel()


def _round256(b):
    return (b + 255) // 256 * 256


def test_calls_of_different_shapes_share_one_workspace(oracle_mod):
    """One workspace serves calls of any shapes in any order: a one-slice
    group (exchange slots), a three-slice matrix (counters and partial sums),
    a small one-slice matrix and a split-K prefill, twice over, each result
    checked against the oracle."""
    big = [Mat(oracle_mod, 12288, 4096, seed=90), Mat(oracle_mod, 12288, 4096, seed=91)]
    tall_k = Mat(oracle_mod, 4096, 12288, seed=92)
    small = Mat(oracle_mod, 1024, 4096, seed=93)
    groups = [[m.dev for m in big], [tall_k.dev], [small.dev]]
    ws = tl.make_workspace(groups + [[small.dev]], 8)
    need = max(ws.numel(), tl.tl_workspace_bytes([small.dev], 300))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    X1 = synth.activations(1, 4096, seed=94)
    X8 = synth.activations(8, 12288, seed=95)
    X3 = synth.activations(3, 4096, seed=96)
    X300 = synth.activations(300, 4096, seed=97)
    for _ in range(2):
        y_small = tl.tl_linear(small.dev, bf16_tensor(X3), workspace=ws)
        y_tall = tl.tl_linear(tall_k.dev, bf16_tensor(X8), workspace=ws)
        y_big = tl.tl_linear_group([m.dev for m in big], bf16_tensor(X1), workspace=ws)
        Q, s, z = tl.tl_quantize_act(bf16_tensor(X300))
        y_pre = tl.tl_linear(small.dev, Q, s, z, mode=tl.TL_MODE_I8, workspace=ws)
        y_small2 = tl.tl_linear(small.dev, bf16_tensor(X3), workspace=ws)
        torch.cuda.synchronize()
        assert rel_err(y_small.cpu().numpy(), oracle_mod.linear_a(small.P, small.scale, 1024, 4096, X3)) <= TOL_A
        assert rel_err(y_small2.cpu().numpy(), oracle_mod.linear_a(small.P, small.scale, 1024, 4096, X3)) <= TOL_A
        assert rel_err(y_tall.cpu().numpy(), oracle_mod.linear_a(tall_k.P, tall_k.scale, 4096, 12288, X8)) <= TOL_A
        for m, y in zip(big, y_big):
            assert rel_err(y.cpu().numpy(), oracle_mod.linear_a(m.P, m.scale, m.M, m.K, X1)) <= TOL_A
        Qr, sr, zr = oracle_mod.quant(X300)
        _, Yr = oracle_mod.linear_b(small.P, small.scale, small.rowsum, 1024, 4096, Qr, sr, zr)
        assert np.array_equal(y_pre.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
    R_big = 2 * 12288 // 16
    front = 256 + _round256(8 * R_big) + _round256(R_big * 1 * 16 * 8)
    assert int(ws[:front].count_nonzero()) == 0


def test_pdl_flag_gives_identical_results(oracle_mod):
    m = Mat(oracle_mod, 4096, 4096, seed=70)
    X = bf16_tensor(synth.activations(8, 4096, seed=71))
    a = tl.tl_linear(m.dev, X)
    b = tl.tl_linear(m.dev, X, flags=tl.TL_FLAG_PDL)
    c = tl.tl_linear(m.dev, X, flags=tl.TL_FLAG_PDL)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(a.view(torch.int32), c.view(torch.int32))


# ---------------------------------------------------------------- prefill (N >= 256, tcgen05)

PREFILL_SHAPES = [(256, 1024), (1024, 4096), (333, 1000), (4096, 12288), (128, 128), (200, 8)]


@pytest.mark.parametrize("M,K", PREFILL_SHAPES)
@pytest.mark.parametrize("N", [256, 300, 512])
def test_prefill_mode_a(oracle_mod, M, K, N):
    m = Mat(oracle_mod, M, K, seed=M + K + N)
    X = synth.activations(N, K, seed=N + 1)
    ref = oracle_mod.linear_a(m.P, m.scale, M, K, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A


@pytest.mark.parametrize("M,K", PREFILL_SHAPES)
@pytest.mark.parametrize("symmetric", [True, False])
def test_prefill_mode_b_bit_exact(oracle_mod, M, K, symmetric):
    N = 512
    m = Mat(oracle_mod, M, K, seed=2 * M + K)
    X = synth.activations(N, K, seed=7)
    Qr, sr, zr = oracle_mod.quant(X, symmetric=symmetric)
    accr, Yr = oracle_mod.linear_b(m.P, m.scale, m.rowsum, M, K, Qr, sr, zr)
    Q, s, z = tl.tl_quantize_act(bf16_tensor(X), symmetric=symmetric)
    ws = tl.make_workspace([[m.dev]], N)
    Y = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, workspace=ws)
    acc = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, out_dtype=tl.TL_OUT_I32_RAW,
                       workspace=ws)
    Yb = tl.tl_linear(m.dev, Q, s, z, mode=tl.TL_MODE_I8, out_dtype=tl.TL_OUT_BF16, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), accr)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
    got = Yb.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, oracle_mod.bf16_rne(Yr))
    R = (M + 15) // 16
    assert int(ws[: 256 + 8 * R].count_nonzero()) == 0   # status word + decode counters untouched


@pytest.mark.parametrize("Ms", [(4096, 1024, 1024), (1024, 1024, 1024)])
def test_prefill_group_and_workspace_shared_with_decode(oracle_mod, Ms):
    """A prefill call and decode calls may share one workspace in any order
    (the second group is small enough that the prefill splits K)."""
    mats = [Mat(oracle_mod, M, 4096, seed=80 + i) for i, M in enumerate(Ms)]
    ws = tl.make_workspace([[m.dev for m in mats]], 512)
    ws = torch.zeros(max(ws.numel(), tl.tl_workspace_bytes([m.dev for m in mats], 8)),
                     dtype=torch.uint8, device="cuda")
    X512 = synth.activations(512, 4096, seed=81)
    X8 = synth.activations(8, 4096, seed=82)
    for _ in range(2):
        Q, s, z = tl.tl_quantize_act(bf16_tensor(X512))
        ys = tl.tl_linear_group([m.dev for m in mats], Q, s, z, mode=tl.TL_MODE_I8, workspace=ws)
        y8 = tl.tl_linear_group([m.dev for m in mats], bf16_tensor(X8), workspace=ws)
        torch.cuda.synchronize()
        for m, y, yd in zip(mats, ys, y8):
            Qr, sr, zr = oracle_mod.quant(X512)
            _, Yr = oracle_mod.linear_b(m.P, m.scale, m.rowsum, m.M, m.K, Qr, sr, zr)
            assert np.array_equal(y.cpu().numpy().view(np.uint32), Yr.view(np.uint32))
            ref8 = oracle_mod.linear_a(m.P, m.scale, m.M, m.K, X8)
            assert rel_err(yd.cpu().numpy(), ref8) <= TOL_A


# ---------------------------------------------------------------- inputs of one sign
# The mode-A kernel sums (1 - w) x with the tensor cores and removes sum x;
# activations of one sign are where the rounding of those partial sums is
# largest compared with the result, so they are checked on their own.

def _one_signed(N, K, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "abs_normal":
        x = np.abs(rng.standard_normal((N, K)))
    elif kind == "lognormal":
        x = rng.lognormal(0.0, 1.5, size=(N, K))
    else:                                      # all negative, SwiGLU-like tail
        x = -np.abs(rng.standard_normal((N, K))) * 0.3
    return synth.to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("kind", ["abs_normal", "lognormal", "negative"])
@pytest.mark.parametrize("K", [4096, 12288])
@pytest.mark.parametrize("N", [1, 8])
def test_mode_a_one_signed_activations(oracle_mod, kind, K, N):
    M = 2048
    m = Mat(oracle_mod, M, K, seed=K + N)
    X = _one_signed(N, K, kind, seed=K * 3 + N)
    ref = oracle_mod.linear_a_mt(m.P, m.scale, M, K, X)
    Y = tl.tl_linear(m.dev, bf16_tensor(X)).cpu().numpy()
    assert rel_err(Y, ref) <= TOL_A


# ---------------------------------------------------------------- the groups the bench runs

def _stack_group(oracle_mod, names, seed):
    shp = synth.NEUTRINO_8B.linear_shapes()
    return [Mat(oracle_mod, shp[p][0], shp[p][1], seed=seed + i,
                p0=synth.zero_fraction(synth.NEUTRINO_8B, 2, p)) for i, p in enumerate(names)]


@pytest.mark.parametrize("names", [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)])
@pytest.mark.parametrize("N", [1, 8])
def test_bench_launch_groups_against_oracle(oracle_mod, names, N):
    """The four launches of an 8B layer at the batch sizes the bench times,
    in both modes, as one grouped call each (mode B bit for bit)."""
    mats = _stack_group(oracle_mod, names, seed=500 + 10 * N)
    K = mats[0].K
    X = synth.activations(N, K, seed=501 + N, outlier_frac=0.01 if N == 8 else 0.0)
    xd = bf16_tensor(X)
    ys = tl.tl_linear_group([m.dev for m in mats], xd, flags=tl.TL_FLAG_PDL)
    Q, s, z = tl.tl_quantize_act(xd)
    yb = tl.tl_linear_group([m.dev for m in mats], Q, s, z, mode=tl.TL_MODE_I8)
    torch.cuda.synchronize()
    Qr, sr, zr = oracle_mod.quant(X)
    assert np.array_equal(Q.cpu().numpy(), Qr)
    for m, y, y8 in zip(mats, ys, yb):
        ref = oracle_mod.linear_a_mt(m.P, m.scale, m.M, m.K, X)
        assert rel_err(y.cpu().numpy(), ref) <= TOL_A
        refb = oracle_mod.linear_b_mt(m.P, m.scale, m.rowsum, m.M, m.K, Qr, sr, zr)
        assert np.array_equal(y8.cpu().numpy().view(np.uint32), refb.view(np.uint32))


# ---------------------------------------------------------------- dependent launches

@pytest.mark.parametrize("mode", [tl.TL_MODE_BF16, tl.TL_MODE_I8])
@pytest.mark.parametrize("N", [1, 8])
def test_chained_pdl_launches_in_a_graph(oracle_mod, mode, N):
    """Eight 4096 x 4096 linears, each reading the bf16 output the previous
    one wrote, launched with the programmatic-dependent flag and replayed
    from a CUDA graph.  Every output is checked against the oracle applied to
    the GPU's own previous output, so a launch that read its input before the
    previous one finished writing it would show."""
    L, K = 8, 4096
    mats = [Mat(oracle_mod, K, K, seed=600 + i) for i in range(L)]
    x0 = synth.activations(N, K, seed=601)
    xs = [bf16_tensor(x0)] + [torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
                              for _ in range(L)]
    qs = [(torch.empty((N, K), dtype=torch.int8, device="cuda"),
           torch.empty(N, dtype=torch.float32, device="cuda"),
           torch.empty(N, dtype=torch.int32, device="cuda")) for _ in range(L)]
    ws = tl.make_workspace([[m.dev] for m in mats], N)

    def run():
        for i, m in enumerate(mats):
            if mode == tl.TL_MODE_I8:
                q, s, z = qs[i]
                tl.tl_quantize_act(xs[i], Q=q, s=s, z=z)
                tl.tl_linear(m.dev, q, s, z, out=xs[i + 1], mode=mode, out_dtype=tl.TL_OUT_BF16,
                             workspace=ws, flags=tl.TL_FLAG_PDL)
            else:
                tl.tl_linear(m.dev, xs[i], out=xs[i + 1], out_dtype=tl.TL_OUT_BF16,
                             workspace=ws, flags=tl.TL_FLAG_PDL)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for rep in range(2):
        for t in xs[1:]:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for i, m in enumerate(mats):
            xin = xs[i].cpu().view(torch.int16).numpy().view(np.uint16)
            got = xs[i + 1].cpu().view(torch.int16).numpy().view(np.uint16)
            if mode == tl.TL_MODE_I8:
                Qr, sr, zr = oracle_mod.quant(xin)
                refb = oracle_mod.linear_b_mt(m.P, m.scale, m.rowsum, K, K, Qr, sr, zr)
                assert np.array_equal(got, oracle_mod.bf16_rne(refb)), (rep, i)
            else:
                ref = oracle_mod.linear_a_mt(m.P, m.scale, K, K, xin)
                y = synth.bf16_bits_to_f32(got)
                assert rel_err(y, ref) <= TOL_A + 2.0 ** -8, (rep, i)
