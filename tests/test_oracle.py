"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against a hand derivation, a closed form, brute
force with numpy on tiny inputs, or an invariant of the definition
y[n,m] = scale[m] * sum_k w[m,k] * x[n,k]  ("state times scale",
"Neutrino-1: quantization is a training decision", "What's actually ternary").
"""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth
from tests.conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

SHAPES = [(16, 128), (32, 256), (5, 37), (17, 129), (1, 1), (48, 300), (128, 128), (3, 260)]


def _rand_case(M, K, seed, p0=0.626):
    W = synth.ternary(M, K, p0, seed)
    scale = synth.scales(M, seed)
    return W, scale


# ---------------------------------------------------------------- format

ZERO_WORD = np.uint32(0x55555555)     # a TL2P v2 word of sixteen zero weights


def test_layout_hand_derived_positions(oracle_mod):
    """Single non-zero weights land on the hand-derived word and bits."""
    for M, K, m, k, w, wi, val in read_golden("tl2p_layout.txt"):
        M, K, m, k, w, wi = map(int, (M, K, m, k, w, wi))
        W = np.zeros((M, K), dtype=np.int8)
        W[m, k] = w
        P = oracle_mod.pack(W)
        assert P.size == ((M + 15) // 16 * 16) * ((K + 127) // 128 * 128) // 16
        nz = np.flatnonzero(P != ZERO_WORD)
        assert list(nz) == [wi], (M, K, m, k, nz)
        assert int(P[wi]) == int(val, 16), (M, K, m, k, hex(int(P[wi])))
        back, bad = oracle_mod.unpack(P, M, K)
        assert bad == 0 and np.array_equal(back, W)


def test_layout_is_a_bijection(oracle_mod):
    """Every (row, column) of a full tile owns a distinct 2-bit field."""
    M, K = 16, 128
    seen = set()
    for m in range(M):
        for k in range(K):
            W = np.zeros((M, K), dtype=np.int8)
            W[m, k] = -1
            P = oracle_mod.pack(W)
            (wi,) = np.flatnonzero(P != ZERO_WORD)
            bits = int(P[wi]) ^ int(ZERO_WORD)       # field 01 -> 10
            assert bin(bits).count("1") == 2
            lo = (bits & -bits).bit_length() - 1
            assert lo % 2 == 0 and bits == (3 << lo)
            seen.add((int(wi), lo))
    assert len(seen) == M * K


@pytest.mark.parametrize("M,K", SHAPES)
def test_pack_unpack_roundtrip(oracle_mod, M, K):
    W, _ = _rand_case(M, K, seed=M * 1000 + K)
    P = oracle_mod.pack(W)
    back, bad = oracle_mod.unpack(P, M, K)
    assert bad == 0
    assert np.array_equal(back, W)


def test_pack_rejects_values_outside_ternary(oracle_mod):
    W = np.zeros((4, 8), dtype=np.int8)
    W[2, 3] = 2
    with pytest.raises(ValueError):
        oracle_mod.pack(W)
    W[2, 3] = -2
    with pytest.raises(ValueError):
        oracle_mod.pack(W)


def test_invalid_code_decodes_to_zero_and_is_counted(oracle_mod):
    W = np.zeros((16, 128), dtype=np.int8)
    P = oracle_mod.pack(W)
    P[0] |= np.uint32(0x3)             # field 11
    back, bad = oracle_mod.unpack(P, 16, 128)
    assert bad == 1 and not back.any()


def test_padding_must_stay_zero(oracle_mod):
    W = np.ones((5, 37), dtype=np.int8)
    P = oracle_mod.pack(W)
    _, bad = oracle_mod.unpack(P, 5, 37)
    assert bad == 0
    P2 = P.copy()
    P2[-1] ^= np.uint32(0x40000000)    # row 15 / far column: padding 01 -> 00 (+1)
    _, bad = oracle_mod.unpack(P2, 5, 37)
    assert bad == 1


@pytest.mark.parametrize("M,K", SHAPES)
def test_rowsum_three_ways(oracle_mod, M, K):
    W, _ = _rand_case(M, K, seed=7 + M + K)
    P = oracle_mod.pack(W)
    rs = oracle_mod.rowsum(P, M, K)
    assert np.array_equal(rs, W.astype(np.int64).sum(axis=1))
    # position-free popcount identity over the whole matrix: each field is
    # 1 - w with its low bit on an even position; +1 = 00, 0 = 01, -1 = 10.
    words = P.astype(np.uint64)
    lo = words & 0x55555555
    hi = (words >> 1) & 0x55555555
    plus = sum(bin(int(v)).count("1") for v in (~lo & ~hi & 0x55555555))
    minus = sum(bin(int(v)).count("1") for v in (hi & ~lo & 0x55555555))
    assert plus - minus == int(rs.sum())
    assert plus == int((W == 1).sum()) and minus == int((W == -1).sum())


# ---------------------------------------------------------------- mode A

def _x(N, K, seed, **kw):
    return synth.activations(N, K, seed, **kw)


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("N", [1, 3, 8])
def test_linear_a_matches_dense_bruteforce(oracle_mod, M, K, N):
    """Mode A equals numpy's float64 dense product on the unpacked weights."""
    W, scale = _rand_case(M, K, seed=11 * M + K)
    X = _x(N, K, seed=M + 3 * K + N)
    P = oracle_mod.pack(W)
    Y, S = oracle_mod.linear_a(P, scale, M, K, X, return_sums=True)
    xf = synth.bf16_bits_to_f32(X).astype(np.float64)
    dense = xf @ W.astype(np.float64).T          # [N, M], exact at these sizes
    assert np.array_equal(S, dense)
    ref = (dense * scale.astype(np.float64)[None, :]).astype(np.float32)
    assert np.array_equal(Y, ref)


def test_linear_a_closed_forms(oracle_mod):
    M, K = 37, 300
    W, scale = _rand_case(M, K, seed=5)
    W[3, :] = 0                                     # an all-zero row
    P = oracle_mod.pack(W)
    # one-hot activations: y = scale * w[m, k] * v (a single term)
    k, v = 201, 1.5
    X = np.zeros((1, K), dtype=np.float32)
    X[0, k] = v
    Y = oracle_mod.linear_a(P, scale, M, K, synth.to_bf16_bits(X))
    expect = (scale.astype(np.float64) * W[:, k] * v).astype(np.float32)
    assert np.array_equal(Y[0], expect)
    # all-ones activations: y = scale * rowsum
    X1 = synth.to_bf16_bits(np.ones((1, K), dtype=np.float32))
    Y1 = oracle_mod.linear_a(P, scale, M, K, X1)
    rs = W.astype(np.int64).sum(axis=1)
    assert np.array_equal(Y1[0], (scale.astype(np.float64) * rs).astype(np.float32))
    # the zero row gives exactly 0 for any input
    Xr = _x(4, K, seed=9)
    Yr = oracle_mod.linear_a(P, scale, M, K, Xr)
    assert np.all(Yr[:, 3] == 0.0)


def test_linear_a_is_linear(oracle_mod):
    """Exact sums are additive: S(x1 + x2) = S(x1) + S(x2) for exact inputs."""
    M, K = 40, 256
    W, scale = _rand_case(M, K, seed=21)
    P = oracle_mod.pack(W)
    rng = np.random.default_rng(3)
    a = rng.integers(-64, 64, size=(2, K)).astype(np.float32)
    b = rng.integers(-64, 64, size=(2, K)).astype(np.float32)
    _, Sa = oracle_mod.linear_a(P, scale, M, K, synth.to_bf16_bits(a), return_sums=True)
    _, Sb = oracle_mod.linear_a(P, scale, M, K, synth.to_bf16_bits(b), return_sums=True)
    _, Sab = oracle_mod.linear_a(P, scale, M, K, synth.to_bf16_bits(a + b), return_sums=True)
    assert np.array_equal(Sab, Sa + Sb)


def test_linear_a_row_independence(oracle_mod):
    """Rows of a 16-row panel computed alone equal the same rows in the whole."""
    M, K = 64, 384
    W, scale = _rand_case(M, K, seed=33)
    X = _x(2, K, seed=4)
    Y = oracle_mod.linear_a(oracle_mod.pack(W), scale, M, K, X)
    P = oracle_mod.pack(W)
    words_per_panel = (K + 127) // 128 * 128
    panel = 2
    Pp = P[panel * words_per_panel:(panel + 1) * words_per_panel]
    Yp = oracle_mod.linear_a(Pp, scale[32:48], 16, K, X)
    assert np.array_equal(Yp, Y[:, 32:48])


# ---------------------------------------------------------------- quant

def test_quant_one_hot_closed_form(oracle_mod):
    K = 512
    for v in (0.75, 3.0, 20.0, 1e-3):
        X = np.zeros((1, K), dtype=np.float32)
        X[0, 17] = v
        Q, s, z = oracle_mod.quant(synth.to_bf16_bits(X))
        assert z[0] == -128
        assert Q[0, 17] == 127
        assert np.all(np.delete(Q[0], 17) == -128)
        vb = float(synth.bf16_bits_to_f32(synth.to_bf16_bits(np.float32([v])))[0])
        assert abs(float(s[0]) * 255.0 - vb) <= 2 * np.spacing(np.float32(vb))


def test_quant_degenerate_zero_token(oracle_mod):
    Q, s, z = oracle_mod.quant(np.zeros((2, 64), dtype=np.uint16))
    assert np.all(Q == 0) and np.all(s == 1.0) and np.all(z == 0)
    Q, s, z = oracle_mod.quant(np.zeros((2, 64), dtype=np.uint16), symmetric=True)
    assert np.all(Q == 0) and np.all(s == 1.0) and np.all(z == 0)


def test_quant_ties_round_to_even(oracle_mod):
    """Hand-derived: with x/s landing exactly on k + 1/2, q rounds to even.

    Asymmetric: a token whose largest value is 255 and smallest is 0 has
    lo = 0, hi = 255, s = 255/255 = 1 exactly and z = -128 - rint(0) = -128,
    so q = rint(x) - 128: 2.5 -> 2 - 128, 0.5 -> 0 - 128, 1.5 -> 2 - 128,
    -> never 3 - 128 or 1 - 128 as rounding half away from zero would give.
    Symmetric: max|x| = 127 gives s = 127/127 = 1, q = rint(x) with no
    offset: 2.5 -> 2, -2.5 -> -2, 0.5 -> 0, -0.5 -> 0, 1.5 -> 2, -1.5 -> -2.
    (Reading: the pages are silent on activation rounding; ties go to even,
    as for every other rounding in the library.)"""
    K = 64
    x = np.zeros((1, K), dtype=np.float32)
    x[0, :6] = [255.0, 2.5, 0.5, 1.5, 3.5, 4.5]
    Q, s, z = oracle_mod.quant(synth.to_bf16_bits(x))
    assert float(s[0]) == 1.0 and int(z[0]) == -128
    assert list(Q[0, :6]) == [127, 2 - 128, 0 - 128, 2 - 128, 4 - 128, 4 - 128]
    assert np.all(Q[0, 6:] == -128)

    xs = np.zeros((1, K), dtype=np.float32)
    xs[0, :7] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5]
    Q, s, z = oracle_mod.quant(synth.to_bf16_bits(xs), symmetric=True)
    assert float(s[0]) == 1.0 and int(z[0]) == 0
    assert list(Q[0, :7]) == [127, 2, -2, 0, 0, 2, -2]


def test_quant_range_includes_zero(oracle_mod):
    """Hand-derived closed forms for one-signed tokens (the range is widened
    to include 0, so zero stays exactly representable).

    All positive (min x > 0): lo = 0, so z = -128 exactly, s = fl(max/255)
    and the largest value maps to rint(max/s) - 128 = 255 - 128 = 127.
    All negative (max x < 0): hi = 0, s = fl(-min/255), z = -128 - rint(min/s)
    = -128 + 255 = 127, and the smallest value maps to -255 + 127 = -128."""
    rng = np.random.default_rng(5)
    K = 300
    for _ in range(4):
        pos = rng.uniform(0.25, 4.0, size=(1, K)).astype(np.float32)
        bits = synth.to_bf16_bits(pos)
        vals = synth.bf16_bits_to_f32(bits)
        Q, s, z = oracle_mod.quant(bits)
        vmax = np.float32(vals.max())
        assert int(z[0]) == -128
        assert float(s[0]) == float(np.float32(vmax / np.float32(255.0)))
        assert Q[0, int(np.argmax(vals))] == 127
        assert Q.min() > -128          # nothing maps below the zero point's code

        bits_n = synth.to_bf16_bits(-pos)
        vals_n = synth.bf16_bits_to_f32(bits_n)
        Q, s, z = oracle_mod.quant(bits_n)
        vmin = np.float32(vals_n.min())
        assert int(z[0]) == 127
        assert float(s[0]) == float(np.float32(np.float32(0.0 - vmin) / np.float32(255.0)))
        assert Q[0, int(np.argmin(vals_n))] == -128
        assert Q.max() < 127


def test_threaded_oracle_equals_single_thread(oracle_mod):
    """The host-core timing drivers compute exactly the single-thread rows."""
    M, K = 77, 1000
    W, scale = _rand_case(M, K, seed=44)
    P = oracle_mod.pack(W)
    rs = oracle_mod.rowsum(P, M, K)
    X = _x(3, K, seed=45, outlier_frac=0.01)
    ya = oracle_mod.linear_a(P, scale, M, K, X)
    for nt in (1, 3, 8):
        assert np.array_equal(oracle_mod.linear_a_mt(P, scale, M, K, X, nthreads=nt), ya)
    Q, s, z = oracle_mod.quant(X)
    _, yb = oracle_mod.linear_b(P, scale, rs, M, K, Q, s, z)
    for nt in (1, 3, 8):
        assert np.array_equal(oracle_mod.linear_b_mt(P, scale, rs, M, K, Q, s, z, nthreads=nt), yb)


@pytest.mark.parametrize("symmetric", [False, True])
def test_quant_properties(oracle_mod, symmetric):
    X = _x(8, 1000, seed=2, outlier_frac=0.01)
    Q, s, z = oracle_mod.quant(X, symmetric=symmetric)
    xf = synth.bf16_bits_to_f32(X).astype(np.float64)
    deq = (Q.astype(np.float64) - z[:, None]) * s[:, None].astype(np.float64)
    err = np.abs(deq - xf)
    # unclamped entries are within half a step, up to fp32 rounding of x/s
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-5) + 1e-30)
    if symmetric:
        assert np.all(z == 0)
        amax = np.abs(xf).max(axis=1)
        assert np.allclose(s, amax / 127.0, rtol=1e-6)
        assert np.all(np.abs(Q).max(axis=1) == 127)
        assert Q.min() >= -127
    else:
        # zero is exact: x = 0 maps to q = z; the minimum maps to -128
        lo = xf.min(axis=1)
        for n in range(8):
            assert Q[n, np.argmin(xf[n])] == -128 or lo[n] == 0
        assert np.all((z >= -128) & (z <= 127))
        Xz = X.copy()
        Xz[:, 5] = 0
        Qz, _, zz = oracle_mod.quant(Xz)
        assert np.all(Qz[:, 5] == zz)


# ---------------------------------------------------------------- mode B

@pytest.mark.parametrize("M,K", SHAPES)
def test_linear_b_integer_sums_match_numpy(oracle_mod, M, K):
    W, scale = _rand_case(M, K, seed=M + 99 * K)
    X = _x(5, K, seed=K)
    Q, s, z = oracle_mod.quant(X)
    P = oracle_mod.pack(W)
    rs = oracle_mod.rowsum(P, M, K)
    acc, Y = oracle_mod.linear_b(P, scale, rs, M, K, Q, s, z)
    assert np.array_equal(acc, Q.astype(np.int64) @ W.astype(np.int64).T)


def test_linear_b_one_hot_identity(oracle_mod):
    """One-hot x: acc - z*rowsum = 255*w[m,k] (q = 127 there, -128 elsewhere)."""
    M, K = 50, 256
    W, scale = _rand_case(M, K, seed=8)
    P = oracle_mod.pack(W)
    rs = oracle_mod.rowsum(P, M, K)
    X = np.zeros((1, K), dtype=np.float32)
    X[0, 77] = 2.5
    Q, s, z = oracle_mod.quant(synth.to_bf16_bits(X))
    acc, Y = oracle_mod.linear_b(P, scale, rs, M, K, Q, s, z)
    corrected = acc[0].astype(np.int64) - int(z[0]) * rs.astype(np.int64)
    assert np.array_equal(corrected, 255 * W[:, 77].astype(np.int64))
    # and y is within two fp32 roundings of scale * w * v
    ref = scale.astype(np.float64) * W[:, 77] * 2.5
    assert np.all(np.abs(Y[0] - ref) <= 4 * np.spacing(np.abs(ref).astype(np.float32)) + 0)


@pytest.mark.parametrize("symmetric", [False, True])
def test_linear_b_tracks_linear_a_within_quant_error(oracle_mod, symmetric):
    """|y_B - y_A| <= scale * sum_k |w| * s / 2 (+ fp32 rounding): pins the
    sign of the zero-point correction and the order of the epilogue."""
    M, K = 64, 1024
    W, scale = _rand_case(M, K, seed=17)
    X = _x(6, K, seed=18, outlier_frac=0.01)
    P = oracle_mod.pack(W)
    rs = oracle_mod.rowsum(P, M, K)
    Q, s, z = oracle_mod.quant(X, symmetric=symmetric)
    _, YB = oracle_mod.linear_b(P, scale, rs, M, K, Q, s, z)
    YA = oracle_mod.linear_a(P, scale, M, K, X)
    absw = np.abs(W).sum(axis=1).astype(np.float64)
    bound = scale[None, :].astype(np.float64) * absw[None, :] * (s[:, None] / 2) * (1 + 1e-4)
    bound += 1e-6 * np.abs(YA)
    assert np.all(np.abs(YB.astype(np.float64) - YA) <= bound)


def test_bf16_rne_matches_hand_values(oracle_mod):
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6: even (1 + 2^-6) wins.
    vals = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, -2.0, 0.0, 65504.0], dtype=np.float32)
    out = oracle_mod.bf16_rne(vals)
    assert list(out) == [0x3F80, 0x3F80, 0x3F82, 0xC000, 0x0000, 0x4780]


# ---------------------------------------------------------------- int8 head and embedding

def _head_case(V, D, seed):
    rng = np.random.default_rng(seed)
    H = rng.integers(-128, 128, size=(V, D)).astype(np.int8)
    scale = rng.uniform(0.005, 0.05, size=V).astype(np.float32)
    return H, scale


@pytest.mark.parametrize("V,D,N", [(37, 64, 1), (100, 160, 3), (5, 16, 8)])
def test_head_integer_sums_and_argmax(oracle_mod, V, D, N):
    """acc is numpy's int64 Q @ H^T; the fused argmax is numpy's argmax
    (first occurrence) over the oracle's own logits."""
    H, scale = _head_case(V, D, V + D)
    X = _x(N, D, seed=D)
    Q, s, z = oracle_mod.quant(X)
    acc, lg, tok, best = oracle_mod.head(H, scale, Q, s, z)
    assert np.array_equal(acc, Q.astype(np.int64) @ H.astype(np.int64).T)
    assert np.array_equal(tok, np.argmax(lg, axis=1))
    assert np.array_equal(best, lg[np.arange(N), tok])


def test_head_ties_go_to_the_smallest_index(oracle_mod):
    """Two identical rows that both hold the largest logit: the smaller index."""
    V, D = 50, 64
    H, scale = _head_case(V, D, 3)
    for a, b in ((7, 31), (0, V - 1), (12, 13)):
        Hc, sc = H.copy(), scale.copy()
        Hc[a] = Hc[b] = 127
        sc[a] = sc[b] = 1.0
        X = synth.to_bf16_bits(np.abs(_f(_x(2, D, seed=a))) + 0.5)
        Q, s, z = oracle_mod.quant(X)
        _, lg, tok, _ = oracle_mod.head(Hc, sc, Q, s, z)
        assert lg[0, a] == lg[0, b] == lg.max(axis=1)[0]
        assert list(tok) == [a, a]


def _f(bits):
    return synth.bf16_bits_to_f32(bits)


def test_head_tracks_the_dense_product(oracle_mod):
    """|logit - scale * sum_d H x| <= scale * sum_d |H| * s / 2 (+ rounding):
    pins the zero-point sign and the epilogue order against a float64
    product of the unquantised activations."""
    V, D = 64, 256
    H, scale = _head_case(V, D, 11)
    X = _x(4, D, seed=12, outlier_frac=0.01)
    Q, s, z = oracle_mod.quant(X)
    _, lg, _, _ = oracle_mod.head(H, scale, Q, s, z)
    dense = _f(X).astype(np.float64) @ H.astype(np.float64).T * scale[None, :].astype(np.float64)
    bound = (scale[None, :].astype(np.float64) * np.abs(H).sum(axis=1)[None, :]
             * (s[:, None] / 2) * (1 + 1e-4) + 1e-6 * np.abs(dense))
    assert np.all(np.abs(lg - dense) <= bound)


def test_head_one_hot_closed_form(oracle_mod):
    """One-hot x = v e_k: q_k = 127, the rest -128, z = -128, so
    acc - z * rowsum = 255 * H[:, k] and logit = scale * H[:, k] * v up to
    fp32 rounding."""
    V, D = 40, 128
    H, scale = _head_case(V, D, 21)
    x = np.zeros((1, D), dtype=np.float32)
    x[0, 70] = 2.5
    Q, s, z = oracle_mod.quant(synth.to_bf16_bits(x))
    acc, lg, tok, _ = oracle_mod.head(H, scale, Q, s, z)
    rs = H.astype(np.int64).sum(axis=1)
    assert np.array_equal(acc[0].astype(np.int64) + 128 * rs, 255 * H[:, 70].astype(np.int64))
    ref = scale.astype(np.float64) * H[:, 70] * 2.5
    assert np.all(np.abs(lg[0] - ref) <= 4 * np.spacing(np.abs(ref).astype(np.float32)))
    assert tok[0] == int(np.argmax(ref))


def test_embed_rows_times_scale(oracle_mod):
    """Powers-of-two scales give exact products (closed form); other scales
    give the bf16 (ties to even) of the fp32 product."""
    V, D = 30, 48
    rng = np.random.default_rng(4)
    E = rng.integers(-128, 128, size=(V, D)).astype(np.int8)
    scale = (2.0 ** rng.integers(-8, 3, size=V)).astype(np.float32)
    toks = np.array([3, 29, 0, 3], dtype=np.int32)
    X = oracle_mod.embed(E, scale, toks)
    exact = E[toks].astype(np.float64) * scale[toks, None]
    assert np.array_equal(_f(X).astype(np.float64), exact)
    scale2 = rng.uniform(0.001, 0.1, size=V).astype(np.float32)
    X2 = oracle_mod.embed(E, scale2, toks)
    prod = E[toks].astype(np.float32) * scale2[toks, None]
    assert np.array_equal(X2, synth.to_bf16_bits(prod))


# ---------------------------------------------------------------- RMSNorm and SwiGLU

def test_rmsnorm_identities(oracle_mod):
    """mean_k (y/gamma)^2 = ms / (ms + eps); y scales with gamma; a constant
    row c gives gamma * c / sqrt(c^2 + eps); y(alpha x) = y(x) up to eps."""
    N, K = 4, 512
    X = _x(N, K, seed=31)
    rng = np.random.default_rng(32)
    gamma = synth.to_bf16_bits(rng.uniform(0.5, 2.0, size=K).astype(np.float32))
    eps = 1e-6
    Y = oracle_mod.rmsnorm(X, gamma, eps)
    xf = _f(X).astype(np.float64)
    gf = _f(gamma).astype(np.float64)
    ms = (xf ** 2).mean(axis=1)
    assert np.allclose(((Y / gf) ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12)
    assert np.allclose(Y / gf, xf / np.sqrt(ms + eps)[:, None], rtol=1e-13)
    c = synth.to_bf16_bits(np.full((1, K), 3.0, dtype=np.float32))
    ones = synth.to_bf16_bits(np.ones(K, dtype=np.float32))
    assert np.allclose(oracle_mod.rmsnorm(c, ones, eps), 3.0 / np.sqrt(9.0 + eps), rtol=1e-14)
    X2 = synth.to_bf16_bits(4.0 * xf.astype(np.float32))      # exact (power of two)
    assert np.allclose(oracle_mod.rmsnorm(X2, gamma, 0.0), oracle_mod.rmsnorm(X, gamma, 0.0),
                       rtol=1e-13)


def test_swiglu_identities(oracle_mod):
    """silu(g) - silu(-g) = g (so with u = 1 the two halves sum to g);
    silu(0) = 0; u = 0 gives 0; silu(g) -> g for large g, -> 0 for very
    negative g."""
    rng = np.random.default_rng(33)
    g = rng.standard_normal((3, 300)).astype(np.float32) * 4
    G = synth.to_bf16_bits(g)
    ones = synth.to_bf16_bits(np.ones_like(g))
    h_pos = oracle_mod.swiglu(G, ones)
    h_neg = oracle_mod.swiglu(synth.to_bf16_bits(-_f(G)), ones)
    assert np.allclose(h_pos - h_neg, _f(G).astype(np.float64), rtol=1e-13, atol=1e-15)
    z = synth.to_bf16_bits(np.zeros((1, 8), dtype=np.float32))
    assert not oracle_mod.swiglu(z, synth.to_bf16_bits(np.ones((1, 8), np.float32))).any()
    assert not oracle_mod.swiglu(G, synth.to_bf16_bits(np.zeros_like(g))).any()
    big = synth.to_bf16_bits(np.float32([[60.0, -60.0]]))
    h = oracle_mod.swiglu(big, synth.to_bf16_bits(np.float32([[1.0, 1.0]])))
    assert abs(h[0, 0] - 60.0) < 1e-20 and abs(h[0, 1]) < 1e-24


# ---------------------------------------------------------------- block scales

def test_absmean_closed_forms(oracle_mod):
    """Hand-derived blocks.  +-c everywhere: scale c, codes sign(w).  60 ones
    and 16 quarters (+-) in 128 columns: scale (60 + 4) / 128 = 0.5 exactly,
    ones give 2 -> clamped to 1, quarters give +-0.5 -> ties to even: 0.
    A short last block (44 columns) has its own mean.  Zeros: scale 0,
    codes 0."""
    M, K = 3, 300                       # blocks of 128, 128 and 44 columns
    W = np.zeros((M, K), dtype=np.float32)
    rng = np.random.default_rng(1)
    W[0] = np.where(rng.random(K) < 0.5, 2.0, -2.0)
    W[1, :60] = 1.0
    W[1, 60:68] = 0.25
    W[1, 68:76] = -0.25
    W[1, 256:300] = 3.0                 # the 44-column block: scale 3, codes 1
    W[1, 299] = -3.0
    T, bs = oracle_mod.absmean_ternarize(W)
    assert np.all(bs[0] == 2.0) and np.array_equal(T[0], np.sign(W[0]).astype(np.int8))
    assert bs[1].tolist() == [0.5, 0.0, 3.0]
    assert np.all(T[1, :60] == 1) and not T[1, 60:256].any()
    assert np.all(T[1, 256:299] == 1) and T[1, 299] == -1
    assert bs[2].tolist() == [0.0, 0.0, 0.0] and not T[2].any()
    T2, bs2 = oracle_mod.absmean_ternarize(np.float32([[1.0, 0.5, -0.5, 0.0]]))   # scale 0.5
    assert bs2.tolist() == [[0.5]] and T2.tolist() == [[1, 1, -1, 0]]


@pytest.mark.parametrize("M,K,N", [(16, 128, 1), (37, 300, 3), (5, 1000, 2)])
def test_blockscale_linear_matches_dense(oracle_mod, M, K, N):
    """Against numpy float64: sum over blocks of scale * (x_block @ w_block)."""
    rng = np.random.default_rng(M + K)
    Wf = rng.standard_normal((M, K)).astype(np.float32)
    T, bs = oracle_mod.absmean_ternarize(Wf)
    P = oracle_mod.pack(T)
    X = _x(N, K, seed=K)
    Y = oracle_mod.linear_blockscale(P, bs, M, K, X)
    xf = _f(X).astype(np.float64)
    ref = np.zeros((N, M))
    for b in range(bs.shape[1]):
        sl = slice(128 * b, min(K, 128 * b + 128))
        ref += (xf[:, sl] @ T[:, sl].astype(np.float64).T) * bs[:, b].astype(np.float64)[None, :]
    assert np.allclose(Y, ref, rtol=1e-6, atol=1e-30)
    # one scale for every block reduces to the per-row linear
    ones = np.ones_like(bs)
    Y1 = oracle_mod.linear_blockscale(P, ones, M, K, X)
    assert np.array_equal(Y1, oracle_mod.linear_a(P, np.ones(M, np.float32), M, K, X))
