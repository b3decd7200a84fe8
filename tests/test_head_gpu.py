"""GPU: the int8 output head with its fused argmax, and the embedding lookup,
through the C ABI, against the CPU oracle.

The head's sums are exact integers and its epilogue is the same two fp32
products on both sides, so logits, chosen tokens and their logits must match
the oracle bit for bit.
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

VOCAB, HIDDEN = 151_936, 4096      # model page "Neutrino-1 8B", "Architecture"


def _table(V, D, seed):
    rng = np.random.default_rng(seed)
    H = rng.integers(-128, 128, size=(V, D), dtype=np.int16).astype(np.int8)
    scale = rng.uniform(0.005, 0.05, size=V).astype(np.float32)
    return H, scale


def _run(head, X):
    Q, s, z = tl.tl_quantize_act(bf16_tensor(X))
    N = X.shape[0]
    logits = torch.empty((N, head.V), dtype=torch.float32, device="cuda")
    tok, best = head.argmax(Q, s, z, logits=logits)
    tok2, best2 = head.argmax(Q, s, z)                  # without writing the logits
    torch.cuda.synchronize()
    return (Q.cpu().numpy(), s.cpu().numpy(), z.cpu().numpy(), logits.cpu().numpy(),
            tok.cpu().numpy(), best.cpu().numpy(), tok2.cpu().numpy(), best2.cpu().numpy())


@pytest.mark.parametrize("V,D", [(1000, 4096), (37, 16), (5003, 144), (300, 1024), (2049, 512)])
@pytest.mark.parametrize("N", [1, 3, 4, 5, 8])
def test_head_matches_oracle_bit_for_bit(oracle_mod, V, D, N):
    H, scale = _table(V, D, V + D)
    head = tl.Head.from_host(H, scale)
    X = synth.activations(N, D, seed=V + N, outlier_frac=0.01 if D >= 100 else 0.0)
    Q, s, z, lg, tok, best, tok2, best2 = _run(head, X)
    acc_r, lg_r, tok_r, best_r = oracle_mod.head(H, scale, Q, s, z)
    assert np.array_equal(lg.view(np.uint32), lg_r.view(np.uint32))
    assert np.array_equal(tok, tok_r) and np.array_equal(tok2, tok_r)
    assert np.array_equal(best.view(np.uint32), best_r.view(np.uint32))
    assert np.array_equal(best2.view(np.uint32), best_r.view(np.uint32))
    ws = head.workspace(N)
    assert int(ws[:512].count_nonzero()) == 0          # status word and counter


def test_head_ties_and_extreme_positions(oracle_mod):
    """Identical best rows give the smaller index, wherever they sit."""
    V, D = 4096, 256
    H, scale = _table(V, D, 5)
    X = synth.to_bf16_bits(np.abs(synth.bf16_bits_to_f32(synth.activations(2, D, seed=6))) + 0.5)
    for a, b in ((0, V - 1), (V - 2, V - 1), (1000, 3000), (2047, 2048)):
        Hc, sc = H.copy(), scale.copy()
        Hc[a] = Hc[b] = 127
        sc[a] = sc[b] = 1.0
        head = tl.Head.from_host(Hc, sc)
        Q, s, z, lg, tok, best, _, _ = _run(head, X)
        _, _, tok_r, best_r = oracle_mod.head(Hc, sc, Q, s, z, return_logits=False)
        assert list(tok) == [a, a] == list(tok_r)
        assert np.array_equal(best.view(np.uint32), best_r.view(np.uint32))


@pytest.mark.parametrize("N", [3, 7, 8])
def test_tensor_core_head_ties_and_largest_sums(oracle_mod, N):
    """Three to eight tokens (the tensor-core form): equal best rows give the
    smaller index, and sums of the largest magnitude -- every product
    -128 x -128, so each warp's fp32 partial sum reaches 2^23 and a row's
    2^26 -- stay exact."""
    V, D = 2000, 4096
    H, scale = _table(V, D, 11)
    H[5] = H[1500] = 127
    scale[5] = scale[1500] = 1.0
    H[7] = -128
    scale[7] = 3.0
    X = synth.to_bf16_bits(np.abs(synth.bf16_bits_to_f32(synth.activations(N, D, seed=12))) + 0.5)
    X[N - 1] = synth.to_bf16_bits(np.full(D, -2.0, dtype=np.float32))   # quantises to -128
    head = tl.Head.from_host(H, scale)
    Q, s, z, lg, tok, best, tok2, best2 = _run(head, X)
    assert (Q[N - 1] == -128).all()
    acc_r, lg_r, tok_r, best_r = oracle_mod.head(H, scale, Q, s, z)
    assert acc_r[N - 1, 7] == 128 * 128 * D
    assert np.array_equal(lg.view(np.uint32), lg_r.view(np.uint32))
    assert np.array_equal(tok, tok_r) and np.array_equal(tok2, tok_r)
    assert list(tok[:N - 1]) == [5] * (N - 1)
    assert np.array_equal(best.view(np.uint32), best_r.view(np.uint32))


@pytest.mark.parametrize("N", [1, 8])
def test_full_size_head(oracle_mod, N):
    """151,936 x 4,096: the fused argmax equals the first argmax of the
    kernel's own logits, and sampled rows' logits equal the oracle's."""
    H, scale = _table(VOCAB, HIDDEN, 7)
    head = tl.Head.from_host(H, scale)
    X = synth.activations(N, HIDDEN, seed=8, outlier_frac=0.01)
    Q, s, z, lg, tok, best, tok2, _ = _run(head, X)
    assert np.array_equal(tok, np.argmax(lg, axis=1)) and np.array_equal(tok2, tok)
    assert np.array_equal(best.view(np.uint32), lg[np.arange(N), tok].view(np.uint32))
    rows = np.unique(np.concatenate([np.random.default_rng(9).integers(0, VOCAB, 400), tok,
                                     [0, VOCAB - 1]]))
    _, lg_r, _, _ = oracle_mod.head(H[rows], scale[rows], Q, s, z)
    assert np.array_equal(lg[:, rows].view(np.uint32), lg_r.view(np.uint32))


def test_embedding_rows(oracle_mod):
    V, D = 2000, 4096
    H, scale = _table(V, D, 10)
    table = tl.Head.from_host(H, scale)
    toks = np.array([0, 1999, 17, 17, 1234, 5, 600, 1999], dtype=np.int32)
    X = table.embed(torch.from_numpy(toks).cuda())
    got = X.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, oracle_mod.embed(H, scale, toks))
    # a token outside the table gives a zero row
    bad = table.embed(torch.tensor([3, -1, V], dtype=torch.int32, device="cuda"))
    b = bad.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b[0], oracle_mod.embed(H, scale, np.array([3], np.int32))[0])
    assert not b[1:].any()
