"""GPU: speculative decoding on a decoder built from the library's calls.

The target is a seeded synthetic decoder (int8 embedding, per layer RMSNorm,
q/k/v, o, RMSNorm, gate/up, SwiGLU, down, final RMSNorm, int8 head with the
fused argmax).  Whatever the draft, the accepted tokens must equal plain
greedy decoding with the target, and every verified position must score
bit-identically alone and inside its batch of up to eight.
"""
import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a CUDA device", allow_module_level=True)

from bit_matvec_ternary_b300 import tl  # noqa: E402
from bit_matvec_ternary_b300.decoder import (TernaryDecoder, certify, greedy_decode,  # noqa: E402
                                             speculative_decode)

SMALL = synth.ModelShape("small", layers=3, hidden=1024, q_heads=16, kv_heads=8, head_dim=128,
                         ffn=3072, vocab=8192, tied_embeddings=False)
DRAFT = synth.ModelShape("draft", layers=2, hidden=512, q_heads=8, kv_heads=4, head_dim=64,
                         ffn=1536, vocab=8192, tied_embeddings=False)


@pytest.fixture(scope="module")
def target():
    return TernaryDecoder(SMALL, vocab=8192, seed=5)


def _perturbed_head(target, frac, seed):
    """The target's head with the scales of a share of its rows changed."""
    rng = np.random.default_rng(seed)
    sc = target.head.scale.cpu().numpy().copy()
    rows = rng.choice(target.V, size=int(frac * target.V), replace=False)
    sc[rows] *= rng.uniform(0.3, 3.0, size=rows.size).astype(np.float32)
    return tl.Head(target.head.table, torch.from_numpy(sc).cuda())


def test_batch_invariance_of_the_decoder(target):
    toks = [1, 77, 4095, 8191, 0, 300, 301, 302]
    nxt8, bits8 = target.next_tokens(toks)
    for i, t in enumerate(toks):
        n1, b1 = target.next_tokens([t])
        assert n1[0] == nxt8[i] and b1[0] == bits8[i]


@pytest.mark.parametrize("kind", ["same_model", "other_model", "perturbed_head"])
def test_speculative_equals_greedy(target, kind):
    if kind == "same_model":
        draft = target
    elif kind == "other_model":
        draft = TernaryDecoder(DRAFT, vocab=8192, seed=9)
    else:
        draft = TernaryDecoder(SMALL, vocab=8192, seed=5,
                               head_table=_perturbed_head(target, 0.3, 3),
                               embed_table=target.embed)
    ref = greedy_decode(target, 17, 48)
    seq, st = speculative_decode(target, draft, 17, 48, k=7)
    cert = certify(target, seq, st, ref)
    assert cert.identical_to_greedy, (seq, ref)
    assert cert.batch_invariant
    if kind == "same_model":
        assert st.acceptance == 1.0
