"""The draft / verify accept loop's host logic, with stand-in models (no GPU).

Whatever the draft proposes, the accepted sequence must be exactly what
plain greedy decoding with the target gives; the statistics must count the
accepted proposals; the certificate must pass for a batch-invariant target
and fail when the target's batched scores differ from its scores alone.
"""
import numpy as np
import pytest

from bit_matvec_ternary_b300.decoder import certify, greedy_decode, speculative_decode


class Affine:
    """next(t) = (a t + b) mod V, optionally overridden on some tokens; the
    'best bits' are a fixed function of the token.  batch_bias makes the
    bits depend on the batch size (a target that is not batch-invariant)."""

    def __init__(self, V, a, b, override=None, batch_bias=False):
        self.V, self.a, self.b = V, a, b
        self.override = override or {}
        self.batch_bias = batch_bias
        self.calls = []

    def next_tokens(self, toks):
        self.calls.append(len(toks))
        nxt = [self.override.get(int(t), (self.a * int(t) + self.b) % self.V) for t in toks]
        bits = [(int(t) * 2654435761 + (len(toks) if self.batch_bias else 0)) & 0x7FFFFFFF
                for t in toks]
        return np.array(nxt, dtype=np.int32), np.array(bits, dtype=np.int32)


@pytest.mark.parametrize("k", [1, 3, 7])
def test_perfect_draft_accepts_everything(k):
    target = Affine(1009, 17, 5)
    seq, st = speculative_decode(target, Affine(1009, 17, 5), 3, 40, k=k)
    assert all(n == k + 1 for n in target.calls)          # one verify batch per round
    assert seq == greedy_decode(target, 3, 40)
    assert st.acceptance == 1.0


def test_wrong_draft_still_gives_the_greedy_sequence():
    target = Affine(1009, 17, 5)
    seq, st = speculative_decode(target, Affine(1009, 3, 1), 3, 25, k=7)
    assert seq == greedy_decode(target, 3, 25)
    assert st.accepted < st.drafted


def test_partly_right_draft():
    V = 1009
    target = Affine(V, 17, 5)
    rng = np.random.default_rng(0)
    bad = {int(t): int((t * 7 + 1) % V) for t in rng.choice(V, size=V // 3, replace=False)}
    draft = Affine(V, 17, 5, override=bad)
    seq, st = speculative_decode(target, draft, 11, 200, k=7)
    assert seq == greedy_decode(target, 11, 200)
    assert 0 < st.accepted < st.drafted
    assert len(seq) == 201


def test_certificate():
    target = Affine(1009, 17, 5)
    seq, st = speculative_decode(target, Affine(1009, 17, 5), 3, 30, k=7)
    cert = certify(target, seq, st, greedy_decode(target, 3, 30))
    assert cert.ok and cert.batch_positions_checked == 8 * st.rounds
    skewed = Affine(1009, 17, 5, batch_bias=True)
    seq2, st2 = speculative_decode(skewed, Affine(1009, 17, 5), 3, 30, k=7)
    cert2 = certify(skewed, seq2, st2, greedy_decode(skewed, 3, 30))
    assert cert2.identical_to_greedy and not cert2.batch_invariant and not cert2.ok


def test_draft_length_is_checked():
    with pytest.raises(ValueError):
        speculative_decode(Affine(7, 1, 1), Affine(7, 1, 1), 0, 5, k=8)


@pytest.mark.parametrize("n", [0, 1, 2])
def test_short_runs_return_exactly_n_tokens(n):
    target = Affine(1009, 17, 5)
    seq, st = speculative_decode(target, Affine(1009, 17, 5), 4, n, k=7)
    assert seq == greedy_decode(target, 4, n) and len(seq) == n + 1
    assert st.rounds == (0 if n == 0 else 1)


@pytest.mark.parametrize("k", range(1, 8))
def test_every_draft_length_gives_greedy_and_consistent_counts(k):
    V = 997
    target = Affine(V, 31, 7)
    rng = np.random.default_rng(k)
    bad = {int(t): int((t + 1) % V) for t in rng.choice(V, size=V // 4, replace=False)}
    seq, st = speculative_decode(target, Affine(V, 31, 7, override=bad), 2, 150, k=k)
    assert seq == greedy_decode(target, 2, 150)
    assert st.drafted == k * st.rounds and 0 <= st.accepted <= st.drafted
    # every round appends its accepted proposals and one token of the target's
    assert st.accepted + st.rounds >= 150
    assert all(len(b) == k + 1 for b, _ in st.verify_batches)
    assert st.tokens_per_round == pytest.approx((st.accepted + st.rounds) / st.rounds)


def test_certificate_rejects_a_sequence_that_differs_from_greedy():
    target = Affine(1009, 17, 5)
    seq, st = speculative_decode(target, Affine(1009, 17, 5), 3, 20, k=4)
    wrong = greedy_decode(target, 3, 20)
    wrong[7] = (wrong[7] + 1) % 1009
    cert = certify(target, seq, st, wrong)
    assert cert.batch_invariant and not cert.identical_to_greedy and not cert.ok
