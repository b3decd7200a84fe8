"""Greedy decoding and the draft / verify accept loop, on the library's calls.

Speculative decoding as the pages describe it: a small draft model proposes
up to seven tokens, the large model checks them all in one batched pass and
accepts a proposal only when it equals the token it would have chosen itself
(fermionresearch.com/models, "Neutrino-1 0.6B"; wiki "Neutrino-1", "What is
actually new"), so the output is token-identical to plain greedy decoding
with the large model (blog "Neutrino-1: quantization is a training decision",
"Serving it: the Neutrino Engine": 27,648 tokens, zero divergences).

``speculative_decode`` runs that loop over any two objects with a
``next_tokens(tokens) -> (next, best_bits)`` method: position i of a batch
is decoded from token i alone.  ``TernaryDecoder`` is such a model built
only from the library's C-ABI calls -- int8 embedding, per layer RMSNorm,
q/k/v, o (reading q), RMSNorm, gate/up, SwiGLU and down, then a final
RMSNorm, per-token quantisation and the int8 head's fused argmax.
Attention and the KV cache are not part of this library (they are not
linears), so the decoder has none: every position depends only on its own
token, which is what lets the verify pass batch the drafted positions, and
it has no residual adds (each layer's output is normalised by the next
RMSNorm).  It is a synthetic stand-in with seeded random weights for
exercising the loop and its certificate, not a language model.

The certificate of a run (``Certificate``): the accepted sequence equals
plain greedy decoding token for token, and every position the verifier
scored inside a batch has bit-identical best logits when scored alone -- the
batch invariance the loop's token identity rests on.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import synth, tl


# ---------------------------------------------------------------- the accept loop

@dataclass
class SpecStats:
    rounds: int = 0
    drafted: int = 0
    accepted: int = 0
    verify_batches: list = field(default_factory=list)   # (tokens in, per-position best bits)

    @property
    def acceptance(self) -> float:
        return self.accepted / self.drafted if self.drafted else 0.0

    @property
    def tokens_per_round(self) -> float:
        return (self.accepted + self.rounds) / self.rounds if self.rounds else 0.0


def greedy_decode(model, t0: int, n: int) -> list[int]:
    """n tokens after t0, one position at a time."""
    seq = [int(t0)]
    for _ in range(n):
        nxt, _ = model.next_tokens([seq[-1]])
        seq.append(int(nxt[0]))
    return seq


def speculative_decode(target, draft, t0: int, n: int, k: int = 7):
    """n tokens after t0: each round the draft proposes k tokens greedily,
    the target scores the last accepted token and the k proposals in one
    batch (k + 1 <= 8 positions), and proposals are accepted while each
    equals the target's own choice; the first disagreement (or, after k
    acceptances, the token after the last proposal) is replaced by the
    target's token.  Returns (sequence, SpecStats)."""
    if not 1 <= k <= 7:
        raise ValueError("k drafted tokens per round must be in 1..7")
    seq = [int(t0)]
    st = SpecStats()
    while len(seq) - 1 < n:
        proposals, t = [], seq[-1]
        for _ in range(k):
            nxt, _ = draft.next_tokens([t])
            t = int(nxt[0])
            proposals.append(t)
        batch = [seq[-1]] + proposals
        verified, bits = target.next_tokens(batch)
        st.verify_batches.append((list(batch), list(bits)))
        j = 0
        while j < k and proposals[j] == int(verified[j]):
            j += 1
        seq += proposals[:j] + [int(verified[j])]
        st.rounds += 1
        st.drafted += k
        st.accepted += j
    return seq[: n + 1], st


@dataclass
class Certificate:
    tokens: int
    identical_to_greedy: bool
    batch_positions_checked: int
    batch_invariant: bool

    @property
    def ok(self) -> bool:
        return self.identical_to_greedy and self.batch_invariant


def certify(target, spec_seq, stats: SpecStats, greedy_seq) -> Certificate:
    """Check a speculative run against plain greedy decoding, and re-score
    every verified position alone: its best logit must carry the same bits
    as inside its batch."""
    same = list(spec_seq) == list(greedy_seq)
    checked, invariant = 0, True
    for batch, bits in stats.verify_batches:
        for tok, b in zip(batch, bits):
            _, alone = target.next_tokens([tok])
            invariant &= int(alone[0]) == int(b)
            checked += 1
    return Certificate(len(spec_seq) - 1, same, checked, invariant)


# ---------------------------------------------------------------- a decoder on the library

class TernaryDecoder:
    """Seeded synthetic decoder of a given geometry on the library's calls
    (mode A linears, bf16 activations between them)."""

    def __init__(self, shape: synth.ModelShape, vocab: int, layers: int | None = None,
                 seed: int = 0, head_table=None, embed_table=None, device: str = "cuda"):
        import torch
        self.torch = torch
        self.shape = shape
        self.layers = shape.layers if layers is None else layers
        self.D = shape.hidden
        self.V = vocab
        self.device = device
        shp = shape.linear_shapes()
        rng = np.random.default_rng(seed)
        self.w = []
        for layer in range(self.layers):
            per = {}
            for p in synth.PROJ_ORDER:
                M, K = shp[p]
                s = synth.matrix_seed(seed, layer, p)
                W = synth.ternary(M, K, synth.zero_fraction(shape, layer, p), s)
                per[p] = tl.TernaryWeight.from_int8(W, synth.scales(M, s), device=device)
            self.w.append(per)

        def bf16(a):
            return torch.from_numpy(synth.to_bf16_bits(a.astype(np.float32)).view(np.int16)) \
                .view(torch.bfloat16).to(device)

        self.gamma = [(bf16(rng.uniform(0.8, 1.2, self.D)), bf16(rng.uniform(0.8, 1.2, self.D)))
                      for _ in range(self.layers)]
        self.gamma_final = bf16(rng.uniform(0.8, 1.2, self.D))

        def table(tseed):
            r = np.random.default_rng(tseed)
            T = r.integers(-128, 128, size=(vocab, self.D), dtype=np.int16).astype(np.int8)
            return tl.Head.from_host(T, r.uniform(0.005, 0.05, vocab).astype(np.float32), device)

        self.embed = embed_table if embed_table is not None else table(seed + 1)
        self.head = head_table if head_table is not None else table(seed + 2)
        groups = [[self.w[l][p] for p in grp] for l in range(self.layers)
                  for grp in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))]
        self.ws = tl.make_workspace(groups, 8, device=device)

    def next_tokens(self, tokens):
        """Greedy next token for each position (1 to 8 positions, each on its
        own), and the bits of each position's best logit."""
        torch = self.torch
        N = len(tokens)
        if not 1 <= N <= 8:
            raise ValueError("1 to 8 positions per call")
        tk = torch.tensor(list(tokens), dtype=torch.int32, device=self.device)
        x = self.embed.embed(tk)
        for l in range(self.layers):
            w, (g1, g2) = self.w[l], self.gamma[l]
            h, *_ = tl.tl_rmsnorm_quant(x, g1, 1e-6, want_q=False)
            q, _, _ = tl.tl_linear_group([w["q"], w["k"], w["v"]], h, out_dtype=tl.TL_OUT_BF16,
                                         workspace=self.ws)
            o = tl.tl_linear(w["o"], q, out_dtype=tl.TL_OUT_BF16, workspace=self.ws)
            h, *_ = tl.tl_rmsnorm_quant(o, g2, 1e-6, want_q=False)
            g, u = tl.tl_linear_group([w["gate"], w["up"]], h, out_dtype=tl.TL_OUT_BF16,
                                      workspace=self.ws)
            a, *_ = tl.tl_swiglu_quant(g, u, want_q=False)
            x = tl.tl_linear(w["down"], a, out_dtype=tl.TL_OUT_BF16, workspace=self.ws)
        _, Q, s, z = tl.tl_rmsnorm_quant(x, self.gamma_final, 1e-6, want_y=False)
        tok, best = self.head.argmax(Q, s, z)
        return tok.cpu().numpy(), best.cpu().view(torch.int32).numpy()
