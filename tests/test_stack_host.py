"""Host logic of the stack's end-to-end graph (no GPU): the chunks its host
copies are grouped in."""
import pytest

from bit_matvec_ternary_b300.stack import copy_chunks


@pytest.mark.parametrize("layers", [1, 2, 3, 4, 5, 28, 36, 100])
def test_copy_chunks_cover_every_layer_once(layers):
    ins, outs = copy_chunks(layers)
    for chunks in (ins, outs):
        covered = [l for lo, hi in chunks for l in range(lo, hi)]
        assert covered == list(range(layers))          # in order, each once
        assert all(lo < hi for lo, hi in chunks)
    # layer 0's inputs arrive on their own, so the first launches wait only
    # for them; the last layer's outputs leave on their own, so the tail
    # after the last launch is one layer's copy
    assert ins[0] == (0, 1) and outs[-1] == (layers - 1, layers)
    assert len(ins) <= 2 and len(outs) <= 5


def test_copy_chunks_of_the_8b_stack():
    ins, outs = copy_chunks(36)
    assert ins == [(0, 1), (1, 36)]
    assert outs == [(0, 9), (9, 18), (18, 27), (27, 35), (35, 36)]
