"""N>1 bookkeeping on CPU: world_size-2 gloo ranks.

The path runs as independent replicas (no collective on the data path); these
tests cover the only cross-rank arithmetic (max time, summed work) and show
that splitting a matrix by 16-row panels across ranks reproduces the
unsharded oracle result exactly.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from bit_matvec_ternary_b300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, units, rate = replicas.aggregate_throughput(10.0 + 5.0 * rank, 1.0)
        out[rank] = (ms, units, rate)
        # each rank computes its panel rows of one matrix with the oracle
        import torch
        from bit_matvec_ternary_b300 import synth
        from oracle import oracle as O
        M, K = 100, 300
        W = synth.ternary(M, K, 0.626, 3)
        sc = synth.scales(M, 3)
        X = synth.activations(2, K, 4)
        m0, m1 = replicas.row_shard(M, rank, world)
        Ys = O.linear_a(O.pack(W[m0:m1]), sc[m0:m1], m1 - m0, K, X) if m1 > m0 else \
            np.zeros((2, 0), np.float32)
        parts = [None] * world
        dist.all_gather_object(parts, (m0, m1, Ys))
        full = np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])], axis=1)
        ref = O.linear_a(O.pack(W), sc, M, K, X)
        out[10 + rank] = bool(np.array_equal(full, ref))
    finally:
        dist.destroy_process_group()


def test_two_rank_replica_aggregation_and_row_sharding():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(2):
            ms, units, rate = out[r]
            assert ms == 15.0 and units == 2.0
            assert rate == pytest.approx(2.0 / 0.015)
            assert out[10 + r] is True


@pytest.mark.parametrize("M,world", [(4096, 2), (1024, 8), (100, 3), (5, 4)])
def test_row_shard_covers_rows_on_panel_boundaries(M, world):
    spans = [replicas.row_shard(M, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == M
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0
    for m0, m1 in spans:
        assert m0 % 16 == 0 and m0 <= m1
