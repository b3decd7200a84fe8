"""The decode kernel's work split, checked on the host against the invariants
the kernel relies on (no GPU needed).

`tl_decode_plan` returns the split the library's planner computes.  The
walk below follows the kernel's own assignment of that split: CTA ranges
inside one K slice, each warp's contiguous share of its CTA's units, the
copies of at most `chunk_tiles` tiles that never cross a row tile, and the
runs that end a row tile or a warp's share.  It checks that

  * every (row tile, block) unit is processed exactly once;
  * no CTA works in two slices, and no CTA touches more row tiles than its
    accumulators hold;
  * a warp leaves at most two partial row tiles per slice (its two boundary
    slots), and a row tile it claims whole belongs to it alone;
  * in a one-slice launch every CTA owns whole row tiles;
  * a (row tile, slice) piece spans one or two CTAs, and the kernel's test
    for "split" (piece_split) agrees; in a one-slice launch a split row tile
    has exactly the two pieces the exchange slots expect;
  * the grid stays within the GPU's CTA slots unless the row-tile limit
    forces more CTAs.
"""
from __future__ import annotations

import numpy as np
import pytest

from bit_matvec_ternary_b300 import tl


def _w(M, K):
    # the planner reads only the shapes
    return tl.tl_weight(0x1000, 0x2000, 0x3000, M, K, tl.TL_LAYOUT_TL2P_V2)


def _cdiv(a, b):
    return (a + b - 1) // b


def _width(p, s):
    return p["KWL"] if s == p["NS"] - 1 else p["KW"]


def _units_per_cta(p, s):
    return p["LcL"] if s == p["NS"] - 1 else p["Lc"]


def _cta_range(p, c):
    s, c_in = divmod(c, p["Pps"])
    if s >= p["NS"]:
        return None
    su = p["R"] * _width(p, s)
    lc = _units_per_cta(p, s)
    off = min(c_in * lc, su)
    return s, off, min(off + lc, su)


def _piece_split(p, r, s):
    kw, lc = _width(p, s), _units_per_cta(p, s)
    u0 = r * kw
    return u0 // lc != (u0 + kw - 1) // lc


def walk(p):
    R, KB, KW = p["R"], p["KB"], p["KW"]
    cover = np.zeros((R, KB), np.int32)
    pieces = {}
    for c in range(p["P"]):
        rng = _cta_range(p, c)
        if rng is None or rng[2] <= rng[1]:
            continue
        s, a0, a1 = rng                       # slice-local units [a0, a1)
        kw = _width(p, s)
        if p["NS"] == 1:                      # one slice: whole row tiles per CTA
            assert a0 % kw == 0 and a1 % kw == 0, (c, a0, a1, kw)
        rf, rl = a0 // kw, (a1 - 1) // kw
        lo_f, hi_l = a0 - rf * kw, a1 - rl * kw
        assert rl - rf + 1 <= p["rows"] <= p["max_cta_rows"]
        span = lambda r: (lo_f if r == rf else 0, hi_l if r == rl else kw)
        npu = a1 - a0
        lw = _cdiv(npu, p["warps"])
        owners, whole = {}, []
        for w in range(p["warps"]):
            u, ue = a0 + min(w * lw, npu), a0 + min(w * lw + lw, npu)
            if u >= ue:
                continue
            r, b = divmod(u, kw)
            run_lo, slots = b, 0
            while u < ue:
                n = min(p["chunk_tiles"], ue - u, kw - b)
                owners.setdefault(r, set()).add(w)
                cover[r, s * KW + b: s * KW + b + n] += 1
                if b + n == kw or u + n == ue:         # a run ends
                    lo, hi = span(r)
                    if run_lo == lo and b + n == hi:
                        whole.append((r, w))
                    else:
                        slots += 1
                    run_lo = b + n if b + n < kw else -1
                u += n
                b += n
                if b == kw:
                    r, b = r + 1, 0
                if run_lo < 0:
                    run_lo = b
            assert slots <= 2
        for r, w in whole:
            assert owners[r] == {w}
        for r in range(rf, rl + 1):
            pieces.setdefault((r, s), []).append((c,) + span(r))
    assert (cover == 1).all(), np.argwhere(cover != 1)[:5]
    for (r, s), lst in pieces.items():
        assert len(lst) in (1, 2), (r, s, lst)
        assert sum(hi - lo for _, lo, hi in lst) == _width(p, s)
        assert (len(lst) == 2) == _piece_split(p, r, s)


SHAPES = [([4096, 1024, 1024], 4096), ([4096], 4096), ([12288, 12288], 4096),
          ([4096], 12288), ([2048], 1024), ([1024], 3072), ([3072], 1024), ([1024], 2048),
          ([5], 37), ([17, 33], 129), ([300], 1000), ([777], 333), ([33], 4099), ([1], 1),
          ([16], 128), ([100000], 128), ([16], 65536), ([40], 20000), ([3000], 6144),
          ([1536], 6272), ([70000], 4096)]


@pytest.mark.parametrize("Ms,K", SHAPES)
@pytest.mark.parametrize("sms", [148, 132, 74, 20, 1])
@pytest.mark.parametrize("N", [1, 8])
def test_decode_plan_covers_every_unit_once(Ms, K, sms, N):
    p = tl.decode_plan([_w(M, K) for M in Ms], N, sms)
    assert p["NS"] == _cdiv(p["KB"], 32) or p["NS"] == _cdiv(p["KB"], p["KW"])
    assert p["P"] == p["NS"] * p["Pps"]
    slots = sms * p["ctas_per_sm"]
    assert p["P"] <= max(slots, p["NS"] * _cdiv(p["R"], p["max_cta_rows"] - 2))
    walk(p)


def test_decode_plan_does_not_depend_on_the_batch():
    ws = [_w(12288, 4096), _w(12288, 4096)]
    plans = [tl.decode_plan(ws, n, 148) for n in (1, 2, 3, 4, 5, 8, 9, 40)]
    keys = [k for k in tl.PLAN_FIELDS if k != "chunk_tiles"]
    for q in plans[1:]:
        assert {k: q[k] for k in keys} == {k: plans[0][k] for k in keys}


def test_decode_plan_rejects_bad_arguments():
    st = tl._lib.tl_decode_plan(None, 1, 1, 148, None)
    assert st == tl.TL_ERR_NULL
    with pytest.raises(Exception):
        tl.decode_plan([_w(16, 128), _w(16, 256)], 1, 148)     # K differs inside a group
    with pytest.raises(Exception):
        tl.decode_plan([_w(16, 128)], 1, 0)


# ---------------------------------------------------------------- prefill plan
# The 8B groups at 512 tokens, as measured on B300: q/k/v and gate+up in
# 256-token tiles unsplit, o in 128-token tiles (128 items, no K split), down
# in 256-token tiles with two K splits.
PREFILL_8B = {
    "qkv": ([4096, 1024, 1024], 4096, (256, 1)),
    "o": ([4096], 4096, (128, 1)),
    "gate_up": ([12288, 12288], 4096, (256, 1)),
    "down": ([4096], 12288, (256, 2)),
}


@pytest.mark.parametrize("name", sorted(PREFILL_8B))
def test_prefill_plan_of_the_8b_groups(name):
    Ms, K, (bn, s) = PREFILL_8B[name]
    p = tl.prefill_plan([_w(M, K) for M in Ms], 512, 148)
    assert (p["BN"], p["S"]) == (bn, s)
    mt = sum(_cdiv(M, 128) for M in Ms)
    assert p["tiles"] == mt * _cdiv(512, bn)
    assert p["grid"] == min(p["tiles"] * p["S"], 148)


@pytest.mark.parametrize("K", [128, 1000, 4096, 12288, 65536])
@pytest.mark.parametrize("Ms", [[128], [777], [4096], [4096, 1024, 1024], [12288, 12288], [20000]])
@pytest.mark.parametrize("N", [256, 300, 512, 1000, 4096])
@pytest.mark.parametrize("sms", [1, 132, 148])
def test_prefill_plan_invariants(K, Ms, N, sms):
    """Whatever the shapes: a width the kernel has, splits of whole 128-column
    blocks (at least four each when K is split) with none empty, the tile
    count of that width, and no more CTAs than SMs or items."""
    p = tl.prefill_plan([_w(M, K) for M in Ms], N, sms)
    KB = _cdiv(K, 128)
    assert p["BN"] in (128, 256)
    assert p["S"] >= 1 and p["KBS"] >= 1
    assert p["S"] == _cdiv(KB, p["KBS"])                 # no empty split
    assert (p["S"] - 1) * p["KBS"] < KB <= p["S"] * p["KBS"]
    if p["S"] > 1:
        assert KB // p["S"] >= 4
    assert p["tiles"] == sum(_cdiv(M, 128) for M in Ms) * _cdiv(N, p["BN"])
    assert 1 <= p["grid"] == min(p["tiles"] * p["S"], sms)


def test_prefill_plan_rejects_bad_arguments():
    import ctypes
    buf = (ctypes.c_int32 * len(tl.PREFILL_PLAN_FIELDS))()
    assert tl._lib.tl_prefill_plan(None, 1, 512, 148, None) == tl.TL_ERR_NULL
    ws = tl._structs([_w(4096, 4096), _w(1024, 2048)])
    assert tl._lib.tl_prefill_plan(ws, 2, 512, 148, buf) == tl.TL_ERR_SHAPE   # K differs
    assert tl._lib.tl_prefill_plan(tl._structs([_w(4096, 4096)]), 1, 0, 148, buf) == tl.TL_ERR_SHAPE
