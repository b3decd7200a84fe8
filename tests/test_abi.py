"""CPU-side checks of the C ABI: the library loads, exports what include/tl.h
declares, packs exactly like the oracle, and rejects bad arguments before it
touches CUDA.  No compute call runs here."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from bit_matvec_ternary_b300 import synth, tl
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "tl.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"TL_API\s+[\w\s\*]+?\b(tl_\w+)\s*\(", text)))


def test_header_declares_what_binding_exports():
    assert declared_functions() == sorted(tl.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = C.CDLL(tl.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings():
    assert tl.tl_version() == 100
    for st in range(0, 10):
        msg = tl.tl_status_string(st)
        assert msg and msg != "unknown status"
    assert tl.tl_status_string(99) == "unknown status"


@pytest.mark.parametrize("M,K,expect", [(2048, 1024, 524288), (16, 128, 512), (5, 37, 512),
                                        (17, 129, 2048), (0, 5, 0), (5, 0, 0),
                                        (4096, 12288, 12582912)])
def test_packed_bytes(M, K, expect):
    assert tl.tl_packed_bytes(M, K) == expect


SHAPES = [(16, 128), (5, 37), (17, 129), (64, 1000), (300, 256), (1, 1), (2048, 1024)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_host_packer_matches_oracle_bytes(oracle_mod, M, K):
    W = synth.ternary(M, K, 0.626, seed=M + K)
    scale = synth.scales(M, seed=1)
    packed, sc, rs = tl.tl_pack(W, scale)
    assert np.array_equal(packed, oracle_mod.pack(W))
    assert np.array_equal(rs, oracle_mod.rowsum(packed, M, K))
    assert np.array_equal(sc, scale)
    assert tl.tl_validate_packed(packed, M, K) == 0


def test_host_packer_large_matrix_threaded(oracle_mod):
    # big enough to take the threaded path
    M, K = 1024, 4096
    W = synth.ternary(M, K, 0.7, seed=3)
    packed, _, rs = tl.tl_pack(W)
    assert np.array_equal(packed, oracle_mod.pack(W))
    assert np.array_equal(rs, W.astype(np.int64).sum(axis=1))


def test_host_packer_rejects_non_ternary():
    W = np.zeros((4, 8), dtype=np.int8)
    W[1, 1] = 3
    with pytest.raises(tl.TLError) as e:
        tl.tl_pack(W)
    assert e.value.status == tl.TL_ERR_BAD_VALUE


def test_validator_counts_invalid_codes_and_padding():
    W = np.ones((5, 37), dtype=np.int8)
    packed, _, _ = tl.tl_pack(W)
    assert tl.tl_validate_packed(packed, 5, 37) == 0
    p2 = packed.copy()
    p2[-1] ^= np.uint32(0x40000000)           # a padding field 01 -> 00 (+1)
    assert tl.tl_validate_packed(p2, 5, 37) == 1
    p3 = np.full_like(packed, 0x55555555)
    p3[0] = 0x55555557                         # field 11
    assert tl.tl_validate_packed(p3, 5, 37) == 1


# ---- argument checks: each returns before any CUDA call ----------------------

def _w(M=16, K=128, layout=tl.TL_LAYOUT_TL2P_V2, packed=0x1000, scale=0x2000, rowsum=0x3000):
    return tl.tl_weight(packed, scale, rowsum, M, K, layout)


def _linear(w, X=0x4000, s=0x5000, z=0x6000, Y=0x7000, N=1, mode=0, out=0, ws=0x8000,
            wsb=1 << 20):
    arr = (tl.tl_weight * 1)(w)
    return tl.raw_call("tl_linear")(arr, X, s, z, Y, N, mode, out, ws, wsb, 0, None)


def test_linear_argument_errors():
    assert _linear(_w(packed=0)) == tl.TL_ERR_NULL
    assert _linear(_w(scale=0)) == tl.TL_ERR_NULL
    assert _linear(_w(rowsum=0), mode=tl.TL_MODE_I8) == tl.TL_ERR_NULL
    assert _linear(_w(M=0)) == tl.TL_ERR_SHAPE
    assert _linear(_w(K=0)) == tl.TL_ERR_SHAPE
    assert _linear(_w(layout=7)) == tl.TL_ERR_UNSUPPORTED
    assert _linear(_w(packed=0x1008)) == tl.TL_ERR_ALIGN
    assert _linear(_w(), X=0) == tl.TL_ERR_NULL
    assert _linear(_w(), N=0) == tl.TL_ERR_SHAPE
    assert _linear(_w(), mode=5) == tl.TL_ERR_MODE
    assert _linear(_w(), out=9) == tl.TL_ERR_MODE
    assert _linear(_w(), out=tl.TL_OUT_I32_RAW, mode=tl.TL_MODE_BF16) == tl.TL_ERR_MODE
    assert _linear(_w(), mode=tl.TL_MODE_I8, s=0) == tl.TL_ERR_NULL
    assert _linear(_w(), mode=tl.TL_MODE_I8, z=0) == tl.TL_ERR_NULL
    assert _linear(_w(), Y=0) == tl.TL_ERR_NULL
    assert _linear(_w(), Y=0x7002) == tl.TL_ERR_ALIGN
    assert _linear(_w(), ws=0) == tl.TL_ERR_WORKSPACE
    assert _linear(_w(), ws=0x8010) == tl.TL_ERR_ALIGN


def test_fused_quant_mode_argument_errors():
    F = tl.TL_MODE_I8_FUSED
    assert _linear(_w(rowsum=0), mode=F) == tl.TL_ERR_NULL       # needs the row sums
    assert _linear(_w(rowsum=0x3002), mode=F) == tl.TL_ERR_ALIGN
    assert _linear(_w(), mode=F, out=tl.TL_OUT_I32_RAW) == tl.TL_ERR_MODE
    assert _linear(_w(), mode=F, X=0x4001) == tl.TL_ERR_ALIGN     # bf16 X
    assert _linear(_w(), mode=3) == tl.TL_ERR_MODE


def test_group_argument_errors():
    f = tl.raw_call("tl_linear_group")
    ys = (C.c_void_p * 5)(0x7000, 0x7100, 0x7200, 0x7300, 0x7400)
    arr = (tl.tl_weight * 5)(_w(), _w(), _w(), _w(), _w())
    assert f(arr, 0, 0x4000, None, None, ys, 1, 0, 0, 0x8000, 1 << 20, 0, None) == tl.TL_ERR_SHAPE
    assert f(arr, 5, 0x4000, None, None, ys, 1, 0, 0, 0x8000, 1 << 20, 0, None) == tl.TL_ERR_SHAPE
    mixed = (tl.tl_weight * 2)(_w(K=128), _w(K=256))
    assert f(mixed, 2, 0x4000, None, None, ys, 1, 0, 0, 0x8000, 1 << 20, 0, None) == tl.TL_ERR_SHAPE
    assert f(None, 1, 0x4000, None, None, ys, 1, 0, 0, 0x8000, 1 << 20, 0, None) == tl.TL_ERR_NULL


def test_quantize_argument_errors():
    f = tl.raw_call("tl_quantize_act")
    assert f(0, 1, 8, 0x100, 0x200, 0x300, 0, None) == tl.TL_ERR_NULL
    assert f(0x1000, 0, 8, 0x100, 0x200, 0x300, 0, None) == tl.TL_ERR_SHAPE
    assert f(0x1000, 1, 0, 0x100, 0x200, 0x300, 0, None) == tl.TL_ERR_SHAPE
    assert f(0x1001, 1, 8, 0x100, 0x200, 0x300, 0, None) == tl.TL_ERR_ALIGN


def test_workspace_query_without_device_is_well_defined():
    arr = (tl.tl_weight * 1)(_w(M=4096, K=4096))
    n1 = tl.raw_call("tl_workspace_bytes")(arr, 1, 1)
    n8 = tl.raw_call("tl_workspace_bytes")(arr, 1, 8)
    assert 0 < n1 <= n8
    assert tl.raw_call("tl_workspace_bytes")(arr, 0, 1) == 0


def test_chain_arguments_checked_without_a_gpu():
    """The chain entry points reject bad arguments before touching a device."""
    assert tl._lib.tl_chain_image_bytes(0, tl.TL_MODE_BF16) == 0
    assert tl._lib.tl_chain_image_bytes(tl.TL_MAX_CHAIN + 1, tl.TL_MODE_BF16) == 0
    one = tl._lib.tl_chain_image_bytes(1, tl.TL_MODE_BF16)
    assert tl._lib.tl_chain_image_bytes(2, tl.TL_MODE_BF16) > one
    assert tl._lib.tl_chain_image_bytes(1, tl.TL_MODE_I8) > one   # a quantiser step per linear
    w = tl.tl_weight(0x1000, 0x2000, 0x3000, 64, 128, tl.TL_LAYOUT_TL2P_V2)
    wa = (tl.tl_weight * 1)(w)
    ya = (C.c_void_p * 1)(0x8000)
    steps = (tl.tl_chain_step * 1)(tl.tl_chain_step(wa, 1, 0x4000, ya))
    img = np.zeros(one, dtype=np.uint8)
    enc = tl._lib.tl_chain_encode
    args = lambda N, mode, out: (steps, 1, N, mode, out, None, 0, 0x100000, 1 << 20,
                                 img.ctypes.data_as(C.c_void_p), img.size)
    assert enc(*args(9, tl.TL_MODE_BF16, tl.TL_OUT_F32)) == tl.TL_ERR_SHAPE
    assert enc(*args(0, tl.TL_MODE_BF16, tl.TL_OUT_F32)) == tl.TL_ERR_SHAPE
    assert enc(*args(1, 7, tl.TL_OUT_F32)) == tl.TL_ERR_MODE
    assert enc(*args(1, tl.TL_MODE_I8_FUSED, tl.TL_OUT_F32)) == tl.TL_ERR_MODE  # chains: A, B
    assert enc(*args(1, tl.TL_MODE_BF16, tl.TL_OUT_I32_RAW)) == tl.TL_ERR_MODE
    assert enc(None, 1, 1, 0, 0, None, 0, 0x100000, 1 << 20,
               img.ctypes.data_as(C.c_void_p), img.size) == tl.TL_ERR_NULL
    # an image that was never encoded is refused before any launch
    assert tl._lib.tl_chain_run(img.ctypes.data_as(C.c_void_p), 0x10000, None) == tl.TL_ERR_BAD_VALUE


def test_head_arguments_checked_without_a_gpu():
    f = tl._lib.tl_head_argmax
    p = 0x10000
    assert tl._lib.tl_head_workspace_bytes(1000, 4096, 9) == 0          # N > 8
    assert tl._lib.tl_head_workspace_bytes(1000, 4100, 1) == 0          # D % 16
    assert tl._lib.tl_head_workspace_bytes(1000, 16384, 8) == 0         # N * D too large
    assert f(None, p, 10, 64, p, p, p, 1, None, p, p, p, 1 << 20, 0, None) == tl.TL_ERR_NULL
    assert f(p, p, 10, 65, p, p, p, 1, None, p, p, p, 1 << 20, 0, None) == tl.TL_ERR_SHAPE
    assert f(p + 8, p, 10, 64, p, p, p, 1, None, p, p, p, 1 << 20, 0, None) == tl.TL_ERR_ALIGN
    assert f(p, p, 10, 64, p, p, p, 1, None, p, p, None, 1 << 20, 0, None) == tl.TL_ERR_WORKSPACE
    assert tl._lib.tl_embed(None, p, 10, 64, p, 1, p, None) == tl.TL_ERR_NULL


def test_blockscale_arguments_checked_without_a_gpu():
    f = tl._lib.tl_linear_blockscale
    p = 0x10000
    ok = dict(packed=p, bscale=p, M=64, K=256, X=p, N=1, Y=p, out=tl.TL_OUT_F32)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["packed"], a["bscale"], a["M"], a["K"], a["X"], a["N"], a["Y"], a["out"], 0, None)

    assert call(packed=None) == tl.TL_ERR_NULL
    assert call(bscale=None) == tl.TL_ERR_NULL
    assert call(X=None) == tl.TL_ERR_NULL
    assert call(Y=None) == tl.TL_ERR_NULL
    assert call(M=0) == tl.TL_ERR_SHAPE
    assert call(K=0) == tl.TL_ERR_SHAPE
    assert call(N=0) == tl.TL_ERR_SHAPE
    assert call(K=(1 << 20) + 1) == tl.TL_ERR_SHAPE
    assert call(out=tl.TL_OUT_I32_RAW) == tl.TL_ERR_MODE
    assert call(packed=p + 8) == tl.TL_ERR_ALIGN          # 16-byte codes
    assert call(bscale=p + 2) == tl.TL_ERR_ALIGN
    assert call(X=p + 1) == tl.TL_ERR_ALIGN
    assert call(Y=p + 2) == tl.TL_ERR_ALIGN               # fp32 out
    assert call(Y=p + 2, out=tl.TL_OUT_BF16) != tl.TL_ERR_ALIGN   # bf16 out: 2 bytes suffice


def test_fused_neighbour_arguments_checked_without_a_gpu():
    rq, sq = tl._lib.tl_rmsnorm_quant, tl._lib.tl_swiglu_quant
    p = 0x10000
    # X, gamma, eps, N, K, Y, Q, s, z, symmetric
    assert rq(None, p, 1e-6, 1, 64, p, p, p, p, 0, None) == tl.TL_ERR_NULL
    assert rq(p, p, 1e-6, 1, 64, None, None, p, p, 0, None) == tl.TL_ERR_NULL   # no output asked
    assert rq(p, p, 1e-6, 1, 64, p, p, None, p, 0, None) == tl.TL_ERR_NULL      # Q without s
    assert rq(p, p, 1e-6, 0, 64, p, p, p, p, 0, None) == tl.TL_ERR_SHAPE
    assert rq(p, p, 1e-6, 1, 32769, p, p, p, p, 0, None) == tl.TL_ERR_SHAPE     # longest row 32768
    assert rq(p + 1, p, 1e-6, 1, 64, p, p, p, p, 0, None) == tl.TL_ERR_ALIGN
    assert rq(p, p, 1e-6, 1, 64, p, p, p + 2, p, 0, None) == tl.TL_ERR_ALIGN
    assert rq(p, p, -1.0, 1, 64, p, p, p, p, 0, None) == tl.TL_ERR_BAD_VALUE
    assert rq(p, p, float("nan"), 1, 64, p, p, p, p, 0, None) == tl.TL_ERR_BAD_VALUE
    # G, U, N, M, H, Q, s, z, symmetric
    assert sq(p, None, 1, 64, p, p, p, p, 0, None) == tl.TL_ERR_NULL
    assert sq(p, p, 65536, 64, p, p, p, p, 0, None) == tl.TL_ERR_SHAPE
    assert sq(p, p, 1, 64, p, p, p, p + 1, 0, None) == tl.TL_ERR_ALIGN


@pytest.mark.parametrize("M,K", [(7, 300), (64, 128), (33, 1000)])
def test_absmean_ternarizer_matches_oracle(oracle_mod, M, K):
    """The library's host ternariser gives the oracle's codes and scales bit
    for bit (both follow the same reading: double mean, fp32 scale, double
    ratio, ties to even)."""
    rng = np.random.default_rng(M * K)
    W = (rng.standard_normal((M, K)) * rng.uniform(0.01, 3.0, size=(M, 1))).astype(np.float32)
    W[0, :128] = 0.0                                    # an all-zero block
    W[1, 5] = 1e6                                       # a block dominated by one value
    T, bs = tl.tl_ternarize_absmean(W)
    To, bso = oracle_mod.absmean_ternarize(W)
    assert np.array_equal(T, To)
    assert np.array_equal(bs.view(np.uint32), bso.view(np.uint32))
    bad = W.copy()
    bad[2, 3] = np.nan
    with pytest.raises(tl.TLError):
        tl.tl_ternarize_absmean(bad)
