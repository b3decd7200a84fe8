"""tl_linear_noalloc: the decode linear for callers that cannot allocate.

Some callers may not call cudaMalloc (or any allocating routine) where they
run a linear: code running inside another runtime's memory pool, loops that
must not allocate after start-up, hosts that only hand over input and output
buffers.  For them the library keeps its split-K scratch in a fixed device
array.  This file runs last (pytest collects files in name order) and checks,
through the C ABI, that two calls in a row give the same results as
tl_linear with a caller workspace: bit for bit in mode B, within the mode-A
tolerance of the other parity tests in mode A.
"""
import ctypes as C

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
    return float(np.max(np.abs(y - ref) / den))


def _bf16(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def _noalloc(w, X, s, z, Y, N, mode, out):
    arr = (tl.tl_weight * 1)(w.struct())
    return tl.raw_call("tl_linear_noalloc")(
        arr, X.data_ptr(), None if s is None else s.data_ptr(),
        None if z is None else z.data_ptr(), Y.data_ptr(), N, mode, out, 0,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("M,K,N", [(4096, 4096, 1), (1024, 4096, 8), (4096, 12288, 8),
                                   (777, 333, 3), (12288, 4096, 8)])
def test_noalloc_matches_workspace_entry_point_twice(M, K, N):
    W = synth.ternary(M, K, 0.626, M + K)
    w = tl.TernaryWeight.from_int8(W, synth.scales(M, M + K))
    for call in range(2):                      # two calls in a row share the array
        X = _bf16(synth.activations(N, K, seed=100 * call + N, outlier_frac=0.01))
        ya = torch.empty((N, M), dtype=torch.float32, device="cuda")
        assert _noalloc(w, X, None, None, ya, N, tl.TL_MODE_BF16, tl.TL_OUT_F32) == tl.TL_OK
        ref_a = tl.tl_linear(w, X)
        Q, s, z = tl.tl_quantize_act(X)
        yb = torch.empty((N, M), dtype=torch.float32, device="cuda")
        assert _noalloc(w, Q, s, z, yb, N, tl.TL_MODE_I8, tl.TL_OUT_F32) == tl.TL_OK
        ref_b = tl.tl_linear(w, Q, s, z, mode=tl.TL_MODE_I8)
        torch.cuda.synchronize()
        assert rel_err(ya.cpu().numpy(), ref_a.cpu().numpy()) <= TOL_A
        assert torch.equal(yb.view(torch.int32), ref_b.view(torch.int32))


@pytest.fixture(scope="module")
def oracle_mod():
    from oracle import oracle
    oracle.lib()
    return oracle


def test_noalloc_against_the_oracle(oracle_mod):
    """The same entry point against the CPU oracle: batches above eight
    (the array reused by successive 8-token chunks), a prefill-sized batch
    (which this entry point runs on the decode kernel), and a small matrix
    right after a large one, so that each call starts from what the previous
    call of another shape left in the array."""
    cases = [(12288, 4096, 8), (64, 256, 2), (4096, 12288, 13), (1024, 4096, 300),
             (33, 4099, 1)]
    for M, K, N in cases:
        W = synth.ternary(M, K, 0.626, 7 * M + K)
        scale = synth.scales(M, 7 * M + K)
        w = tl.TernaryWeight.from_int8(W, scale)
        P = oracle_mod.pack(W)
        rs = oracle_mod.rowsum(P, M, K)
        Xh = synth.activations(N, K, seed=N + K, outlier_frac=0.01)
        X = _bf16(Xh)
        ya = torch.empty((N, M), dtype=torch.float32, device="cuda")
        assert _noalloc(w, X, None, None, ya, N, tl.TL_MODE_BF16, tl.TL_OUT_F32) == tl.TL_OK
        Q, s, z = tl.tl_quantize_act(X)
        yb = torch.empty((N, M), dtype=torch.float32, device="cuda")
        assert _noalloc(w, Q, s, z, yb, N, tl.TL_MODE_I8, tl.TL_OUT_F32) == tl.TL_OK
        torch.cuda.synchronize()
        ref = oracle_mod.linear_a_mt(P, scale, M, K, Xh)
        assert rel_err(ya.cpu().numpy(), ref) <= TOL_A, (M, K, N)
        Qr, sr, zr = oracle_mod.quant(Xh)
        refb = oracle_mod.linear_b_mt(P, scale, rs, M, K, Qr, sr, zr)
        assert np.array_equal(yb.cpu().numpy().view(np.uint32), refb.view(np.uint32)), (M, K, N)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # a matrix whose split-K scratch would not fit the fixed array: refused
    # with TL_ERR_WORKSPACE before anything is launched
    M, K = 70000, 4096                # 4375 row tiles: ~4.5 MB of split-K scratch at 8 tokens
    w = tl.tl_weight(0x1000, 0x2000, 0x3000, M, K, tl.TL_LAYOUT_TL2P_V2)
    arr = (tl.tl_weight * 1)(w)
    st = tl.raw_call("tl_linear_noalloc")(arr, 0x4000, None, None, 0x8000, 8, tl.TL_MODE_BF16,
                                          tl.TL_OUT_F32, 0, None)
    assert st == tl.TL_ERR_WORKSPACE
