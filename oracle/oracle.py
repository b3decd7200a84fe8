"""numpy-facing wrapper of the CPU oracle (tl_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the library in
bit_matvec_ternary_b300/ never does, and the two share no code.

Every function here marshals numpy arrays into the C oracle; the arithmetic is
in tl_oracle.c, which cites the passages it follows.  bf16 data travels as
uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def load(path: str) -> C.CDLL:
    """Open an oracle shared library and declare its C signatures."""
    L = C.CDLL(path)
    i64, i32, p = C.c_int64, C.c_int, C.c_void_p
    L.oracle_tl2p_words.argtypes = [i64, i64]
    L.oracle_tl2p_words.restype = i64
    L.oracle_pack.argtypes = [p, i64, i64, p]
    L.oracle_pack.restype = i64
    L.oracle_unpack.argtypes = [p, i64, i64, p]
    L.oracle_unpack.restype = i64
    L.oracle_rowsum.argtypes = [p, i64, i64, p]
    L.oracle_rowsum.restype = None
    L.oracle_bf16_rne.argtypes = [C.c_float]
    L.oracle_bf16_rne.restype = C.c_uint16
    L.oracle_bf16_rne_array.argtypes = [p, i64, p]
    L.oracle_bf16_rne_array.restype = None
    L.oracle_quant.argtypes = [p, i64, i64, i32, p, p, p]
    L.oracle_quant.restype = None
    L.oracle_linear_a.argtypes = [p, p, i64, i64, p, i64, p, p]
    L.oracle_linear_a.restype = None
    L.oracle_linear_b.argtypes = [p, p, p, i64, i64, p, p, p, i64, p, p]
    L.oracle_linear_b.restype = None
    L.oracle_linear_a_mt.argtypes = [p, p, i64, i64, p, i64, p, i32]
    L.oracle_linear_a_mt.restype = None
    L.oracle_linear_b_mt.argtypes = [p, p, p, i64, i64, p, p, p, i64, p, i32]
    L.oracle_linear_b_mt.restype = None
    L.oracle_head.argtypes = [p, p, i64, i64, p, p, p, i64, p, p, p, p]
    L.oracle_head.restype = None
    L.oracle_embed.argtypes = [p, p, i64, i64, p, i64, p]
    L.oracle_embed.restype = None
    L.oracle_rmsnorm.argtypes = [p, p, C.c_double, i64, i64, p]
    L.oracle_rmsnorm.restype = None
    L.oracle_swiglu.argtypes = [p, p, i64, i64, p]
    L.oracle_swiglu.restype = None
    L.oracle_absmean_ternarize.argtypes = [p, i64, i64, p, p]
    L.oracle_absmean_ternarize.restype = None
    L.oracle_linear_blockscale.argtypes = [p, p, i64, i64, p, i64, p]
    L.oracle_linear_blockscale.restype = None
    return L


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = load(_build.build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def tl2p_words(M: int, K: int) -> int:
    return int(lib().oracle_tl2p_words(M, K))


def pack(W: np.ndarray) -> np.ndarray:
    """int8 W[M, K] in {-1, 0, 1} -> TL2P v2 words (uint32)."""
    W = _c(W, np.int8)
    M, K = W.shape
    P = np.zeros(max(tl2p_words(M, K), 1), dtype=np.uint32)
    bad = lib().oracle_pack(_ptr(W), M, K, _ptr(P))
    if bad:
        raise ValueError(f"{bad} weights outside {{-1, 0, 1}}")
    return P[: tl2p_words(M, K)]


def unpack(P: np.ndarray, M: int, K: int) -> tuple[np.ndarray, int]:
    """TL2P v2 words -> (int8 W[M, K], count of invalid codes / bad padding)."""
    P = _c(P, np.uint32)
    W = np.zeros((M, K), dtype=np.int8)
    bad = lib().oracle_unpack(_ptr(P), M, K, _ptr(W))
    return W, int(bad)


def rowsum(P: np.ndarray, M: int, K: int) -> np.ndarray:
    P = _c(P, np.uint32)
    out = np.zeros(M, dtype=np.int32)
    lib().oracle_rowsum(_ptr(P), M, K, _ptr(out))
    return out


def bf16_rne(y: np.ndarray) -> np.ndarray:
    y = _c(y, np.float32)
    out = np.zeros(y.shape, dtype=np.uint16)
    lib().oracle_bf16_rne_array(_ptr(y), y.size, _ptr(out))
    return out


def quant(X: np.ndarray, symmetric: bool = False):
    """bf16 X[N, K] (uint16 bits) -> (int8 Q, fp32 s[N], int32 z[N])."""
    X = _c(X, np.uint16)
    N, K = X.shape
    Q = np.zeros((N, K), dtype=np.int8)
    s = np.zeros(N, dtype=np.float32)
    z = np.zeros(N, dtype=np.int32)
    lib().oracle_quant(_ptr(X), N, K, int(symmetric), _ptr(Q), _ptr(s), _ptr(z))
    return Q, s, z


def linear_a(P, scale, M: int, K: int, X, return_sums: bool = False):
    """Mode A: fp32 Y[N, M] from bf16 X[N, K]; optionally the exact sums."""
    P = _c(P, np.uint32); scale = _c(scale, np.float32); X = _c(X, np.uint16)
    N = X.shape[0]
    Y = np.zeros((N, M), dtype=np.float32)
    S = np.zeros((N, M), dtype=np.float64) if return_sums else None
    lib().oracle_linear_a(_ptr(P), _ptr(scale), M, K, _ptr(X), N, _ptr(Y), _ptr(S))
    return (Y, S) if return_sums else Y


def linear_b(P, scale, rsum, M: int, K: int, Q, s, z):
    """Mode B: (int32 acc[N, M], fp32 Y[N, M]) from int8 Q[N, K]."""
    P = _c(P, np.uint32); scale = _c(scale, np.float32); rsum = _c(rsum, np.int32)
    Q = _c(Q, np.int8); s = _c(s, np.float32); z = _c(z, np.int32)
    N = Q.shape[0]
    acc = np.zeros((N, M), dtype=np.int32)
    Y = np.zeros((N, M), dtype=np.float32)
    lib().oracle_linear_b(_ptr(P), _ptr(scale), _ptr(rsum), M, K, _ptr(Q), _ptr(s),
                          _ptr(z), N, _ptr(acc), _ptr(Y))
    return acc, Y


def linear_a_mt(P, scale, M: int, K: int, X, nthreads: int | None = None):
    """Mode A on all host cores (same per-row arithmetic); for timing."""
    P = _c(P, np.uint32); scale = _c(scale, np.float32); X = _c(X, np.uint16)
    N = X.shape[0]
    Y = np.zeros((N, M), dtype=np.float32)
    lib().oracle_linear_a_mt(_ptr(P), _ptr(scale), M, K, _ptr(X), N, _ptr(Y),
                             nthreads or host_cores())
    return Y


def linear_b_mt(P, scale, rsum, M: int, K: int, Q, s, z, nthreads: int | None = None):
    P = _c(P, np.uint32); scale = _c(scale, np.float32); rsum = _c(rsum, np.int32)
    Q = _c(Q, np.int8); s = _c(s, np.float32); z = _c(z, np.int32)
    N = Q.shape[0]
    Y = np.zeros((N, M), dtype=np.float32)
    lib().oracle_linear_b_mt(_ptr(P), _ptr(scale), _ptr(rsum), M, K, _ptr(Q), _ptr(s),
                             _ptr(z), N, _ptr(Y), nthreads or host_cores())
    return Y


def head(H, scale, Q, s, z, return_logits: bool = True):
    """int8 head on quantised activations: (acc int32 [N, V], logits fp32
    [N, V], token int32 [N], best fp32 [N]); acc/logits None unless asked."""
    H = _c(H, np.int8); scale = _c(scale, np.float32)
    Q = _c(Q, np.int8); s = _c(s, np.float32); z = _c(z, np.int32)
    V, D = H.shape
    N = Q.shape[0]
    acc = np.zeros((N, V), dtype=np.int32) if return_logits else None
    lg = np.zeros((N, V), dtype=np.float32) if return_logits else None
    tok = np.zeros(N, dtype=np.int32)
    best = np.zeros(N, dtype=np.float32)
    lib().oracle_head(_ptr(H), _ptr(scale), V, D, _ptr(Q), _ptr(s), _ptr(z), N, _ptr(acc),
                      _ptr(lg), _ptr(tok), _ptr(best))
    return acc, lg, tok, best


def embed(E, scale, tokens):
    """int8 embedding rows times their scales, as bf16 bits [N, D]."""
    E = _c(E, np.int8); scale = _c(scale, np.float32); tokens = _c(tokens, np.int32)
    V, D = E.shape
    N = tokens.shape[0]
    X = np.zeros((N, D), dtype=np.uint16)
    lib().oracle_embed(_ptr(E), _ptr(scale), V, D, _ptr(tokens), N, _ptr(X))
    return X


def rmsnorm(X, gamma, eps: float = 1e-6):
    """RMSNorm of bf16 rows X [N, K] with bf16 gamma [K], in float64."""
    X = _c(X, np.uint16); gamma = _c(gamma, np.uint16)
    N, K = X.shape
    Y = np.zeros((N, K), dtype=np.float64)
    lib().oracle_rmsnorm(_ptr(X), _ptr(gamma), float(eps), N, K, _ptr(Y))
    return Y


def swiglu(G, U):
    """silu(g) * u of bf16 [N, M] gate and up, in float64."""
    G = _c(G, np.uint16); U = _c(U, np.uint16)
    N, M = G.shape
    H = np.zeros((N, M), dtype=np.float64)
    lib().oracle_swiglu(_ptr(G), _ptr(U), N, M, _ptr(H))
    return H


def absmean_ternarize(Wf):
    """float W [M, K] -> (int8 ternary W, fp32 scale per (row, 128-column block))."""
    Wf = _c(Wf, np.float32)
    M, K = Wf.shape
    KB = (K + 127) // 128
    T = np.zeros((M, K), dtype=np.int8)
    bs = np.zeros((M, KB), dtype=np.float32)
    lib().oracle_absmean_ternarize(_ptr(Wf), M, K, _ptr(T), _ptr(bs))
    return T, bs


def linear_blockscale(P, bscale, M: int, K: int, X):
    """y = sum over 128-column blocks of scale[m, b] * block sum, fp32 [N, M]."""
    P = _c(P, np.uint32); bscale = _c(bscale, np.float32); X = _c(X, np.uint16)
    N = X.shape[0]
    Y = np.zeros((N, M), dtype=np.float32)
    lib().oracle_linear_blockscale(_ptr(P), _ptr(bscale), M, K, _ptr(X), N, _ptr(Y))
    return Y


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
