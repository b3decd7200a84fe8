"""Python binding of the C ABI in include/tl.h (ctypes over libtl.so).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels (or, for ``tl_pack``, its host packer).  PyTorch
supplies device memory and the current CUDA stream.  Importing this module
fails loudly when libtl.so has not been built -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtl.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m bit_matvec_ternary_b300.build` "
        "(the ternary linears have no non-CUDA implementation)")

_lib = C.CDLL(LIB_PATH)

TL_OK = 0
TL_ERR_NULL, TL_ERR_SHAPE, TL_ERR_ALIGN, TL_ERR_BAD_VALUE = 1, 2, 3, 4
TL_ERR_MODE, TL_ERR_UNSUPPORTED, TL_ERR_CUDA, TL_ERR_TIMEOUT, TL_ERR_WORKSPACE = 5, 6, 7, 8, 9
TL_MODE_BF16, TL_MODE_I8, TL_MODE_I8_FUSED = 0, 1, 2
TL_OUT_F32, TL_OUT_BF16, TL_OUT_I32_RAW = 0, 1, 2
TL_FLAG_PDL, TL_FLAG_SYMMETRIC = 1, 2
TL_LAYOUT_TL2P_V2 = 2
TL_MAX_GROUP = 4

# Every symbol include/tl.h declares.
EXPORTS = ("tl_packed_bytes", "tl_pack", "tl_validate_packed", "tl_workspace_bytes",
           "tl_decode_plan", "tl_prefill_plan", "tl_quantize_act", "tl_linear", "tl_linear_group",
           "tl_head_workspace_bytes", "tl_head_argmax", "tl_embed",
           "tl_rmsnorm_quant", "tl_swiglu_quant", "tl_ternarize_absmean",
           "tl_linear_blockscale",
           "tl_chain_image_bytes", "tl_chain_workspace_bytes", "tl_chain_encode",
           "tl_chain_run", "tl_linear_noalloc", "tl_status_string", "tl_version")
TL_MAX_CHAIN = 4096
TL_DEVERR_TIMEOUT = 1
TL_NOALLOC_SCRATCH_BYTES = 4 << 20


class tl_weight(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("scale", C.c_void_p), ("rowsum", C.c_void_p),
                ("M", C.c_int32), ("K", C.c_int32), ("layout", C.c_uint32)]


class tl_chain_step(C.Structure):
    _fields_ = [("Ws", C.POINTER(tl_weight)), ("G", C.c_int), ("X", C.c_void_p),
                ("Ys", C.POINTER(C.c_void_p))]


_p, _i64, _int, _sz = C.c_void_p, C.c_int64, C.c_int, C.c_size_t
_lib.tl_packed_bytes.argtypes = [_i64, _i64]
_lib.tl_packed_bytes.restype = _sz
_lib.tl_pack.argtypes = [_p, _i64, _i64, _p, _p, _p, _p]
_lib.tl_pack.restype = _int
_lib.tl_validate_packed.argtypes = [_p, _i64, _i64, C.POINTER(C.c_int64)]
_lib.tl_validate_packed.restype = _int
_lib.tl_workspace_bytes.argtypes = [C.POINTER(tl_weight), _int, _int]
_lib.tl_workspace_bytes.restype = _sz
_lib.tl_decode_plan.argtypes = [C.POINTER(tl_weight), _int, _int, _int, C.POINTER(C.c_int32)]
_lib.tl_decode_plan.restype = _int
_lib.tl_prefill_plan.argtypes = [C.POINTER(tl_weight), _int, _int, _int, C.POINTER(C.c_int32)]
_lib.tl_prefill_plan.restype = _int
_lib.tl_quantize_act.argtypes = [_p, _int, _int, _p, _p, _p, _int, _p]
_lib.tl_quantize_act.restype = _int
_lib.tl_linear.argtypes = [C.POINTER(tl_weight), _p, _p, _p, _p, _int, _int, _int, _p, _sz,
                           C.c_uint, _p]
_lib.tl_linear.restype = _int
_lib.tl_linear_group.argtypes = [C.POINTER(tl_weight), _int, _p, _p, _p, C.POINTER(_p), _int,
                                 _int, _int, _p, _sz, C.c_uint, _p]
_lib.tl_linear_group.restype = _int
_lib.tl_head_workspace_bytes.argtypes = [_i64, _int, _int]
_lib.tl_head_workspace_bytes.restype = _sz
_lib.tl_head_argmax.argtypes = [_p, _p, _i64, _int, _p, _p, _p, _int, _p, _p, _p, _p, _sz,
                                C.c_uint, _p]
_lib.tl_head_argmax.restype = _int
_lib.tl_embed.argtypes = [_p, _p, _i64, _int, _p, _int, _p, _p]
_lib.tl_embed.restype = _int
_lib.tl_rmsnorm_quant.argtypes = [_p, _p, C.c_float, _int, _int, _p, _p, _p, _p, _int, _p]
_lib.tl_rmsnorm_quant.restype = _int
_lib.tl_swiglu_quant.argtypes = [_p, _p, _int, _int, _p, _p, _p, _p, _int, _p]
_lib.tl_swiglu_quant.restype = _int
_lib.tl_ternarize_absmean.argtypes = [_p, _i64, _i64, _p, _p]
_lib.tl_ternarize_absmean.restype = _int
_lib.tl_linear_blockscale.argtypes = [_p, _p, _int, _int, _p, _int, _p, _int, C.c_uint, _p]
_lib.tl_linear_blockscale.restype = _int
_lib.tl_chain_image_bytes.argtypes = [_int, _int]
_lib.tl_chain_image_bytes.restype = _sz
_lib.tl_chain_workspace_bytes.argtypes = [C.POINTER(tl_chain_step), _int, _int, _int]
_lib.tl_chain_workspace_bytes.restype = _sz
_lib.tl_chain_encode.argtypes = [C.POINTER(tl_chain_step), _int, _int, _int, _int, _p,
                                 C.c_longlong, _p, _sz, _p, _sz]
_lib.tl_chain_encode.restype = _int
_lib.tl_chain_run.argtypes = [_p, _p, _p]
_lib.tl_chain_run.restype = _int
_lib.tl_linear_noalloc.argtypes = [C.POINTER(tl_weight), _p, _p, _p, _p, _int, _int, _int,
                                   C.c_uint, _p]
_lib.tl_linear_noalloc.restype = _int
_lib.tl_status_string.argtypes = [_int]
_lib.tl_status_string.restype = C.c_char_p
_lib.tl_version.argtypes = []
_lib.tl_version.restype = _int


class TLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tl_status_string(status)} (status {status})")


def _check(status: int, where: str) -> None:
    if status != TL_OK:
        raise TLError(status, where)


def tl_status_string(status: int) -> str:
    return _lib.tl_status_string(int(status)).decode()


def tl_version() -> int:
    return int(_lib.tl_version())


def tl_packed_bytes(M: int, K: int) -> int:
    return int(_lib.tl_packed_bytes(M, K))


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def tl_pack(W: np.ndarray, scale: np.ndarray | None = None):
    """Host packer: int8 W[M, K] -> (uint32 words, fp32 scale copy, int32 rowsum)."""
    W = np.ascontiguousarray(W, dtype=np.int8)
    M, K = W.shape
    packed = np.zeros(max(tl_packed_bytes(M, K), 4) // 4, dtype=np.uint32)
    rowsum = np.zeros(M, dtype=np.int32)
    if scale is not None:
        scale = np.ascontiguousarray(scale, dtype=np.float32)
        scale_out = np.empty(M, dtype=np.float32)
        st = _lib.tl_pack(_np_ptr(W), M, K, _np_ptr(scale), _np_ptr(packed),
                          _np_ptr(scale_out), _np_ptr(rowsum))
    else:
        scale_out = None
        st = _lib.tl_pack(_np_ptr(W), M, K, None, _np_ptr(packed), None, _np_ptr(rowsum))
    _check(st, "tl_pack")
    return packed[: tl_packed_bytes(M, K) // 4], scale_out, rowsum


def tl_ternarize_absmean(W: np.ndarray):
    """Host: float W [M, K] -> (int8 ternary codes, fp32 scale per (row,
    128-column block)) by the block's mean |w|."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    M, K = W.shape
    T = np.zeros((M, K), dtype=np.int8)
    bs = np.zeros((M, (K + 127) // 128), dtype=np.float32)
    _check(_lib.tl_ternarize_absmean(_np_ptr(W), M, K, _np_ptr(T), _np_ptr(bs)),
           "tl_ternarize_absmean")
    return T, bs


def tl_validate_packed(packed: np.ndarray, M: int, K: int) -> int:
    """Host validator: number of invalid codes / non-zero padding weights."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    bad = C.c_int64(0)
    st = _lib.tl_validate_packed(_np_ptr(packed), M, K, C.byref(bad))
    if st not in (TL_OK, TL_ERR_BAD_VALUE):
        _check(st, "tl_validate_packed")
    return int(bad.value)


# ---------------------------------------------------------------- device side
def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> int | None:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class TernaryWeight:
    """A packed matrix resident on the device (caller-owned torch tensors)."""
    packed: "object"   # torch.int32 tensor, tl_packed_bytes(M, K) bytes
    scale: "object"    # torch.float32 [M]
    rowsum: "object"   # torch.int32 [M]
    M: int
    K: int

    @classmethod
    def from_host(cls, packed: np.ndarray, scale: np.ndarray, rowsum: np.ndarray, M: int, K: int,
                  device="cuda") -> "TernaryWeight":
        torch = _torch()
        p = torch.from_numpy(np.ascontiguousarray(packed).view(np.int32)).to(device)
        s = torch.from_numpy(np.ascontiguousarray(scale, dtype=np.float32)).to(device)
        r = torch.from_numpy(np.ascontiguousarray(rowsum, dtype=np.int32)).to(device)
        return cls(p, s, r, M, K)

    @classmethod
    def from_int8(cls, W: np.ndarray, scale: np.ndarray, device="cuda") -> "TernaryWeight":
        packed, sc, rs = tl_pack(W, scale)
        return cls.from_host(packed, sc, rs, W.shape[0], W.shape[1], device)

    def struct(self) -> tl_weight:
        return tl_weight(self.packed.data_ptr(), self.scale.data_ptr(), self.rowsum.data_ptr(),
                         self.M, self.K, TL_LAYOUT_TL2P_V2)


@dataclass
class BlockScaledWeight:
    """Packed ternary codes with one scale per (row, 128-column block)."""
    packed: "object"   # torch.int32 tensor, tl_packed_bytes(M, K) bytes
    bscale: "object"   # torch.float32 [M, ceil(K / 128)]
    M: int
    K: int

    @classmethod
    def from_float(cls, W: np.ndarray, device="cuda") -> "BlockScaledWeight":
        torch = _torch()
        T, bs = tl_ternarize_absmean(W)
        packed, _, _ = tl_pack(T)
        return cls(torch.from_numpy(packed.view(np.int32)).to(device),
                   torch.from_numpy(bs).to(device), W.shape[0], W.shape[1])


def tl_linear_blockscale(weight: BlockScaledWeight, X, out=None, out_dtype: int = TL_OUT_F32,
                         flags: int = 0, stream=None):
    """y = sum over blocks of scale[m, b] * block sum, bf16 X [N, K]."""
    torch = _torch()
    N = X.shape[0]
    if out is None:
        dt = torch.float32 if out_dtype == TL_OUT_F32 else torch.bfloat16
        out = torch.empty((N, weight.M), dtype=dt, device=X.device)
    st = _lib.tl_linear_blockscale(weight.packed.data_ptr(), weight.bscale.data_ptr(), weight.M,
                                   weight.K, X.data_ptr(), N, out.data_ptr(), out_dtype, flags,
                                   _stream_ptr(stream))
    _check(st, "tl_linear_blockscale")
    return out


def _structs(ws):
    arr = (tl_weight * len(ws))()
    for i, w in enumerate(ws):
        arr[i] = w.struct() if isinstance(w, TernaryWeight) else w
    return arr


def tl_workspace_bytes(weights, N: int) -> int:
    ws = weights if isinstance(weights, (list, tuple)) else [weights]
    return int(_lib.tl_workspace_bytes(_structs(ws), len(ws), N))


PLAN_FIELDS = ("R", "KB", "NS", "KW", "KWL", "Pps", "P", "Lc", "LcL", "rows",
               "warps", "chunk_tiles", "ctas_per_sm", "max_cta_rows")


def decode_plan(weights, N: int, sms: int) -> dict:
    """The decode kernel's work split for these shapes (host only)."""
    ws = weights if isinstance(weights, (list, tuple)) else [weights]
    out = (C.c_int32 * len(PLAN_FIELDS))()
    _check(_lib.tl_decode_plan(_structs(ws), len(ws), N, sms, out), "tl_decode_plan")
    return dict(zip(PLAN_FIELDS, list(out)))


PREFILL_PLAN_FIELDS = ("BN", "S", "KBS", "tiles", "grid")


def prefill_plan(weights, N: int, sms: int) -> dict:
    """The tensor-core kernel's tile width, K splits and grid for these
    shapes (host only)."""
    ws = weights if isinstance(weights, (list, tuple)) else [weights]
    out = (C.c_int32 * len(PREFILL_PLAN_FIELDS))()
    _check(_lib.tl_prefill_plan(_structs(ws), len(ws), N, sms, out), "tl_prefill_plan")
    return dict(zip(PREFILL_PLAN_FIELDS, list(out)))


def make_workspace(weights_lists, N: int, device="cuda"):
    """Zero-filled workspace large enough for every group in weights_lists."""
    torch = _torch()
    need = max(tl_workspace_bytes(w, N) for w in weights_lists)
    return torch.zeros(max(need, 256), dtype=torch.uint8, device=device)


def tl_quantize_act(X, symmetric: bool = False, Q=None, s=None, z=None, stream=None):
    """bf16 X[N, K] (cuda) -> (int8 Q[N, K], fp32 s[N], int32 z[N])."""
    torch = _torch()
    N, K = X.shape
    if Q is None:
        Q = torch.empty((N, K), dtype=torch.int8, device=X.device)
    if s is None:
        s = torch.empty(N, dtype=torch.float32, device=X.device)
    if z is None:
        z = torch.empty(N, dtype=torch.int32, device=X.device)
    st = _lib.tl_quantize_act(X.data_ptr(), N, K, Q.data_ptr(), s.data_ptr(), z.data_ptr(),
                              int(bool(symmetric)), _stream_ptr(stream))
    _check(st, "tl_quantize_act")
    return Q, s, z


_OUT_TORCH = {TL_OUT_F32: "float32", TL_OUT_BF16: "bfloat16", TL_OUT_I32_RAW: "int32"}


def tl_linear_group(weights, X, s=None, z=None, outs=None, mode: int = TL_MODE_BF16,
                    out_dtype: int = TL_OUT_F32, workspace=None, flags: int = 0, stream=None):
    """Y_g = linear(W_g, X) for matrices sharing X; returns the list of Y_g."""
    torch = _torch()
    ws = list(weights)
    N = X.shape[0]
    if outs is None:
        dt = getattr(torch, _OUT_TORCH[out_dtype])
        outs = [torch.empty((N, w.M), dtype=dt, device=X.device) for w in ws]
    if workspace is None:
        workspace = make_workspace([ws], N, device=X.device)
    ys = (C.c_void_p * len(outs))(*[o.data_ptr() for o in outs])
    st = _lib.tl_linear_group(_structs(ws), len(ws), X.data_ptr(),
                              None if s is None else s.data_ptr(),
                              None if z is None else z.data_ptr(), ys, N, mode, out_dtype,
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              flags, _stream_ptr(stream))
    _check(st, "tl_linear_group")
    return outs


def tl_linear(weight, X, s=None, z=None, out=None, mode: int = TL_MODE_BF16,
              out_dtype: int = TL_OUT_F32, workspace=None, flags: int = 0, stream=None):
    """Y = linear(W, X) for one matrix."""
    torch = _torch()
    N = X.shape[0]
    if out is None:
        dt = getattr(torch, _OUT_TORCH[out_dtype])
        out = torch.empty((N, weight.M), dtype=dt, device=X.device)
    if workspace is None:
        workspace = make_workspace([[weight]], N, device=X.device)
    w = _structs([weight])
    st = _lib.tl_linear(w, X.data_ptr(), None if s is None else s.data_ptr(),
                        None if z is None else z.data_ptr(), out.data_ptr(), N, mode, out_dtype,
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(), flags,
                        _stream_ptr(stream))
    _check(st, "tl_linear")
    return out


def tl_linear_noalloc(weight, X, s=None, z=None, out=None, mode: int = TL_MODE_BF16,
                      out_dtype: int = TL_OUT_F32, flags: int = 0, stream=None):
    """Y = linear(W, X) with the library's fixed scratch array: no workspace
    argument, nothing allocated by the library (the output is allocated
    here only when `out` is None)."""
    torch = _torch()
    N = X.shape[0]
    if out is None:
        dt = getattr(torch, _OUT_TORCH[out_dtype])
        out = torch.empty((N, weight.M), dtype=dt, device=X.device)
    st = _lib.tl_linear_noalloc(_structs([weight]), X.data_ptr(),
                                None if s is None else s.data_ptr(),
                                None if z is None else z.data_ptr(), out.data_ptr(), N, mode,
                                out_dtype, flags, _stream_ptr(stream))
    _check(st, "tl_linear_noalloc")
    return out


def _fused_outs(N, K, device, want_y, want_q):
    torch = _torch()
    y = torch.empty((N, K), dtype=torch.bfloat16, device=device) if want_y else None
    if want_q:
        return (y, torch.empty((N, K), dtype=torch.int8, device=device),
                torch.empty(N, dtype=torch.float32, device=device),
                torch.empty(N, dtype=torch.int32, device=device))
    return y, None, None, None


def _ptr_or_none(t):
    return None if t is None else t.data_ptr()


def tl_rmsnorm_quant(X, gamma, eps: float = 1e-6, want_y: bool = True, want_q: bool = True,
                     symmetric: bool = False, stream=None):
    """RMSNorm of bf16 X [N, K] -> (bf16 Y or None, int8 Q, s, z or Nones)."""
    N, K = X.shape
    y, q, s, z = _fused_outs(N, K, X.device, want_y, want_q)
    st = _lib.tl_rmsnorm_quant(X.data_ptr(), gamma.data_ptr(), float(eps), N, K, _ptr_or_none(y),
                               _ptr_or_none(q), _ptr_or_none(s), _ptr_or_none(z),
                               int(bool(symmetric)), _stream_ptr(stream))
    _check(st, "tl_rmsnorm_quant")
    return y, q, s, z


def tl_swiglu_quant(G, U, want_y: bool = True, want_q: bool = True, symmetric: bool = False,
                    stream=None):
    """silu(G) * U of bf16 [N, M] -> (bf16 H or None, int8 Q, s, z or Nones)."""
    N, M = G.shape
    y, q, s, z = _fused_outs(N, M, G.device, want_y, want_q)
    st = _lib.tl_swiglu_quant(G.data_ptr(), U.data_ptr(), N, M, _ptr_or_none(y), _ptr_or_none(q),
                              _ptr_or_none(s), _ptr_or_none(z), int(bool(symmetric)),
                              _stream_ptr(stream))
    _check(st, "tl_swiglu_quant")
    return y, q, s, z


class Head:
    """An int8 output head (or embedding table) resident on the device:
    int8 [V, D] rows and one fp32 scale per row (caller-owned tensors)."""

    def __init__(self, table, scale):
        self.table, self.scale = table, scale
        self.V, self.D = table.shape
        self._ws = {}

    @classmethod
    def from_host(cls, H: np.ndarray, scale: np.ndarray, device="cuda") -> "Head":
        torch = _torch()
        return cls(torch.from_numpy(np.ascontiguousarray(H, dtype=np.int8)).to(device),
                   torch.from_numpy(np.ascontiguousarray(scale, dtype=np.float32)).to(device))

    def workspace(self, N: int):
        if N not in self._ws:
            need = int(_lib.tl_head_workspace_bytes(self.V, self.D, N))
            if need == 0:
                raise TLError(TL_ERR_SHAPE, "tl_head_workspace_bytes")
            self._ws[N] = _torch().zeros(need, dtype=_torch().uint8, device=self.table.device)
        return self._ws[N]

    def argmax(self, Q, s, z, logits=None, token=None, best=None, flags: int = 0, stream=None):
        """(token int32 [N], best fp32 [N]); fills `logits` [N, V] when given."""
        torch = _torch()
        N = Q.shape[0]
        dev = self.table.device
        token = torch.empty(N, dtype=torch.int32, device=dev) if token is None else token
        best = torch.empty(N, dtype=torch.float32, device=dev) if best is None else best
        ws = self.workspace(N)
        st = _lib.tl_head_argmax(self.table.data_ptr(), self.scale.data_ptr(), self.V, self.D,
                                 Q.data_ptr(), s.data_ptr(), z.data_ptr(), N,
                                 None if logits is None else logits.data_ptr(), token.data_ptr(),
                                 best.data_ptr(), ws.data_ptr(), ws.numel(), flags,
                                 _stream_ptr(stream))
        _check(st, "tl_head_argmax")
        return token, best

    def embed(self, tokens, out=None, stream=None):
        """bf16 [N, D] rows of the table for int32 device tokens [N]."""
        torch = _torch()
        N = tokens.shape[0]
        out = torch.empty((N, self.D), dtype=torch.bfloat16, device=self.table.device) \
            if out is None else out
        st = _lib.tl_embed(self.table.data_ptr(), self.scale.data_ptr(), self.V, self.D,
                           tokens.data_ptr(), N, out.data_ptr(), _stream_ptr(stream))
        _check(st, "tl_embed")
        return out


class Chain:
    """A chain of (grouped) linears run by one persistent launch per pass.

    ``steps`` is a list of (weights, X, outs): the TernaryWeight objects of a
    group that reads the bf16 tensor X [N, K], and its output tensors.  A
    step's X may be an earlier step's output.  Encodes the chain on the host,
    keeps the image on the device and owns the chain's zero-filled workspace.
    """

    def __init__(self, steps, N: int, mode: int = TL_MODE_BF16, out_dtype: int = TL_OUT_F32,
                 gate=None, wait_limit: int = 0, device="cuda"):
        torch = _torch()
        self.N, self.mode, self.out_dtype = N, mode, out_dtype
        self._keep = []
        arr = (tl_chain_step * len(steps))()
        for i, (ws, X, outs) in enumerate(steps):
            ws = list(ws)
            wa = _structs(ws)
            ya = (C.c_void_p * len(outs))(*[o.data_ptr() for o in outs])
            self._keep += [wa, ya, X, outs, ws]
            arr[i] = tl_chain_step(wa, len(ws), X.data_ptr(), ya)
        self._steps = arr
        self.nsteps = len(steps)
        need = int(_lib.tl_chain_workspace_bytes(arr, len(steps), N, mode))
        if need == 0:
            raise TLError(TL_ERR_SHAPE, "tl_chain_workspace_bytes")
        self.workspace = torch.zeros(need, dtype=torch.uint8, device=device)
        nimg = int(_lib.tl_chain_image_bytes(len(steps), mode))
        self.image = np.zeros(nimg, dtype=np.uint8)
        self.gate = gate
        st = _lib.tl_chain_encode(arr, len(steps), N, mode, out_dtype,
                                  None if gate is None else gate.data_ptr(), int(wait_limit),
                                  self.workspace.data_ptr(), need, _np_ptr(self.image), nimg)
        _check(st, "tl_chain_encode")
        self.image_dev = torch.from_numpy(self.image).to(device)

    def run(self, stream=None) -> None:
        _check(_lib.tl_chain_run(_np_ptr(self.image), self.image_dev.data_ptr(),
                                 _stream_ptr(stream)), "tl_chain_run")

    def status(self) -> int:
        """The device status word (0: every wait of the last pass succeeded)."""
        return int(self.workspace[:4].view(_torch().int32).item())


def raw_call(name: str):
    """The ctypes function of one ABI symbol (for tests of argument checks)."""
    return getattr(_lib, name)
