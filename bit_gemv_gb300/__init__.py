"""Python binding of libninfer_ternary.so (the GB300 Hadamard-rotated ternary
projection). Argument marshalling only: every step of the computation runs in
the library's CUDA kernels or its host C++ code. There is no fallback: if the
shared library is missing, importing this package raises ImportError.

Names match the C entry points of include/ninfer_ternary.h. Host entry points
take and return numpy arrays; device entry points take torch CUDA tensors and
run on the current torch CUDA stream.
"""
from __future__ import annotations

import ctypes as C
import os
from collections import namedtuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libninfer_ternary.so")

if not os.path.exists(LIBRARY_PATH):
    raise ImportError(f"{LIBRARY_PATH} is not built; run `python bit_gemv_gb300/build.py` "
                      "(or __graft_entry__.build()) first")
_lib = C.CDLL(LIBRARY_PATH)

PQ2_0_G128 = 142
PTQ1_0_G128 = 143
FORMATS = {"PQ2_0_G128": PQ2_0_G128, "PTQ1_0_G128": PTQ1_0_G128}
F32, BF16, F16 = 0, 1, 2

GEOMETRY_FIELDS = ("n", "k", "k_pad", "groups_per_row", "base_bytes_per_group",
                   "high_bytes_per_group", "base_row_bytes", "high_row_bytes",
                   "scale_row_bytes", "base_offset", "base_bytes", "high_offset",
                   "high_bytes", "scale_offset", "scale_bytes", "payload_bytes")
RowSplitGeometry = namedtuple("RowSplitGeometry", GEOMETRY_FIELDS)


class _Geom(C.Structure):
    _fields_ = [(f, C.c_uint64) for f in GEOMETRY_FIELDS]


class NinferError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = _lib.ninfer_status_name(status).decode()
        super().__init__(f"{self.status_name}: {message}")


_u64, _int, _vp = C.c_uint64, C.c_int, C.c_void_p
_sig = {
    "ninfer_last_error": (C.c_char_p, []),
    "ninfer_status_name": (C.c_char_p, [_int]),
    "ninfer_abi_version": (_int, []),
    "ninfer_ternary_geometry": (_int, [_int, _u64, _u64, C.POINTER(_Geom)]),
    "ninfer_ternary_pack": (_int, [_int, _u64, _u64, _vp, _vp, _vp, _u64]),
    "ninfer_ternary_unpack": (_int, [_int, _u64, _u64, _vp, _u64, _vp, _vp]),
    "ninfer_blocks_to_planes": (_int, [_int, _u64, _u64, _vp, _u64, _vp, _u64]),
    "ninfer_planes_to_blocks": (_int, [_int, _u64, _u64, _vp, _u64, _vp, _u64]),
    "ninfer_blocks_to_planes_device": (_int, [_int, _u64, _u64, _vp, _u64, _vp, _u64, _vp]),
    "ninfer_planes_to_blocks_device": (_int, [_int, _u64, _u64, _vp, _u64, _vp, _u64, _vp]),
    "ninfer_validate_signs": (_int, [_vp, _u64]),
    "ninfer_hadamard_fwd": (_int, [_vp, _int, _vp, _int, _vp, _u64, _u64, _vp]),
    "ninfer_hadamard_inv": (_int, [_vp, _int, _vp, _int, _vp, _u64, _u64, _vp]),
    "ninfer_ternary_matmul_workspace": (_int, [_int, _u64, _u64, _u64, _int, C.POINTER(_u64)]),
    "ninfer_ternary_matmul": (_int, [_int, _vp, _u64, _u64, _u64, _vp, _int, _vp, _vp, _int, _u64, _vp, _u64, _vp]),
    "ninfer_ternary_embed": (_int, [_int, _vp, _u64, _u64, _u64, _vp, _u64, _vp, _vp, _int, _vp, _vp]),
    "ninfer_device_errors": (_int, [C.POINTER(C.c_uint32), _int]),
    "ninfer_set_prefetch_before_dependency": (_int, [_int]),
    "ninfer_set_wait_limit": (_int, [C.c_longlong]),
    "ninfer_ternary_matmul_noalloc": (_int, [_int, _vp, _u64, _u64, _u64, _vp, _int, _vp, _vp, _int, _u64, _vp]),
    "ninfer_ternary_gate_up_workspace": (_int, [_int, _u64, _u64, _u64, _int, _int, C.POINTER(_u64)]),
    "ninfer_ternary_gate_up": (_int, [_int, _vp, _vp, _u64, _u64, _u64, _vp, _int, _vp, _vp, _vp, _int, _u64, _vp,
                                      _u64, _vp]),
}
NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_sig)


def _check(status: int):
    if status != 0:
        raise NinferError(status, _lib.ninfer_last_error().decode(errors="replace"))


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def ninfer_abi_version() -> int:
    return _lib.ninfer_abi_version()


# ------------------------------------------------------------------ host ---
def ninfer_ternary_geometry(fmt, n: int, k: int) -> RowSplitGeometry:
    g = _Geom()
    _check(_lib.ninfer_ternary_geometry(_fmt(fmt), n, k, C.byref(g)))
    return RowSplitGeometry(*[getattr(g, f) for f in GEOMETRY_FIELDS])


def ninfer_ternary_pack(fmt, values: np.ndarray, scales_f16: np.ndarray) -> np.ndarray:
    values = np.ascontiguousarray(values, dtype=np.int8)
    scales_f16 = np.ascontiguousarray(scales_f16, dtype=np.uint16)
    n, k = values.shape
    g = ninfer_ternary_geometry(fmt, n, k)
    if scales_f16.size != n * g.groups_per_row:
        raise ValueError("scales must hold n * groups_per_row binary16 words")
    out = np.empty(g.payload_bytes, dtype=np.uint8)
    _check(_lib.ninfer_ternary_pack(_fmt(fmt), n, k, _np_ptr(values), _np_ptr(scales_f16), _np_ptr(out), out.size))
    return out


def ninfer_ternary_unpack(fmt, n: int, k: int, payload: np.ndarray):
    payload = np.ascontiguousarray(payload, dtype=np.uint8).reshape(-1)
    g = ninfer_ternary_geometry(fmt, n, k)
    values = np.empty((n, k), dtype=np.int8)
    scales = np.empty((n, g.groups_per_row), dtype=np.uint16)
    _check(_lib.ninfer_ternary_unpack(_fmt(fmt), n, k, _np_ptr(payload), payload.size, _np_ptr(values), _np_ptr(scales)))
    return values, scales


def ninfer_blocks_to_planes(fmt, n: int, k: int, blocks: np.ndarray) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    g = ninfer_ternary_geometry(fmt, n, k)
    out = np.empty(g.payload_bytes, dtype=np.uint8)
    _check(_lib.ninfer_blocks_to_planes(_fmt(fmt), n, k, _np_ptr(blocks), blocks.size, _np_ptr(out), out.size))
    return out


def ninfer_planes_to_blocks(fmt, n: int, k: int, payload: np.ndarray) -> np.ndarray:
    payload = np.ascontiguousarray(payload, dtype=np.uint8).reshape(-1)
    g = ninfer_ternary_geometry(fmt, n, k)
    nb = 34 if _fmt(fmt) == PQ2_0_G128 else 28
    out = np.empty(n * g.groups_per_row * nb, dtype=np.uint8)
    _check(_lib.ninfer_planes_to_blocks(_fmt(fmt), n, k, _np_ptr(payload), payload.size, _np_ptr(out), out.size))
    return out


def ninfer_blocks_to_planes_device(fmt, n: int, k: int, blocks, out=None):
    """Device version of ninfer_blocks_to_planes: blocks is a uint8 CUDA tensor;
    returns (or fills) the uint8 CUDA payload tensor, on the current stream."""
    torch = _torch()
    g = ninfer_ternary_geometry(fmt, n, k)
    if out is None:
        out = torch.empty(g.payload_bytes, dtype=torch.uint8, device=blocks.device)
    _check(_lib.ninfer_blocks_to_planes_device(_fmt(fmt), n, k, _dev(blocks, "blocks"), blocks.numel(),
                                               _dev(out, "payload"), out.numel(), _stream(blocks)))
    return out


def ninfer_planes_to_blocks_device(fmt, n: int, k: int, payload, out=None):
    torch = _torch()
    g = ninfer_ternary_geometry(fmt, n, k)
    nb = 34 if _fmt(fmt) == PQ2_0_G128 else 28
    if out is None:
        out = torch.empty(n * g.groups_per_row * nb, dtype=torch.uint8, device=payload.device)
    _check(_lib.ninfer_planes_to_blocks_device(_fmt(fmt), n, k, _dev(payload, "payload"), payload.numel(),
                                               _dev(out, "blocks"), out.numel(), _stream(payload)))
    return out


def ninfer_device_errors(clear: bool = True) -> int:
    v = C.c_uint32()
    _check(_lib.ninfer_device_errors(C.byref(v), int(bool(clear))))
    return v.value


def ninfer_set_prefetch_before_dependency(enable: bool) -> None:
    _check(_lib.ninfer_set_prefetch_before_dependency(int(bool(enable))))


WAIT_LIMIT_DEFAULT = 4_000_000_000


def ninfer_set_wait_limit(cycles: int) -> None:
    _check(_lib.ninfer_set_wait_limit(int(cycles)))


# ---------------------------------------------------------------- device ---
def _torch():
    import torch
    return torch


def _dt(t) -> int:
    torch = _torch()
    return {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}[t]


def _stream(t):
    torch = _torch()
    return C.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dev(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return C.c_void_p(t.data_ptr())


def ninfer_validate_signs(signs) -> None:
    """Raise NinferError unless signs (host uint16/int16 bfloat16 bits, length K,
    K % 1024 == 0) holds only +1 and -1."""
    a = np.ascontiguousarray(np.asarray(signs).view(np.uint16).reshape(-1))
    _check(_lib.ninfer_validate_signs(a.ctypes.data_as(C.c_void_p), a.size))


def ninfer_hadamard_fwd(x, signs, out=None, out_dtype=None):
    """Forward signed block transform of a (M, K) CUDA tensor; signs is a (K,)
    CUDA tensor of bfloat16 +-1 (dtype bfloat16, int16 or uint16 bit patterns)."""
    return _hadamard(_lib.ninfer_hadamard_fwd, x, signs, out, out_dtype)


def ninfer_hadamard_inv(x, signs, out=None, out_dtype=None):
    return _hadamard(_lib.ninfer_hadamard_inv, x, signs, out, out_dtype)


def _hadamard(fn, x, signs, out, out_dtype):
    torch = _torch()
    x2 = x.reshape(-1, x.shape[-1])
    if out is None:
        out = torch.empty(x2.shape, dtype=out_dtype or torch.float32, device=x.device)
    _check(fn(_dev(x2, "x"), _dt(x2.dtype), _dev(out, "out"), _dt(out.dtype), _dev(signs, "signs"),
              x2.shape[0], x2.shape[1], _stream(x)))
    return out.reshape(x.shape[:-1] + (x.shape[-1],))


def ninfer_ternary_matmul_workspace(fmt, n: int, k: int, M: int, rotate: bool = True) -> int:
    b = C.c_uint64()
    _check(_lib.ninfer_ternary_matmul_workspace(_fmt(fmt), n, k, M, int(bool(rotate)), C.byref(b)))
    return b.value


def ninfer_ternary_matmul(fmt, payload, n: int, k: int, x, signs=None, y=None, y_dtype=None, workspace=None):
    """y (M, n) = ternary W (n, k) applied to the forward-transformed x (M, k)."""
    torch = _torch()
    x2 = x.reshape(-1, k)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, n), dtype=y_dtype or torch.float32, device=x.device)
    need = ninfer_ternary_matmul_workspace(fmt, n, k, M, signs is not None)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.ninfer_ternary_matmul(
        _fmt(fmt), _dev(payload, "payload"), payload.numel(), n, k, _dev(x2, "x"), _dt(x2.dtype),
        _dev(signs, "signs") if signs is not None else None, _dev(y, "y"), _dt(y.dtype), M,
        ws_ptr, ws_bytes, _stream(x)))
    return y


def ninfer_ternary_gate_up_workspace(fmt, n: int, k: int, M: int, rotate: bool, distinct_signs: bool) -> int:
    v = _u64()
    _check(_lib.ninfer_ternary_gate_up_workspace(_fmt(fmt), n, k, M, int(bool(rotate)), int(bool(distinct_signs)),
                                                 C.byref(v)))
    return v.value


def ninfer_ternary_gate_up(fmt, payload_gate, payload_up, n: int, k: int, x, signs_gate=None, signs_up=None, y=None,
                           y_dtype=None, workspace=None):
    """y (M, n) = silu(gate projection) * (up projection) of x (M, k); each
    projection rotates x with its own signs (both or neither given)."""
    torch = _torch()
    x2 = x.reshape(-1, k)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, n), dtype=y_dtype or torch.float32, device=x.device)
    distinct = signs_gate is not None and signs_up is not None and signs_gate.data_ptr() != signs_up.data_ptr()
    need = ninfer_ternary_gate_up_workspace(fmt, n, k, M, signs_gate is not None, distinct)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_ptr = _dev(workspace, "workspace") if need else None
    ws_bytes = workspace.numel() * workspace.element_size() if need else 0
    _check(_lib.ninfer_ternary_gate_up(
        _fmt(fmt), _dev(payload_gate, "payload_gate"), _dev(payload_up, "payload_up"), payload_gate.numel(), n, k,
        _dev(x2, "x"), _dt(x2.dtype), _dev(signs_gate, "signs_gate") if signs_gate is not None else None,
        _dev(signs_up, "signs_up") if signs_up is not None else None, _dev(y, "y"), _dt(y.dtype), M,
        ws_ptr, ws_bytes, _stream(x)))
    return y


def ninfer_ternary_matmul_noalloc(fmt, payload, n: int, k: int, x, signs=None, y=None, y_dtype=None):
    """As ninfer_ternary_matmul, for callers that cannot allocate device memory:
    the workspace comes from the library's fixed device array."""
    torch = _torch()
    x2 = x.reshape(-1, k)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, n), dtype=y_dtype or torch.float32, device=x.device)
    _check(_lib.ninfer_ternary_matmul_noalloc(
        _fmt(fmt), _dev(payload, "payload"), payload.numel(), n, k, _dev(x2, "x"), _dt(x2.dtype),
        _dev(signs, "signs") if signs is not None else None, _dev(y, "y"), _dt(y.dtype), M, _stream(x)))
    return y


def ninfer_ternary_embed(fmt, payload, n: int, k: int, ids, signs=None, out=None, out_dtype=None, status=None):
    """out (count, k) = inverse transform of the dequantised rows ids (int32 CUDA)."""
    torch = _torch()
    count = ids.numel()
    if out is None:
        out = torch.empty((count, k), dtype=out_dtype or torch.float32, device=ids.device)
    _check(_lib.ninfer_ternary_embed(
        _fmt(fmt), _dev(payload, "payload"), payload.numel(), n, k, _dev(ids, "ids"), count,
        _dev(signs, "signs") if signs is not None else None, _dev(out, "out"), _dt(out.dtype),
        _dev(status, "status") if status is not None else None, _stream(ids)))
    return out
