"""Python binding of libcpattn (causal blockwise ring attention on GB300).

Argument marshalling only: every computation runs in the library's CUDA kernels.
The functions carry the C names; tensors are torch tensors (or raw device
pointers as ints), the stream defaults to torch's current CUDA stream, and each
call returns the ``cpattn_status`` code (0 = OK).  ``check(status)`` turns a
non-zero code into ``CpattnError``.

The shared library is built in-tree by ``build_lib.build()``; importing this
package without it raises ImportError (there is no fallback).  With the
environment variable CPATTN_DEBUG_LIB=1 the package loads the CPATTN_DEBUG build
(``libcpattn_debug.so``, the same kernels with bounds checks) instead.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
DEBUG_LIB = os.environ.get("CPATTN_DEBUG_LIB") == "1"
LIB_PATH = os.path.join(_PKG, "libcpattn_debug.so" if DEBUG_LIB else "libcpattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = 0, 1, 2, 3, 4, 5
F32, BF16 = 0, 1
CONTIGUOUS, ZIGZAG = 0, 1
ZIGZAG_FWD, ZIGZAG_INV, A2A_FWD, A2A_INV = 0, 1, 2, 3


class CpattnDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("T", ctypes.c_int32), ("D", ctypes.c_int32), ("cp", ctypes.c_int32),
                ("a2a", ctypes.c_int32), ("layout", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("debug_fault", ctypes.c_int32)]


class CpattnError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"cpattn status {status}: {cpattn_status_string(status)}")
        self.status = status


def make_desc(B, H_q, H_kv, T, D, cp, layout="zigzag", dtype="bf16", a2a=1, scale=None,
              causal=1, debug_fault=0) -> CpattnDesc:
    lay = {"contiguous": CONTIGUOUS, "zigzag": ZIGZAG}.get(layout, layout)
    dt = {"f32": F32, "bf16": BF16}.get(dtype, dtype)
    return CpattnDesc(B, H_q, H_kv, T, D, cp, a2a, lay, dt,
                      1.0 / math.sqrt(D) if scale is None else scale, causal, debug_fault)


_vp = ctypes.c_void_p
_st = ctypes.c_int
_sigs = {
    "cpattn_partial_fwd": (_st, [ctypes.POINTER(CpattnDesc), ctypes.c_int, ctypes.c_int, _vp, _vp,
                                 _vp, _vp, _vp, _vp]),
    "cpattn_partial_bwd_workspace": (ctypes.c_size_t, [ctypes.POINTER(CpattnDesc)]),
    "cpattn_partial_bwd_stats": (_st, [ctypes.POINTER(CpattnDesc), _vp, _vp, _vp, _vp,
                                       ctypes.c_size_t, _vp]),
    "cpattn_partial_bwd": (_st, [ctypes.POINTER(CpattnDesc), ctypes.c_int, ctypes.c_int, _vp, _vp,
                                 _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_size_t,
                                 _vp]),
    "cpattn_merge": (_st, [ctypes.c_int64, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "cpattn_ring_fwd": (_st, [ctypes.POINTER(CpattnDesc), _vp, _vp, _vp, _vp, _vp, _vp]),
    "cpattn_ring_bwd_workspace": (ctypes.c_size_t, [ctypes.POINTER(CpattnDesc)]),
    "cpattn_ring_bwd": (_st, [ctypes.POINTER(CpattnDesc), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _vp, _vp, ctypes.c_size_t, _vp]),
    "cpattn_ring_bwd_noalloc": (_st, [ctypes.POINTER(CpattnDesc), _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp]),
    "cpattn_ring_step_host_workspace": (ctypes.c_size_t, [ctypes.POINTER(CpattnDesc)]),
    "cpattn_ring_step_host": (_st, [ctypes.POINTER(CpattnDesc), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "cpattn_packed_workspace": (ctypes.c_size_t, [ctypes.POINTER(CpattnDesc)]),
    "cpattn_ring_fwd_packed": (_st, [ctypes.POINTER(CpattnDesc), _vp, ctypes.c_int, _vp, _vp, _vp,
                                     _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "cpattn_ring_bwd_packed": (_st, [ctypes.POINTER(CpattnDesc), _vp, ctypes.c_int, _vp, _vp, _vp,
                                     _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "cpattn_allgather_fwd": (_st, [ctypes.POINTER(CpattnDesc), ctypes.c_int, _vp, _vp, _vp, _vp,
                                   _vp, _vp]),
    "cpattn_allgather_bwd_workspace": (ctypes.c_size_t, [ctypes.POINTER(CpattnDesc)]),
    "cpattn_allgather_bwd": (_st, [ctypes.POINTER(CpattnDesc), ctypes.c_int, _vp, _vp, _vp, _vp,
                                   _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_size_t,
                                   _vp]),
    "cpattn_layout": (_st, [ctypes.c_int, ctypes.POINTER(CpattnDesc), _vp, _vp, ctypes.c_int, _vp]),
    "cpattn_layout_batch": (_st, [ctypes.c_int, ctypes.POINTER(CpattnDesc), ctypes.c_int,
                                  ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                  ctypes.POINTER(ctypes.c_int), _vp]),
    "cpattn_check": (_st, [_vp]),
    "cpattn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "cpattn_timing_enable": (_st, [ctypes.c_int]),
    "cpattn_timing_collect": (_st, []),
    "cpattn_timing_count": (ctypes.c_int, []),
    "cpattn_timing_get": (_st, [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]),
    "cpattn_timing_reset": (_st, []),
}
for _name, (_res, _args) in _sigs.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int) -> None:
    if status != OK:
        raise CpattnError(status)


def cpattn_partial_fwd(desc, q_rank, kv_rank, q, k, v, o_part, lse_part, stream=None) -> int:
    return _lib.cpattn_partial_fwd(ctypes.byref(desc), q_rank, kv_rank, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(o_part), _ptr(lse_part), _stream(stream))


def cpattn_partial_bwd_workspace(desc) -> int:
    return _lib.cpattn_partial_bwd_workspace(ctypes.byref(desc))


def cpattn_partial_bwd_stats(desc, o, lse, dO, workspace, ws_bytes=None, stream=None) -> int:
    return _lib.cpattn_partial_bwd_stats(ctypes.byref(desc), _ptr(o), _ptr(lse), _ptr(dO),
                                         _ptr(workspace), _ws_bytes(workspace, ws_bytes),
                                         _stream(stream))


def cpattn_partial_bwd(desc, q_rank, kv_rank, q, k, v, dO, dq_part, dk_part, dv_part, accumulate,
                       workspace, ws_bytes=None, stream=None) -> int:
    return _lib.cpattn_partial_bwd(ctypes.byref(desc), q_rank, kv_rank, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(dO), _ptr(dq_part), _ptr(dk_part), _ptr(dv_part),
                                   int(accumulate), _ptr(workspace),
                                   _ws_bytes(workspace, ws_bytes), _stream(stream))


def cpattn_merge(rows, D, o_a, lse_a, o_b, lse_b, o_out, lse_out, stream=None) -> int:
    return _lib.cpattn_merge(rows, D, _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out),
                             _ptr(lse_out), _stream(stream))


def cpattn_ring_fwd(desc, q, k, v, o, lse, stream=None) -> int:
    return _lib.cpattn_ring_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                _stream(stream))


def cpattn_ring_bwd_workspace(desc) -> int:
    return _lib.cpattn_ring_bwd_workspace(ctypes.byref(desc))


def cpattn_ring_bwd(desc, q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes=None,
                    stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    return _lib.cpattn_ring_bwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), ws_bytes,
                                _stream(stream))


def cpattn_ring_bwd_noalloc(desc, q, k, v, o, lse, dO, dq, dk, dv, stream=None) -> int:
    """The backward without a caller workspace (for callers that cannot allocate
    device memory): the library's own 16 MiB scratch per device is used instead."""
    return _lib.cpattn_ring_bwd_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                        _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                                        _stream(stream))


def cpattn_ring_step_host_workspace(desc) -> int:
    return _lib.cpattn_ring_step_host_workspace(ctypes.byref(desc))


def cpattn_ring_step_host(desc, q, k, v, dO, o, lse, dq, dk, dv, workspace, ws_bytes=None,
                          stream=None) -> int:
    """One fwd+bwd step over HOST tensors (natural order; pinned for overlap): uploads,
    permutes, ring forward and backward, permutes back and downloads, the transfers
    overlapping the compute."""
    return _lib.cpattn_ring_step_host(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(dO),
                                      _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                                      _ptr(workspace), _ws_bytes(workspace, ws_bytes),
                                      _stream(stream))


def cpattn_packed_workspace(desc) -> int:
    return _lib.cpattn_packed_workspace(ctypes.byref(desc))


def _ws_bytes(workspace, ws_bytes):
    return workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes


def cpattn_ring_fwd_packed(desc, starts, n_docs, q, k, v, o, lse, workspace, ws_bytes=None,
                           stream=None) -> int:
    return _lib.cpattn_ring_fwd_packed(ctypes.byref(desc), _ptr(starts), n_docs, _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                       _ws_bytes(workspace, ws_bytes), _stream(stream))


def cpattn_ring_bwd_packed(desc, starts, n_docs, q, k, v, o, lse, dO, dq, dk, dv, workspace,
                           ws_bytes=None, stream=None) -> int:
    return _lib.cpattn_ring_bwd_packed(ctypes.byref(desc), _ptr(starts), n_docs, _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                       _ptr(dv), _ptr(workspace), _ws_bytes(workspace, ws_bytes),
                                       _stream(stream))


def cpattn_allgather_fwd(desc, q_rank, q, k, v, o, lse, stream=None) -> int:
    return _lib.cpattn_allgather_fwd(ctypes.byref(desc), q_rank, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                     _ptr(lse), _stream(stream))


def cpattn_allgather_bwd_workspace(desc) -> int:
    return _lib.cpattn_allgather_bwd_workspace(ctypes.byref(desc))


def cpattn_allgather_bwd(desc, q_rank, q, k, v, o, lse, dO, dq, dk_sum, dv_sum, accumulate,
                         workspace, ws_bytes=None, stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    return _lib.cpattn_allgather_bwd(ctypes.byref(desc), q_rank, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                     _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk_sum), _ptr(dv_sum),
                                     int(accumulate), _ptr(workspace), ws_bytes, _stream(stream))


def cpattn_layout(permute, desc, src, dst, n_heads, stream=None) -> int:
    return _lib.cpattn_layout(permute, ctypes.byref(desc), _ptr(src), _ptr(dst), n_heads,
                              _stream(stream))


def cpattn_layout_batch(permute, desc, srcs, dsts, n_heads, stream=None) -> int:
    """cpattn_layout over several tensors at once: srcs[i] -> dsts[i], n_heads[i] heads."""
    n = len(srcs)
    if len(dsts) != n or len(n_heads) != n:
        raise ValueError("srcs, dsts and n_heads must have the same length")
    src_arr = (_vp * n)(*[_ptr(x) for x in srcs])
    dst_arr = (_vp * n)(*[_ptr(x) for x in dsts])
    heads = (ctypes.c_int * n)(*[int(h) for h in n_heads])
    return _lib.cpattn_layout_batch(permute, ctypes.byref(desc), n, src_arr, dst_arr, heads,
                                    _stream(stream))


def cpattn_check(stream=None) -> int:
    return _lib.cpattn_check(_stream(stream))


def cpattn_status_string(status: int) -> str:
    return _lib.cpattn_status_string(status).decode()


def cpattn_timing_enable(on: bool) -> int:
    return _lib.cpattn_timing_enable(1 if on else 0)


def cpattn_timing_collect() -> int:
    return _lib.cpattn_timing_collect()


def cpattn_timing_reset() -> int:
    return _lib.cpattn_timing_reset()


def cpattn_timing_table() -> dict:
    """{kernel name: (total ms, launches)} accumulated since the last reset."""
    out = {}
    for i in range(_lib.cpattn_timing_count()):
        name = ctypes.c_char_p()
        ms = ctypes.c_double()
        n = ctypes.c_int64()
        check(_lib.cpattn_timing_get(i, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(n)))
        out[name.value.decode()] = (ms.value, n.value)
    return out
