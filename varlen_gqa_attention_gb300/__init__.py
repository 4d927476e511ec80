"""Length-aware GQA attention over a per-sequence KV column store, for GB300 (sm_103a).

A thin ctypes binding over ``libsdpa_varlen.so`` (C interface in include/sdpa_varlen.h):
it only checks tensor dtypes/devices, reads strides and pointers, allocates outputs and
workspace with torch, and passes the given (else the current) CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; there is no other implementation to fall back on, so a
missing library is an error.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "sdpa_varlen", "sdpa_varlen_modes", "sdpa_varlen_append", "sdpa_seq_clone", "sdpa_causal_prefill",
    "sdpa_varlen_splitk_static", "workspace_bytes", "workspace_status", "prefill_available", "set_route_policy",
    "set_timing_events", "library",
    "SDPA_OK", "SEG_BAD_QRANGE", "SEG_BAD_COL", "SEG_BAD_KV", "SEG_SPAN", "SEG_OVERLAP",
    "DEV_TIMEOUT", "ROUTE_AUTO", "ROUTE_SPLITK", "ROUTE_PREFILL", "SdpaError",
]

SDPA_OK = 0
SEG_BAD_QRANGE, SEG_BAD_COL, SEG_BAD_KV, SEG_SPAN, SEG_OVERLAP, DEV_TIMEOUT = 1, 2, 4, 8, 16, 32
ROUTE_AUTO, ROUTE_SPLITK, ROUTE_PREFILL = 0, 1, 2

STATUS_NAMES = {
    0: "SDPA_OK", 1: "SDPA_ERR_NULL", 2: "SDPA_ERR_SHAPE", 3: "SDPA_ERR_HEAD_DIM", 4: "SDPA_ERR_GQA",
    5: "SDPA_ERR_STRIDE", 6: "SDPA_ERR_ALIGN", 7: "SDPA_ERR_WORKSPACE", 8: "SDPA_ERR_ARG",
    9: "SDPA_ERR_CUDA",
}

EXPORTS = [
    "sdpa_varlen_workspace_bytes", "sdpa_varlen", "sdpa_causal_prefill", "sdpa_set_route_policy",
    "sdpa_set_timing_events", "sdpa_last_error", "sdpa_version", "sdpa_varlen_splitk_static",
    "sdpa_varlen_append", "sdpa_seq_clone", "sdpa_varlen_modes", "sdpa_prefill_available",
    "sdpa_workspace_status",
]


class SdpaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib: Optional[ctypes.CDLL] = None


def library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libsdpa_varlen.so (building it first when it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.lib_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"{path} is missing; run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    c_i64, c_int, c_vp, c_f = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
    lib.sdpa_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.sdpa_varlen_workspace_bytes.argtypes = [c_i64, c_int, c_int, c_int, c_int]
    lib.sdpa_varlen.restype = c_int
    lib.sdpa_varlen.argtypes = [c_vp, c_i64, c_int, c_int, c_i64, c_i64, c_vp, c_vp, c_i64, c_int,
                                c_int, c_vp, c_int, c_int, c_int, c_f, c_vp, c_i64, c_i64, c_vp,
                                ctypes.c_size_t, c_vp, c_vp]
    lib.sdpa_varlen_append.restype = c_int
    lib.sdpa_varlen_append.argtypes = [c_vp, c_i64, c_int, c_int, c_i64, c_i64, c_vp, c_vp, c_i64, c_i64,
                                       c_vp, c_vp, c_i64, c_int, c_int, c_vp, c_int, c_int, c_int, c_f,
                                       c_vp, c_i64, c_i64, c_vp, ctypes.c_size_t, c_vp, c_vp]
    lib.sdpa_varlen_modes.restype = c_int
    lib.sdpa_varlen_modes.argtypes = [c_vp, c_i64, c_int, c_int, c_i64, c_i64, c_vp, c_vp, c_i64, c_int,
                                      c_int, c_vp, c_vp, c_int, c_f, c_vp, c_i64, c_i64, c_vp,
                                      ctypes.c_size_t, c_vp, c_vp]
    lib.sdpa_seq_clone.restype = c_int
    lib.sdpa_seq_clone.argtypes = [c_vp, c_vp, c_i64, c_int, c_int, c_int, c_int, c_int, c_i64, c_vp]
    lib.sdpa_causal_prefill.restype = c_int
    lib.sdpa_causal_prefill.argtypes = [c_vp, c_vp, c_vp, c_i64, c_i64, c_int, c_int, c_int, c_f,
                                        c_vp, c_vp, ctypes.c_size_t, c_vp]
    lib.sdpa_set_route_policy.restype = c_int
    lib.sdpa_set_route_policy.argtypes = [c_int]
    lib.sdpa_set_timing_events.restype = c_int
    lib.sdpa_set_timing_events.argtypes = [ctypes.POINTER(c_vp), c_int]
    lib.sdpa_last_error.restype = ctypes.c_char_p
    lib.sdpa_last_error.argtypes = []
    lib.sdpa_prefill_available.restype = c_int
    lib.sdpa_prefill_available.argtypes = [c_int]
    lib.sdpa_version.restype = c_int
    lib.sdpa_version.argtypes = []
    lib.sdpa_varlen_splitk_static.restype = c_int
    lib.sdpa_varlen_splitk_static.argtypes = [c_vp, c_i64, c_int, c_int, c_i64, c_i64, c_vp, c_vp, c_i64, c_int,
                                              c_int, c_vp, c_int, c_int, c_int, c_f, c_vp, c_i64, c_i64, c_vp,
                                              c_vp]
    lib.sdpa_workspace_status.restype = c_int
    lib.sdpa_workspace_status.argtypes = [c_vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int32), c_vp]
    _lib = lib
    return lib


def _check(code: int):
    if code != SDPA_OK:
        raise SdpaError(code, library().sdpa_last_error().decode())


def workspace_bytes(T: int, Hq: int, Hkv: int, D: int, S: int) -> int:
    return int(library().sdpa_varlen_workspace_bytes(T, Hq, Hkv, D, S))


def workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Status word of the last call that used ``workspace``: its SDPA_SEG_* bits and
    DEV_TIMEOUT.  Waits for the stream, so it is not for use inside graph capture."""
    v = ctypes.c_int32(0)
    _check(library().sdpa_workspace_status(workspace.data_ptr(), workspace.numel(), ctypes.byref(v),
                                           _stream_ptr(stream)))
    return int(v.value)


def prefill_available(D: int) -> bool:
    """Whether the tensor-memory prefill kernel runs for head dim D on the current device."""
    lib = library()
    r = lib.sdpa_prefill_available(D)
    if r < 0:
        raise SdpaError(9 if D in (64, 128, 256) else 3, lib.sdpa_last_error().decode())
    return r == 1


def set_route_policy(policy: int) -> None:
    _check(library().sdpa_set_route_policy(policy))


def set_timing_events(events) -> None:
    """Record 5 torch.cuda.Event objects at the kernel boundaries of this thread's next calls
    (scheduler | prefill | split-K | combine); ``None`` switches the hook off."""
    lib = library()
    if events is None:
        _check(lib.sdpa_set_timing_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib.sdpa_set_timing_events(arr, len(events)))


def _on_stream(t: torch.Tensor, stream) -> torch.Tensor:
    """A tensor this module allocated on the current stream and hands to work on `stream`:
    the caching allocator must not reuse its memory before that work is done."""
    if stream is not None:
        t.record_stream(stream)
    return t


def _workspace(nbytes: int, device, stream=None) -> torch.Tensor:
    return _on_stream(torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device), stream)


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check_attention_args(q, k_store, v_store, seq_info, out=None, seg_mode=None):
    """The tensor checks every attention entry makes before its C call: shapes, dtypes
    (bf16 data, int32 tables), layouts (contiguous stores and tables, unit inner strides) and
    one CUDA device for all of them.  Raises ValueError; returns (T, Hq, D, rows, cols, Hkv, S)."""
    if q.dim() != 3 or k_store.dim() != 4 or tuple(v_store.shape) != tuple(k_store.shape):
        raise ValueError("q must be [T, Hq, D] and the stores [rows, cols, Hkv, D]")
    for name, t in (("q", q), ("k_store", k_store), ("v_store", v_store)):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bf16, not {t.dtype}")
    T, Hq, D = q.shape
    rows, cols, Hkv, Dk = k_store.shape
    if Dk != D:
        raise ValueError("head dims of q and the stores differ")
    if q.stride(2) != 1:
        raise ValueError("q must have unit inner stride")
    if not (k_store.is_contiguous() and v_store.is_contiguous()):
        raise ValueError("k_store and v_store must be contiguous")
    if seq_info.dtype != torch.int32 or not seq_info.is_contiguous() or \
            (seq_info.numel() and (seq_info.dim() != 2 or seq_info.shape[1] != 4)):
        raise ValueError("seq_info must be a contiguous int32 [S, 4] tensor")
    S = seq_info.shape[0] if seq_info.numel() else 0
    if out is not None and (out.dtype != torch.bfloat16 or tuple(out.shape) != (T, Hq, D) or out.stride(2) != 1):
        raise ValueError("out must be bf16 [T, Hq, D] with unit inner stride")
    if seg_mode is not None:
        if seg_mode.dtype != torch.int32 or not seg_mode.is_contiguous() or (S and tuple(seg_mode.shape) != (S, 2)):
            raise ValueError("seg_mode must be a contiguous int32 [S, 2] tensor")
    tensors = [q, k_store, v_store, seq_info] + [t for t in (out, seg_mode) if t is not None]
    if not all(t.is_cuda for t in tensors) or len({t.device for t in tensors}) != 1:
        raise ValueError("every tensor must be on the same CUDA device")
    return T, Hq, D, rows, cols, Hkv, S


def sdpa_varlen(q: torch.Tensor, k_store: torch.Tensor, v_store: torch.Tensor, seq_info: torch.Tensor,
                *, causal: bool, window: int = 0, scale: Optional[float] = None,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[T, Hq, D] = length-aware GQA attention of q over the column stores.

    q: bf16 [T, Hq, D] (inner stride 1); k_store, v_store: bf16 [rows, cols, Hkv, D]
    contiguous; seq_info: int32 [S, 4] contiguous on the same device.  ``status`` (an int32
    device tensor, optional) receives the OR of the device status bits.
    """
    T, Hq, D, rows, cols, Hkv, S = _check_attention_args(q, k_store, v_store, seq_info, out)
    lib = library()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = _on_stream(torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q.device), stream)
    need = workspace_bytes(T, Hq, Hkv, D, S)
    if workspace is None:
        workspace = _workspace(need, q.device, stream)
    st_ptr = status.data_ptr() if status is not None else None
    code = lib.sdpa_varlen(q.data_ptr(), T, Hq, D, q.stride(0), q.stride(1), k_store.data_ptr(),
                           v_store.data_ptr(), rows, cols, Hkv, seq_info.data_ptr() if S else None,
                           S, int(bool(causal)), int(window), float(scale), out.data_ptr(),
                           out.stride(0), out.stride(1), workspace.data_ptr(), workspace.numel(),
                           st_ptr, _stream_ptr(stream))
    _check(code)
    return out


def sdpa_varlen_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_store: torch.Tensor,
                       v_store: torch.Tensor, seq_info: torch.Tensor, *, causal: bool, window: int = 0,
                       scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """Write the step's keys and values into the stores, then attend (one enqueued call).

    k_new, v_new: bf16 [T, Hkv, D] (inner stride 1), row t the new key / value of packed
    query row t; they go to store row (kv_end - q_len + i) % rows of each live segment's
    column.  The stores are modified in place; everything else is as ``sdpa_varlen``.
    """
    T, Hq, D, rows, cols, Hkv, S = _check_attention_args(q, k_store, v_store, seq_info, out)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.device != q.device:
            raise ValueError(f"{name} must be a bf16 tensor on q's CUDA device")
    if tuple(k_new.shape) != (T, Hkv, D) or tuple(v_new.shape) != (T, Hkv, D):
        raise ValueError("k_new and v_new must be [T, Hkv, D]")
    if k_new.stride() != v_new.stride() or k_new.stride(2) != 1:
        raise ValueError("k_new and v_new must share strides, with unit inner stride")
    lib = library()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = _on_stream(torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q.device), stream)
    if workspace is None:
        workspace = _workspace(workspace_bytes(T, Hq, Hkv, D, S), q.device, stream)
    st_ptr = status.data_ptr() if status is not None else None
    code = lib.sdpa_varlen_append(q.data_ptr(), T, Hq, D, q.stride(0), q.stride(1), k_new.data_ptr(),
                                  v_new.data_ptr(), k_new.stride(0), k_new.stride(1), k_store.data_ptr(),
                                  v_store.data_ptr(), rows, cols, Hkv, seq_info.data_ptr() if S else None,
                                  S, int(bool(causal)), int(window), float(scale), out.data_ptr(),
                                  out.stride(0), out.stride(1), workspace.data_ptr(), workspace.numel(),
                                  st_ptr, _stream_ptr(stream))
    _check(code)
    return out


def sdpa_varlen_modes(q: torch.Tensor, k_store: torch.Tensor, v_store: torch.Tensor, seq_info: torch.Tensor,
                      seg_mode: torch.Tensor, *, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """``sdpa_varlen`` with a mask mode per segment: seg_mode int32 [S, 2] = (causal, window)
    on the device, in place of the call's causal / window."""
    T, Hq, D, rows, cols, Hkv, S = _check_attention_args(q, k_store, v_store, seq_info, out, seg_mode)
    lib = library()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = _on_stream(torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q.device), stream)
    if workspace is None:
        workspace = _workspace(workspace_bytes(T, Hq, Hkv, D, S), q.device, stream)
    st_ptr = status.data_ptr() if status is not None else None
    code = lib.sdpa_varlen_modes(q.data_ptr(), T, Hq, D, q.stride(0), q.stride(1), k_store.data_ptr(),
                                 v_store.data_ptr(), rows, cols, Hkv, seq_info.data_ptr() if S else None,
                                 seg_mode.data_ptr() if S else None, S, float(scale), out.data_ptr(),
                                 out.stride(0), out.stride(1), workspace.data_ptr(), workspace.numel(),
                                 st_ptr, _stream_ptr(stream))
    _check(code)
    return out


def sdpa_seq_clone(k_store: torch.Tensor, v_store: torch.Tensor, src_col: int, dst_col: int, n: int,
                   stream=None) -> None:
    """Column dst_col of both stores takes over the first n positions of column src_col
    (ring-aware: store rows [0, min(n, rows)) are copied).  In place, on the device."""
    lib = library()
    if k_store.dim() != 4 or tuple(v_store.shape) != tuple(k_store.shape):
        raise ValueError("the stores must both be [rows, cols, Hkv, D]")
    for name, t in (("k_store", k_store), ("v_store", v_store)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    rows, cols, Hkv, D = k_store.shape
    _check(lib.sdpa_seq_clone(k_store.data_ptr(), v_store.data_ptr(), rows, cols, Hkv, D, int(src_col),
                              int(dst_col), int(n), _stream_ptr(stream)))


def sdpa_causal_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
                        *, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """Dense causal GQA attention: q [Lq, Hq, D] against k, v [Lkv, Hkv, D], queries being
    the last Lq positions.  All tensors contiguous bf16 on one CUDA device."""
    lib = library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous 3-d bf16 CUDA tensor")
    Lq, Hq, D = q.shape
    Lkv, Hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = _on_stream(torch.empty_like(q), stream)
    need = workspace_bytes(Lq, Hq, Hkv, D, 1)
    if workspace is None:
        workspace = _workspace(need, q.device, stream)
    code = lib.sdpa_causal_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), Lq, Lkv, Hq, Hkv, D,
                                   float(scale), out.data_ptr(), workspace.data_ptr(),
                                   workspace.numel(), _stream_ptr(stream))
    _check(code)
    return out


def sdpa_varlen_splitk_static(q: torch.Tensor, k_store: torch.Tensor, v_store: torch.Tensor,
                              seq_info: torch.Tensor, *, causal: bool, window: int = 0,
                              scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                              status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """sdpa_varlen for callers that cannot allocate device scratch: the library's own static
    device array (SDPA_STATIC_SCRATCH_BYTES) serves as the workspace and every segment runs on
    the split-K kernel.  Pass ``out`` to allocate nothing at all.  Calls must not overlap on
    the GPU (they share the array); make the first call on a device outside stream capture.
    The tensors are checked as for ``sdpa_varlen``."""
    T, Hq, D, rows, cols, Hkv, S = _check_attention_args(q, k_store, v_store, seq_info, out)
    if status is not None and (status.dtype != torch.int32 or status.device != q.device):
        raise ValueError("status must be an int32 tensor on q's CUDA device")
    lib = library()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = _on_stream(torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q.device), stream)
    code = lib.sdpa_varlen_splitk_static(
        q.data_ptr(), T, Hq, D, q.stride(0), q.stride(1), k_store.data_ptr(), v_store.data_ptr(), rows, cols, Hkv,
        seq_info.data_ptr() if S else None, S, int(bool(causal)), int(window), float(scale), out.data_ptr(),
        out.stride(0), out.stride(1), status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(code)
    return out
