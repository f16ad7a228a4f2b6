"""Thin Python binding of ``libridgefill.so`` (argument marshalling only).

The functions take torch tensors for device memory and streams, check their
dtype, device and layout, fill the C argument structs and call the library.
Every step of the fill and the fit runs in the library's CUDA kernels; there
is no fallback: if the library is missing or fails to load, these functions
raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

from . import build as _build

_libs = {}
_use_debug = False

RF_FIT_ACCUMULATE = 1
RF_FIT_SOLVE = 2

STATUS = {
    0: "RF_OK", 1: "RF_ERR_ARG", 2: "RF_ERR_SHAPE", 3: "RF_ERR_ALIGN", 4: "RF_ERR_NOT_PINNED",
    5: "RF_ERR_CUDA", 6: "RF_ERR_TIMEOUT", 7: "RF_ERR_NUMERIC", 8: "RF_ERR_WORKSPACE",
    9: "RF_ERR_SOURCE", 10: "RF_ERR_BOUNDS",
}

_vp = ctypes.c_void_p

# int32_t (*)(void* user, int32_t layer, void* dst, size_t bytes): the host map source
MAP_SOURCE_FN = ctypes.CFUNCTYPE(ctypes.c_int32, _vp, ctypes.c_int32, _vp, ctypes.c_size_t)


class FillArgs(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("d_in", ctypes.c_int32), ("d_out", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("maps_on_host", ctypes.c_int32), ("rows", ctypes.c_int64), ("pos0", ctypes.c_int64),
        ("cache_len", ctypes.c_int64), ("rows_per_chunk", ctypes.c_int64),
        ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double),
        ("H", _vp), ("A", _vp), ("bias", _vp), ("gain", _vp), ("Wk", _vp), ("Wv", _vp),
        ("Kc", _vp), ("Vc", _vp), ("stage_events", _vp), ("copy_events", _vp),
        ("k_scale", _vp), ("v_scale", _vp), ("A_scale", _vp), ("row_idx", _vp),
        ("h_rows", ctypes.c_int64), ("h_on_host", ctypes.c_int32),
        ("q8_group_layers", ctypes.c_int32), ("map_source", MAP_SOURCE_FN),
        ("map_source_user", _vp), ("map_staging", _vp), ("host_wait_ms", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class GdnArgs(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("d_in", ctypes.c_int32), ("d_out", ctypes.c_int32),
        ("n_heads", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
        ("chunk", ctypes.c_int32), ("maps_on_host", ctypes.c_int32),
        ("rows", ctypes.c_int64), ("rows_per_chunk", ctypes.c_int64),
        ("rms_eps", ctypes.c_double), ("l2_eps", ctypes.c_double),
        ("H", _vp), ("A", _vp), ("bias", _vp), ("gain", _vp), ("Wk", _vp), ("Wv", _vp),
        ("Wa", _vp), ("Wb", _vp), ("S0", _vp), ("S", _vp), ("stage_events", _vp),
        ("A_scale", _vp), ("exact_idx", _vp), ("n_exact", ctypes.c_int64), ("X_exact", _vp),
        ("rho", _vp), ("delta_M", _vp), ("h_on_host", ctypes.c_int32),
        ("q8_group_layers", ctypes.c_int32),
    ]


class FitArgs(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("d_in", ctypes.c_int32), ("d_out", ctypes.c_int32),
        ("flags", ctypes.c_int32), ("rows", ctypes.c_int64), ("lam", ctypes.c_double),
        ("X", _vp), ("Y", _vp), ("G", _vp), ("C", _vp), ("sx", _vp), ("sy", _vp),
        ("count", _vp), ("A_out", _vp), ("A_out_f32", _vp), ("b_out", _vp), ("alpha_out", _vp),
    ]


class RescaleArgs(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("d_in", ctypes.c_int32), ("d_out", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("which", ctypes.c_int32),
        ("tail_rows", ctypes.c_int64), ("rows", ctypes.c_int64), ("pos0", ctypes.c_int64),
        ("cache_len", ctypes.c_int64), ("rms_eps", ctypes.c_double),
        ("H_tail", _vp), ("X_true", _vp), ("A", _vp), ("bias", _vp), ("gain", _vp),
        ("Wk", _vp), ("Wv", _vp), ("Kc", _vp), ("Vc", _vp), ("scale", _vp), ("A_scale", _vp),
    ]


class QuantizeArgs(ctypes.Structure):
    _fields_ = [
        ("n_maps", ctypes.c_int32), ("d_out", ctypes.c_int32), ("d_in", ctypes.c_int32),
        ("src_bf16", ctypes.c_int32), ("A", _vp), ("q", _vp), ("scale", _vp),
    ]


RF_RESCALE_VALUES, RF_RESCALE_KEYS = 1, 2
Q8_GROUP = 128  # map weights of a row sharing one bf16 scale


class RidgeFillError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


# the argument structs below match include/ridgefill.h at this version
ABI_VERSION = 10


def library_path(debug: Optional[bool] = None) -> str:
    return _build.LIB_DEBUG if (_use_debug if debug is None else debug) else _build.LIB


@contextlib.contextmanager
def debug_library():
    """Within the block every call of this binding goes through ``libridgefill_debug.so``:
    the same kernels with every plain global store checked against its buffer and guard
    bands around the workspace regions (reported as RF_ERR_BOUNDS by device_error)."""
    global _use_debug
    prev, _use_debug = _use_debug, True
    try:
        yield load()
    finally:
        _use_debug = prev


def load(rebuild: bool = True, debug: Optional[bool] = None) -> ctypes.CDLL:
    """Load ``libridgefill.so`` (building it first if it is stale); with ``debug`` (or
    inside :func:`debug_library`) the debug build of the same sources."""
    dbg = _use_debug if debug is None else debug
    if dbg in _libs:
        return _libs[dbg]
    path = _build.build(debug=dbg) if rebuild else library_path(dbg)
    if not os.path.exists(path):
        raise RuntimeError(f"RidgeFill CUDA library not found at {path}")
    lib = ctypes.CDLL(path)
    lib.ridgefill_fill_workspace_size.argtypes = [ctypes.POINTER(FillArgs)]
    lib.ridgefill_fill_workspace_size.restype = ctypes.c_size_t
    lib.ridgefill_fill.argtypes = [ctypes.POINTER(FillArgs), _vp, ctypes.c_size_t, _vp]
    lib.ridgefill_fill.restype = ctypes.c_int
    lib.ridgefill_gdn_workspace_size.argtypes = [ctypes.POINTER(GdnArgs)]
    lib.ridgefill_gdn_workspace_size.restype = ctypes.c_size_t
    lib.ridgefill_fill_gdn.argtypes = [ctypes.POINTER(GdnArgs), _vp, ctypes.c_size_t, _vp]
    lib.ridgefill_fill_gdn.restype = ctypes.c_int
    lib.ridgefill_fit_workspace_size.argtypes = [ctypes.POINTER(FitArgs)]
    lib.ridgefill_fit_workspace_size.restype = ctypes.c_size_t
    lib.ridgefill_fit.argtypes = [ctypes.POINTER(FitArgs), _vp, ctypes.c_size_t, _vp]
    lib.ridgefill_fit.restype = ctypes.c_int
    lib.ridgefill_rescale_workspace_size.argtypes = [ctypes.POINTER(RescaleArgs)]
    lib.ridgefill_rescale_workspace_size.restype = ctypes.c_size_t
    lib.ridgefill_rescale.argtypes = [ctypes.POINTER(RescaleArgs), _vp, ctypes.c_size_t, _vp]
    lib.ridgefill_rescale.restype = ctypes.c_int
    lib.ridgefill_quantize_maps.argtypes = [ctypes.POINTER(QuantizeArgs), _vp]
    lib.ridgefill_quantize_maps.restype = ctypes.c_int
    lib.ridgefill_wait_selftest.argtypes = [ctypes.c_int32, _vp]
    lib.ridgefill_wait_selftest.restype = ctypes.c_int
    lib.ridgefill_workspace_size.argtypes = [ctypes.c_int32, _vp]
    lib.ridgefill_workspace_size.restype = ctypes.c_size_t
    lib.ridgefill_status_string.argtypes = [ctypes.c_int]
    lib.ridgefill_status_string.restype = ctypes.c_char_p
    lib.ridgefill_last_error.argtypes = []
    lib.ridgefill_last_error.restype = ctypes.c_char_p
    lib.ridgefill_device_error.argtypes = [_vp, ctypes.POINTER(ctypes.c_int)]
    lib.ridgefill_device_error.restype = ctypes.c_int
    lib.ridgefill_compute_share.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                            ctypes.c_int64]
    lib.ridgefill_compute_share.restype = ctypes.c_double
    lib.ridgefill_abi_version.argtypes = []
    lib.ridgefill_abi_version.restype = ctypes.c_int32
    if lib.ridgefill_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{path} has ABI version {lib.ridgefill_abi_version()}, this binding "
                           f"expects {ABI_VERSION}: rebuild the library")
    _libs[dbg] = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        raise RidgeFillError(status, load().ridgefill_last_error().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_maps(A, A_scale) -> bool:
    """Maps are bf16 [L, d_out, d_in], or int8 codes with group-major bf16 scales
    [L, d_in / 128, d_out] when ``A_scale`` is given; device tensors, or pinned
    host tensors to stream.  Returns whether they live in host memory."""
    host = not A.is_cuda
    L, d_out, d_in = A.shape
    items = [(A, "A", torch.int8 if A_scale is not None else torch.bfloat16, None)]
    if A_scale is not None:
        items.append((A_scale, "A_scale", torch.bfloat16, (L, d_in // Q8_GROUP, d_out)))
    for t, name, dt, shape in items:
        if host:
            if t.is_cuda or t.dtype != dt or not t.is_contiguous() or not t.is_pinned():
                raise ValueError(f"host {name} must be contiguous, pinned {dt}")
            if shape is not None and tuple(t.shape) != shape:
                raise ValueError(f"{name} must have shape {shape}")
        else:
            _dev(t, name, dt, shape)
    return host


def map_slot_bytes(d_out: int, d_in: int, int8: bool) -> int:
    """Bytes of one layer's map as a host map source writes it: bf16 [d_out, d_in], or int8
    codes followed, at a 256-byte boundary, by the bf16 scales [d_in / 128, d_out]."""
    n = d_out * d_in
    return 2 * n if not int8 else (n + 255) // 256 * 256 + d_out * (d_in // Q8_GROUP) * 2


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _event_array(events):
    if events is None:
        return None
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return arr


def fill_args(H, A, bias, gain, Wk, Wv, Kc, Vc, *, head_dim: int, rope_theta: float,
              rms_eps: float, pos0: int = 0, rows_per_chunk: int = 0,
              stage_events=None, copy_events=None, k_scale=None, v_scale=None,
              A_scale=None, row_idx=None, q8_group_layers: int = 0, map_source=None,
              map_staging=None, host_wait_ms: int = 0, map_shape=None) -> FillArgs:
    """With ``map_source`` (a callable ``(layer, dst_address, nbytes) -> int``) the maps
    come from the host one layer at a time through the pinned ``map_staging`` buffer;
    ``A`` may then be None, with ``map_shape`` = (L, d_out, d_in) giving the sizes."""
    if map_source is not None and A is None:
        L, d_out, d_in = map_shape
    else:
        L, d_out, d_in = A.shape
    rows = H.shape[0] if row_idx is None else row_idx.shape[0]
    h_rows = H.shape[0] if row_idx is not None else 0
    if row_idx is not None:
        _dev(row_idx, "row_idx", torch.int32, (rows,))
    n_kv = Kc.shape[1]
    cache_len = Kc.shape[2]
    h_host = not H.is_cuda
    if h_host:
        if H.dtype != torch.bfloat16 or not H.is_contiguous() or not H.is_pinned():
            raise ValueError("host H must be contiguous, pinned bf16")
        if tuple(H.shape) != (H.shape[0], d_in):
            raise ValueError("H must be [rows, d_in]")
    else:
        _dev(H, "H", torch.bfloat16, (H.shape[0], d_in))
    if map_source is not None:
        host = True
        if map_staging is None or map_staging.is_cuda or not map_staging.is_pinned():
            raise ValueError("map_source needs a pinned host map_staging buffer")
        need = 2 * map_slot_bytes(d_out, d_in, A_scale is not None)
        if map_staging.numel() * map_staging.element_size() < need:
            raise ValueError(f"map_staging needs {need} bytes (two layers)")
        if A is not None:
            _check_maps(A, A_scale)
    else:
        host = _check_maps(A, A_scale)
    _dev(bias, "bias", torch.float32, (L, d_out))
    if gain is not None:
        _dev(gain, "gain", torch.bfloat16, (L, d_out))
    _dev(Wk, "Wk", torch.bfloat16, (L, n_kv * head_dim, d_out))
    _dev(Wv, "Wv", torch.bfloat16, (L, n_kv * head_dim, d_out))
    _dev(Kc, "Kc", torch.bfloat16, (L, n_kv, cache_len, head_dim))
    _dev(Vc, "Vc", torch.bfloat16, (L, n_kv, cache_len, head_dim))
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t is not None:
            _dev(t, name, torch.float32, (L, n_kv))
    ev = _event_array(stage_events)
    cev = _event_array(copy_events)
    if cev is not None and len(copy_events) != 2 * L:
        raise ValueError("copy_events needs two events per layer")
    a = FillArgs(L, d_in, d_out, n_kv, head_dim, 1 if host else 0, rows, pos0, cache_len,
                 rows_per_chunk, float(rope_theta), float(rms_eps), _ptr(H), _ptr(A),
                 _ptr(bias), _ptr(gain), _ptr(Wk), _ptr(Wv), _ptr(Kc), _ptr(Vc),
                 ctypes.cast(ev, ctypes.c_void_p) if ev is not None else None,
                 ctypes.cast(cev, ctypes.c_void_p) if cev is not None else None,
                 _ptr(k_scale), _ptr(v_scale), _ptr(A_scale), _ptr(row_idx), h_rows,
                 1 if h_host else 0, int(q8_group_layers))
    cb = None
    if map_source is not None:
        def _source(user, layer, dst, nbytes, _f=map_source):
            try:
                return int(_f(int(layer), int(dst), int(nbytes)))
            except Exception:  # an exception must not cross the C frame
                return -1
        cb = MAP_SOURCE_FN(_source)
        a.map_source = cb
        a.map_staging = _ptr(map_staging)
        a.host_wait_ms = int(host_wait_ms)
    a._events_keepalive = (ev, cev, cb)
    return a


RF_CALL_FILL, RF_CALL_FILL_GDN, RF_CALL_FIT, RF_CALL_RESCALE = 0, 1, 2, 3


def ridgefill_workspace_size(which: int, args) -> int:
    """Workspace bytes of call `which` (RF_CALL_*) for an argument struct; 0 if rejected."""
    return int(load().ridgefill_workspace_size(which, ctypes.cast(ctypes.byref(args), _vp)))


def fill_workspace_size(args: FillArgs) -> int:
    return int(load().ridgefill_fill_workspace_size(ctypes.byref(args)))


def gdn_workspace_size(args: GdnArgs) -> int:
    return int(load().ridgefill_gdn_workspace_size(ctypes.byref(args)))


def ridgefill_fill(H, A, bias, gain, Wk, Wv, Kc, Vc, *, head_dim: int, rope_theta: float,
                   rms_eps: float, pos0: int = 0, rows_per_chunk: int = 0,
                   workspace: Optional[torch.Tensor] = None, stream=None,
                   stage_events=None, copy_events=None, k_scale=None, v_scale=None,
                   A_scale=None, row_idx=None, q8_group_layers: int = 0, map_source=None,
                   map_staging=None, host_wait_ms: int = 0, map_shape=None) -> None:
    """Write the K/V cache of the prefix rows of every late attention layer.

    ``H`` [rows, d_in] bf16, ``A`` [L, d_out, d_in] bf16 (device, or pinned host
    memory to stream the maps), ``bias`` [L, d_out] f32, ``gain`` [L, d_out] bf16
    or None, ``Wk``/``Wv`` [L, n_kv*hd, d_out] bf16, ``Kc``/``Vc``
    [L, n_kv, cache_len, hd] bf16 (positions ``pos0 .. pos0+rows-1`` written).
    ``stage_events``: optional three ``torch.cuda.Event`` recorded around the
    first chunk's map GEMM and K/V GEMM.  ``k_scale``/``v_scale``: optional
    [L, n_kv] f32 per-head factors applied to the keys / values before rounding
    (the rescale of section 2.3 folded into the fill).  ``A_scale``: with int8
    maps ``A`` [L, d_out, d_in], their bf16 scales [L, d_in / 128, d_out]
    (section 2.2 "Size and cost"; see :func:`ridgefill_quantize_maps`).  ``row_idx``:
    optional int32 [rows] prefix rows to fill (section 2.4): ``H`` then holds every
    prefix row, row ``row_idx[r]`` is filled at position ``pos0 + row_idx[r]`` and the
    unlisted (exact) rows are left alone.  ``H`` may be a pinned host tensor: it is
    then copied by the library, overlapped with the map GEMM.  ``q8_group_layers``:
    resident int8 maps are dequantised 4 (or this many) layers at a time into the
    workspace ahead of the bf16 map GEMM; -1 converts them inside the GEMM instead
    (no extra workspace, slower; bitwise the same results).  ``map_source``: a callable
    ``(layer, dst_address, nbytes) -> int`` that writes one layer's map (in the layout of
    one layer of ``A``, int8 scales after the codes at a 256-byte boundary) into pinned
    staging memory and returns 0; the maps then stream from it through ``map_staging``
    (pinned, two layers' bytes) instead of from ``A``, which may be None with
    ``map_shape`` = (L, d_out, d_in).  Host waits of such a call are bounded by
    ``host_wait_ms`` (0: ten seconds); see the C header for what a timeout leaves behind.
    """
    args = fill_args(H, A, bias, gain, Wk, Wv, Kc, Vc, head_dim=head_dim, rope_theta=rope_theta,
                     rms_eps=rms_eps, pos0=pos0, rows_per_chunk=rows_per_chunk,
                     stage_events=stage_events, copy_events=copy_events, k_scale=k_scale,
                     v_scale=v_scale, A_scale=A_scale, row_idx=row_idx,
                     q8_group_layers=q8_group_layers, map_source=map_source,
                     map_staging=map_staging, host_wait_ms=host_wait_ms, map_shape=map_shape)
    lib = load()
    need = int(lib.ridgefill_fill_workspace_size(ctypes.byref(args)))
    if need == 0:
        _check(lib.ridgefill_fill(ctypes.byref(args), None, 0, _stream(stream)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Kc.device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    _check(lib.ridgefill_fill(ctypes.byref(args), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)))


def gdn_args(H, A, bias, gain, Wk, Wv, Wa, Wb, S, *, n_heads: int, rms_eps: float,
             l2_eps: float = 1e-6, S0=None, chunk: int = 64, rows_per_chunk: int = 0,
             stage_events=None, A_scale=None, exact_idx=None, X_exact=None, rho=None,
             delta_M=None, q8_group_layers: int = 0) -> GdnArgs:
    L, d_out, d_in = A.shape
    rows = H.shape[0]
    d_k = Wk.shape[1] // n_heads
    d_v = Wv.shape[1] // n_heads
    h_host = not H.is_cuda
    if h_host:
        if H.dtype != torch.bfloat16 or not H.is_contiguous() or not H.is_pinned():
            raise ValueError("host H must be contiguous, pinned bf16")
        if tuple(H.shape) != (rows, d_in):
            raise ValueError("H must be [rows, d_in]")
    else:
        _dev(H, "H", torch.bfloat16, (rows, d_in))
    host = _check_maps(A, A_scale)
    _dev(bias, "bias", torch.float32, (L, d_out))
    if gain is not None:
        _dev(gain, "gain", torch.bfloat16, (L, d_out))
    _dev(Wk, "Wk", torch.bfloat16, (L, n_heads * d_k, d_out))
    _dev(Wv, "Wv", torch.bfloat16, (L, n_heads * d_v, d_out))
    _dev(Wa, "Wa", torch.bfloat16, (L, n_heads, d_out))
    _dev(Wb, "Wb", torch.bfloat16, (L, n_heads, d_out))
    _dev(S, "S", torch.float32, (L, n_heads, d_v, d_k))
    if S0 is not None:
        _dev(S0, "S0", torch.float32, (L, n_heads, d_v, d_k))
    n_exact = 0
    if exact_idx is not None:
        n_exact = exact_idx.shape[0]
        _dev(exact_idx, "exact_idx", torch.int32, (n_exact,))
        _dev(X_exact, "X_exact", torch.bfloat16, (L, n_exact, d_out))
    if rho is not None:
        _dev(rho, "rho", torch.float32, (L, n_heads))
    if delta_M is not None:
        _dev(delta_M, "delta_M", torch.float32, (L, n_heads, d_v, d_k))
    ev = _event_array(stage_events)
    a = GdnArgs(L, d_in, d_out, n_heads, d_k, d_v, chunk, 1 if host else 0, rows,
                rows_per_chunk, float(rms_eps), float(l2_eps), _ptr(H), _ptr(A), _ptr(bias),
                _ptr(gain), _ptr(Wk), _ptr(Wv), _ptr(Wa), _ptr(Wb), _ptr(S0), _ptr(S),
                ctypes.cast(ev, ctypes.c_void_p) if ev is not None else None, _ptr(A_scale),
                _ptr(exact_idx), n_exact, _ptr(X_exact) if n_exact else None, _ptr(rho),
                _ptr(delta_M), 1 if h_host else 0, int(q8_group_layers))
    a._events_keepalive = ev
    return a


def ridgefill_fill_gdn(H, A, bias, gain, Wk, Wv, Wa, Wb, S, *, n_heads: int, rms_eps: float,
                       l2_eps: float = 1e-6, S0=None, chunk: int = 64, rows_per_chunk: int = 0,
                       workspace: Optional[torch.Tensor] = None, stream=None,
                       stage_events=None, A_scale=None, exact_idx=None, X_exact=None,
                       rho=None, delta_M=None, q8_group_layers: int = 0) -> None:
    """End-of-fill recurrent state ``S`` [L, H, dv, dk] f32 of Gated DeltaNet layers.

    ``stage_events``: optional four ``torch.cuda.Event`` recorded around the first
    chunk's map GEMM, projection GEMM and state kernel.  ``A_scale``: int8 maps, as
    for :func:`ridgefill_fill`.  ``exact_idx`` (int32 [n]) and ``X_exact`` ([L, n, d_out]
    bf16): exact prefix rows and their true inputs (section 2.4).  ``rho``: optional
    [L, H] f32 output of the filled rows' share of the state; ``delta_M``: optional
    [L, H, dv, dk] f32 terminal-state correction ``S += rho * delta_M`` (section 2.3).
    ``q8_group_layers``: as for :func:`ridgefill_fill`."""
    args = gdn_args(H, A, bias, gain, Wk, Wv, Wa, Wb, S, n_heads=n_heads, rms_eps=rms_eps,
                    l2_eps=l2_eps, S0=S0, chunk=chunk, rows_per_chunk=rows_per_chunk,
                    stage_events=stage_events, A_scale=A_scale, exact_idx=exact_idx,
                    X_exact=X_exact, rho=rho, delta_M=delta_M, q8_group_layers=q8_group_layers)
    lib = load()
    need = int(lib.ridgefill_gdn_workspace_size(ctypes.byref(args)))
    if need == 0:
        _check(lib.ridgefill_fill_gdn(ctypes.byref(args), None, 0, _stream(stream)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=S.device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    _check(lib.ridgefill_fill_gdn(ctypes.byref(args), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def rescale_args(H_tail, X_true, A, bias, gain, Wk, Wv, Kc, Vc, *, which: int, head_dim: int,
                 rms_eps: float, rows: int, pos0: int = 0, scale=None,
                 A_scale=None) -> RescaleArgs:
    L, d_out, d_in = A.shape
    if _check_maps(A, A_scale):
        raise ValueError("the rescale needs the maps in device memory")
    c = H_tail.shape[0]
    if X_true.shape != (L, c, d_out):
        raise ValueError("X_true must be [L, tail_rows, d_out]")
    n_kv = Kc.shape[1]
    a = RescaleArgs()
    a.n_layers, a.d_in, a.d_out, a.n_kv_heads, a.head_dim = L, d_in, d_out, n_kv, head_dim
    a.which, a.tail_rows, a.rows, a.pos0, a.cache_len = which, c, rows, pos0, Kc.shape[2]
    a.rms_eps = rms_eps
    a.H_tail, a.X_true, a.A, a.bias = _ptr(H_tail), _ptr(X_true), _ptr(A), _ptr(bias)
    a.gain = _ptr(gain) if gain is not None else None
    a.Wk, a.Wv, a.Kc, a.Vc = _ptr(Wk), _ptr(Wv), _ptr(Kc), _ptr(Vc)
    a.scale = _ptr(scale) if scale is not None else None
    a.A_scale = _ptr(A_scale)
    return a


def ridgefill_rescale(H_tail, X_true, A, bias, gain, Wk, Wv, Kc, Vc, *, which: int, head_dim: int,
                      rms_eps: float, rows: int, pos0: int = 0, scale=None,
                      workspace: Optional[torch.Tensor] = None, stream=None,
                      A_scale=None) -> None:
    """Value (or key) rescale of the filled cache rows [pos0, pos0 + rows), section 2.3.

    ``H_tail`` [c, d_in] bf16 and ``X_true`` [L, c, d_out] bf16 are the split states and
    the true late-layer inputs of the first c tail rows; ``scale`` an optional
    [L, n_kv] f32 output of the per-head scales.  Other arguments as for
    :func:`ridgefill_fill`."""
    args = rescale_args(H_tail, X_true, A, bias, gain, Wk, Wv, Kc, Vc, which=which,
                        head_dim=head_dim, rms_eps=rms_eps, rows=rows, pos0=pos0, scale=scale,
                        A_scale=A_scale)
    lib = load()
    need = int(lib.ridgefill_rescale_workspace_size(ctypes.byref(args)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=H_tail.device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    _check(lib.ridgefill_rescale(ctypes.byref(args), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def ridgefill_quantize_maps(A, q=None, scale=None, stream=None):
    """int8 codes and bf16 scales of maps ``A`` [L, d_out, d_in] (f32 or bf16, device):
    one scale per 128 weights of a row, section 2.2 ("Size and cost").  Returns
    ``(q, scale)``: [L, d_out, d_in] int8 and [L, d_in / 128, d_out] bf16 (the scale
    of weights 128g .. 128g + 127 of row j at [l, g, j])."""
    if A.dim() != 3:
        raise ValueError("A must be [L, d_out, d_in]")
    L, d_out, d_in = A.shape
    if A.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("A must be float32 or bfloat16")
    _dev(A, "A", A.dtype)
    if q is None:
        q = torch.empty((L, d_out, d_in), dtype=torch.int8, device=A.device)
    if scale is None:
        scale = torch.empty((L, d_in // Q8_GROUP, d_out), dtype=torch.bfloat16, device=A.device)
    _dev(q, "q", torch.int8, (L, d_out, d_in))
    _dev(scale, "scale", torch.bfloat16, (L, d_in // Q8_GROUP, d_out))
    args = QuantizeArgs(L, d_out, d_in, 1 if A.dtype == torch.bfloat16 else 0, _ptr(A), _ptr(q),
                        _ptr(scale))
    _check(load().ridgefill_quantize_maps(ctypes.byref(args), _stream(stream)))
    return q, scale


class FitSums:
    """Caller-owned f64 running sums of the ridge fit (device tensors)."""

    def __init__(self, n_layers: int, d_in: int, d_out: int, device="cuda"):
        f64 = torch.float64
        self.n_layers, self.d_in, self.d_out = n_layers, d_in, d_out
        self.G = torch.zeros((d_in, d_in), dtype=f64, device=device)
        self.C = torch.zeros((n_layers, d_out, d_in), dtype=f64, device=device)
        self.sx = torch.zeros((d_in,), dtype=f64, device=device)
        self.sy = torch.zeros((n_layers, d_out), dtype=f64, device=device)
        self.count = torch.zeros((1,), dtype=f64, device=device)


def _fit_call(sums: FitSums, flags: int, X=None, Y=None, lam: float = 0.0, A_out=None,
              A_out_f32=None, b_out=None, alpha_out=None, workspace=None, stream=None):
    L, d_in, d_out = sums.n_layers, sums.d_in, sums.d_out
    rows = 0
    if X is not None:
        rows = X.shape[0]
        _dev(X, "X", torch.bfloat16, (rows, d_in))
        _dev(Y, "Y", torch.bfloat16, (L, rows, d_out))
    if A_out is not None:
        _dev(A_out, "A_out", torch.bfloat16, (L, d_out, d_in))
    if A_out_f32 is not None:
        _dev(A_out_f32, "A_out_f32", torch.float32, (L, d_out, d_in))
    if b_out is not None:
        _dev(b_out, "b_out", torch.float32, (L, d_out))
    args = FitArgs(L, d_in, d_out, flags, rows, float(lam), _ptr(X), _ptr(Y), _ptr(sums.G),
                   _ptr(sums.C), _ptr(sums.sx), _ptr(sums.sy), _ptr(sums.count), _ptr(A_out),
                   _ptr(A_out_f32), _ptr(b_out), _ptr(alpha_out))
    lib = load()
    need = int(lib.ridgefill_fit_workspace_size(ctypes.byref(args)))
    if workspace is None:
        dev = sums.G.device
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    _check(lib.ridgefill_fit(ctypes.byref(args), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)))


def ridgefill_fit_accumulate(sums: FitSums, X, Y, *, workspace=None, stream=None) -> None:
    """Add calibration pairs ``X`` [n, d_in], ``Y`` [L, n, d_out] (bf16) to the sums."""
    _fit_call(sums, RF_FIT_ACCUMULATE, X=X, Y=Y, workspace=workspace, stream=stream)


def ridgefill_fit_solve(sums: FitSums, lam: float, *, A_out=None, A_out_f32=None, b_out=None,
                        alpha_out=None, workspace=None, stream=None) -> None:
    """Solve the ridge maps from the sums (``alpha = lam * tr(X~^T X~)/d_in``)."""
    _fit_call(sums, RF_FIT_SOLVE, lam=lam, A_out=A_out, A_out_f32=A_out_f32, b_out=b_out,
              alpha_out=alpha_out, workspace=workspace, stream=stream)


def device_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error word."""
    code = ctypes.c_int(0)
    load().ridgefill_device_error(_stream(stream), ctypes.byref(code))
    return int(code.value)


def wait_selftest(which: int, stream=None) -> None:
    """Enqueue a kernel whose bounded device wait runs out (0: mbarrier, 1: flag); read
    the outcome with :func:`device_error` (code 20 + which)."""
    _check(load().ridgefill_wait_selftest(int(which), _stream(stream)))


def compute_share(split: int, n_layers: int, tail: int, prompt: int) -> float:
    return float(load().ridgefill_compute_share(split, n_layers, tail, prompt))
