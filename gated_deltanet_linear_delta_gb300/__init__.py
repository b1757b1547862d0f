"""GB300 (sm_103a) gated delta rule layer: thin Python binding of the C ABI.

Every function here only marshals arguments (shapes, dtypes, device pointers,
the current CUDA stream) and calls the entry point of the same name in
``libgdn_gb300.so`` (declared in ``include/gdn.h``). All arithmetic runs in
the library's CUDA kernels. There is no CPU fallback: if the library is not
built, every call raises.

Tensors are torch CUDA tensors, contiguous, in the layouts of ``gdn.h``:
q, k [Ttot, Hk, dk]; v, out [Ttot, Hv, dv]; g, b [Ttot, Hv] (bf16 or fp32,
all the same dtype); states [B, Hv, dv, dk] fp32; cu_seqlens int32 [B+1].

The per-call host cost is kept small because a decode step of a few
sequences runs in a few microseconds on the GPU: the library handle and its
function objects are looked up once, pointers go to ctypes as plain integers,
and the current stream is read as a raw handle. Size and alignment checks are
the C library's (it returns an error before queueing anything).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = ["GDNError", "gdn_prefill", "gdn_prefill_ws", "gdn_prefill_workspace_size", "gdn_prefill_static",
           "gdn_prefill_from_host",
           "gdn_decode_step", "gdn_decode_step_slots", "gdn_prepass", "gdn_prefill_path",
           "gdn_get_device_status", "gdn_status_string", "library", "library_path",
           "GDN_OK", "GDN_ERR_INVALID_ARG", "GDN_ERR_UNSUPPORTED", "GDN_ERR_CUDA",
           "GDN_ERR_DEVICE_CHECK", "GDN_BF16", "GDN_F32"]

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEVICE_CHECK = 0, -1, -2, -3, -4
GDN_BF16, GDN_F32 = 0, 1

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_DTYPE = {torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}
# the current stream of a device as a raw cudaStream_t (falls back to the Stream object)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} returned {gdn_status_string(status)} ({status})")


def library_path() -> str:
    return _build.lib_path()


def library() -> ctypes.CDLL:
    """Load libgdn_gb300.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    lib = _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"the CUDA library {path} is not built; run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            lib.gdn_prefill.argtypes = [_P] * 9 + [_I] * 8 + [_P]
            lib.gdn_prefill.restype = _I
            lib.gdn_prefill_static.argtypes = [_P] * 9 + [_I] * 8 + [_P]
            lib.gdn_prefill_static.restype = _I
            lib.gdn_prefill_ws.argtypes = [_P] * 9 + [_I] * 8 + [_P, ctypes.c_size_t, _P]
            lib.gdn_prefill_ws.restype = _I
            lib.gdn_prefill_workspace_size.argtypes = [_I] * 8
            lib.gdn_prefill_workspace_size.restype = ctypes.c_size_t
            lib.gdn_decode_step.argtypes = [_P] * 7 + [_I] * 6 + [_P]
            lib.gdn_decode_step.restype = _I
            lib.gdn_prefill_from_host.argtypes = [_P] * 15 + [_I] * 8 + [_P]
            lib.gdn_prefill_from_host.restype = _I
            lib.gdn_decode_step_slots.argtypes = [_P] * 8 + [_I] * 7 + [_P]
            lib.gdn_decode_step_slots.restype = _I
            lib.gdn_prepass.argtypes = [_P] * 5 + [_I] * 7 + [_P] * 4 + [_P]
            lib.gdn_prepass.restype = _I
            lib.gdn_prefill_path.argtypes = [_I] * 8
            lib.gdn_prefill_path.restype = _I
            lib.gdn_get_device_status.argtypes = [_P]
            lib.gdn_get_device_status.restype = _I
            lib.gdn_status_string.argtypes = [_I]
            lib.gdn_status_string.restype = ctypes.c_char_p
            _lib = lib
        return _lib


def gdn_status_string(status: int) -> str:
    return library().gdn_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    code = _DTYPE.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")
    return code


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _stream(stream, t: torch.Tensor | None = None):
    """cudaStream_t of `stream`, or of the current stream of t's device (None: the current device)."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(t.get_device() if t is not None else torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str) -> None:
    if rc != GDN_OK:
        raise GDNError(rc, where)


def _prefill_sizes(q, v, g, b, out, state_in, state_out, cu_seqlens, B, T):
    Ttot, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
        B, T = cu_seqlens.numel() - 1, Ttot
    else:
        B = 1 if B is None else B
        T = Ttot // B if T is None else T
    for t in (v, g, b, out):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, g, b and out must share one dtype")
    for t in (state_in, state_out):
        if t is not None and t.dtype != torch.float32:
            raise TypeError("states are fp32")
    return B, T, Hk, Hv, dk, dv


def gdn_prefill(q, k, v, g, b, state_in, state_out, out, cu_seqlens=None, B=None, T=None, chunk=64,
                stream=None) -> None:
    """Chunked prefill over packed sequences; writes `out` and `state_out` (may alias state_in)."""
    lib = _lib or library()
    if k.dtype != q.dtype:
        raise TypeError("q, k, v, g, b and out must share one dtype")
    B, T, Hk, Hv, dk, dv = _prefill_sizes(q, v, g, b, out, state_in, state_out, cu_seqlens, B, T)
    rc = lib.gdn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(state_in), _ptr(state_out), _ptr(out),
                         _ptr(cu_seqlens), B, T, Hk, Hv, dk, dv, chunk, _dtype_code(q), _stream(stream, q))
    _check(rc, "gdn_prefill")


def gdn_prefill_static(q, k, v, g, b, state_in, state_out, out, cu_seqlens=None, B=None, T=None, chunk=64,
                       stream=None) -> None:
    """gdn_prefill that allocates nothing at call time: the tensor-core path's scratch is a fixed
    array in the library's device image, shared by all calls on a device (overlapping calls race)."""
    lib = _lib or library()
    if k.dtype != q.dtype:
        raise TypeError("q, k, v, g, b and out must share one dtype")
    B, T, Hk, Hv, dk, dv = _prefill_sizes(q, v, g, b, out, state_in, state_out, cu_seqlens, B, T)
    rc = lib.gdn_prefill_static(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(state_in), _ptr(state_out),
                                _ptr(out), _ptr(cu_seqlens), B, T, Hk, Hv, dk, dv, chunk, _dtype_code(q),
                                _stream(stream, q))
    _check(rc, "gdn_prefill_static")


def gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, dtype) -> int:
    """Bytes of device workspace gdn_prefill_ws needs for these sizes (0: none)."""
    if isinstance(dtype, torch.dtype):
        dtype = _DTYPE[dtype]
    return int(library().gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, int(dtype)))


def gdn_prefill_ws(q, k, v, g, b, state_in, state_out, out, workspace, cu_seqlens=None, B=None, T=None, chunk=64,
                   stream=None) -> None:
    """gdn_prefill with a caller-owned device workspace (a uint8 CUDA tensor, or None when none is needed)."""
    lib = _lib or library()
    if k.dtype != q.dtype:
        raise TypeError("q, k, v, g, b and out must share one dtype")
    B, T, Hk, Hv, dk, dv = _prefill_sizes(q, v, g, b, out, state_in, state_out, cu_seqlens, B, T)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.gdn_prefill_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(state_in), _ptr(state_out), _ptr(out),
                            _ptr(cu_seqlens), B, T, Hk, Hv, dk, dv, chunk, _dtype_code(q), _ptr(workspace), nbytes,
                            _stream(stream, q))
    _check(rc, "gdn_prefill_ws")


def _host_ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("host arrays must be contiguous CPU tensors")
    return t.data_ptr()


def gdn_prefill_from_host(q, k, v, g, b, state_in, state_out, out, dev, chunk=64, fragment=1024,
                          stream=None) -> None:
    """Prefill of one sequence from host tensors (pinned for overlap): q..b, state_in (or None),
    state_out and out are CPU tensors; `dev` holds the device buffers of the same shapes (keys
    q, k, v, g, b, out, state). Copies overlap the computation fragment by fragment."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    for t in (state_in, state_out):
        if t is not None and t.dtype != torch.float32:
            raise TypeError("states are fp32")
    rc = library().gdn_prefill_from_host(
        _host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(g), _host_ptr(b), _host_ptr(state_in),
        _host_ptr(state_out), _host_ptr(out), _ptr(dev["q"]), _ptr(dev["k"]), _ptr(dev["v"]), _ptr(dev["g"]),
        _ptr(dev["b"]), _ptr(dev["state"]), _ptr(dev["out"]), T, Hk, Hv, dk, dv, chunk, _dtype_code(q),
        fragment, _stream(stream, dev["q"]))
    _check(rc, "gdn_prefill_from_host")


def gdn_decode_step(q, k, v, g, b, state, out, stream=None) -> None:
    """One decode step for N sequences; updates `state` in place and writes `out`."""
    lib = _lib or library()
    N, Hk, dk = q.shape
    _, Hv, dv = v.shape
    if state.dtype != torch.float32:
        raise TypeError("the state is fp32")
    rc = lib.gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(state), _ptr(out),
                             N, Hk, Hv, dk, dv, _dtype_code(q), _stream(stream, q))
    if rc:
        raise GDNError(rc, "gdn_decode_step")


def gdn_decode_step_slots(q, k, v, g, b, state_pool, slots, out, stream=None) -> None:
    """One decode step; sequence n updates state_pool[slots[n]] in place (slots[n] < 0: padding)."""
    lib = _lib or library()
    N, Hk, dk = q.shape
    _, Hv, dv = v.shape
    if state_pool.dtype != torch.float32:
        raise TypeError("the state pool is fp32")
    if slots.dtype != torch.int32 or slots.numel() != N:
        raise TypeError("slots must be int32 with one entry per sequence")
    rc = lib.gdn_decode_step_slots(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(state_pool), _ptr(slots),
                                   _ptr(out), N, state_pool.shape[0], Hk, Hv, dk, dv, _dtype_code(q),
                                   _stream(stream, q))
    if rc:
        raise GDNError(rc, "gdn_decode_step_slots")


def gdn_prepass(q, k, g, b, rq, rk, beta, gcum, cu_seqlens=None, B=None, T=None, chunk=64,
                stream=None) -> None:
    """Per-token inverse norms, beta and in-block cumulative gate (fp32 outputs)."""
    Ttot, Hk, dk = q.shape
    Hv = g.shape[1]
    if cu_seqlens is not None:
        B, T = cu_seqlens.numel() - 1, Ttot
    else:
        B = 1 if B is None else B
        T = Ttot // B if T is None else T
    rc = library().gdn_prepass(_ptr(q), _ptr(k), _ptr(g), _ptr(b), _ptr(cu_seqlens), B, T, Hk, Hv, dk,
                               chunk, _dtype_code(q), _ptr(rq), _ptr(rk), _ptr(beta), _ptr(gcum),
                               _stream(stream, q))
    _check(rc, "gdn_prepass")


def gdn_prefill_path(B, T, Hk, Hv, dk, dv, chunk, dtype) -> int:
    """2 = token scan, 1 = tensor-core kernel, 0 = CUDA-core kernel, <0 = the status gdn_prefill would return."""
    if isinstance(dtype, torch.dtype):
        dtype = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    return library().gdn_prefill_path(B, T, Hk, Hv, dk, dv, chunk, int(dtype))


def gdn_get_device_status(stream=None) -> int:
    """Synchronise the stream, return and clear the device status word."""
    return library().gdn_get_device_status(_stream(stream))
