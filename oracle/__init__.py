"""fp64 CPU oracle for the gated delta rule.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The CUDA library under
``gated_deltanet_linear_delta_gb300`` never imports it and shares no code with
it; the only thing both sides use is the seeded input generator module, which
holds no arithmetic of the method.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, no fast-math, no FMA
contraction); this module compiles it with gcc on first use and marshals numpy
arrays. See the header of ``gdn_oracle.c`` for the recurrence and the pages it
follows ("Optimiser l'inference sur appareil pour Apple Silicon", sections
"Qwen cree trois formes de charges de travail" and "Maintenir l'etat recurrent
sur la puce").

Every input is upcast exactly to float64 (bf16 and fp32 values are exactly
representable), so the oracle sees precisely the values the GPU sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}

_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)


def lib_path(mutation: int = 0) -> str:
    name = "libgdn_oracle.so" if mutation == 0 else f"libgdn_oracle_mut{mutation}.so"
    return os.path.join(_BUILD, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile gdn_oracle.c (optionally with a planted mistake) and return the .so path."""
    out = lib_path(mutation)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           f"-DORACLE_MUTATION={mutation}", _SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutation: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutation not in _libs:
            lib = ctypes.CDLL(build(mutation))
            common = [_D, _D, _D, _D, _D, _D, _D, _D, _I32] + [ctypes.c_int] * 6
            lib.oracle_gdn_sequential.argtypes = common + [ctypes.c_int]
            lib.oracle_gdn_sequential.restype = ctypes.c_int
            lib.oracle_gdn_chunked.argtypes = common + [ctypes.c_int, ctypes.c_int]
            lib.oracle_gdn_chunked.restype = ctypes.c_int
            lib.oracle_gdn_prepass.argtypes = [_D, _D, _D, _D, _I32] + [ctypes.c_int] * 6 + [_D] * 4
            lib.oracle_gdn_prepass.restype = ctypes.c_int
            _libs[mutation] = lib
        return _libs[mutation]


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact upcast on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_D)


def _seqlens(cu_seqlens):
    if cu_seqlens is None:
        return None, None
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return cu, cu.ctypes.data_as(_I32)


def _shapes(q, v, B, T, cu):
    Ttot, Hk, dk = q.shape
    _, Hv, dv = v.shape
    if cu is not None:
        B = len(cu) - 1
        if int(cu[-1]) != Ttot or int(cu[0]) != 0 or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must start at 0, be non-decreasing and end at the token count")
        T = Ttot
    else:
        if B is None:
            B = 1
        if Ttot % B:
            raise ValueError("token count is not a multiple of B")
        T = Ttot // B
    return B, T, Ttot, Hk, Hv, dk, dv


def gdn_sequential(q, k, v, g, beta, state_in=None, cu_seqlens=None, B=None, threads=1, mutation=0):
    """Token-by-token scan (the definition). Returns (out [Ttot,Hv,dv], state_out [B,Hv,dv,dk])."""
    q, k, v, g, beta, state_in = (_f64(x) for x in (q, k, v, g, beta, state_in))
    cu, cup = _seqlens(cu_seqlens)
    B, T, Ttot, Hk, Hv, dk, dv = _shapes(q, v, B, T=None, cu=cu)
    out = np.zeros((Ttot, Hv, dv))
    state_out = np.zeros((B, Hv, dv, dk))
    rc = _lib(mutation).oracle_gdn_sequential(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(state_out), _ptr(out),
        cup, B, T, Hk, Hv, dk, dv, int(threads))
    if rc != 0:
        raise ValueError("oracle_gdn_sequential rejected its arguments")
    return out, state_out


def gdn_chunked(q, k, v, g, beta, state_in=None, cu_seqlens=None, B=None, chunk=64, threads=1, mutation=0):
    """Block (WY/UT) evaluation with chunk size `chunk`; same outputs as gdn_sequential."""
    q, k, v, g, beta, state_in = (_f64(x) for x in (q, k, v, g, beta, state_in))
    cu, cup = _seqlens(cu_seqlens)
    B, T, Ttot, Hk, Hv, dk, dv = _shapes(q, v, B, T=None, cu=cu)
    out = np.zeros((Ttot, Hv, dv))
    state_out = np.zeros((B, Hv, dv, dk))
    rc = _lib(mutation).oracle_gdn_chunked(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(state_out), _ptr(out),
        cup, B, T, Hk, Hv, dk, dv, int(chunk), int(threads))
    if rc != 0:
        raise ValueError("oracle_gdn_chunked rejected its arguments")
    return out, state_out


def gdn_prepass(q, k, g, beta, cu_seqlens=None, B=None, chunk=64):
    """Per-token rq, rk [Ttot,Hk], beta, gcum [Ttot,Hv] of the block form."""
    q, k, g, beta = (_f64(x) for x in (q, k, g, beta))
    cu, cup = _seqlens(cu_seqlens)
    Ttot, Hk, dk = q.shape
    Hv = g.shape[1]
    if cu is not None:
        B, T = len(cu) - 1, Ttot
    else:
        B = 1 if B is None else B
        T = Ttot // B
    rq = np.zeros((Ttot, Hk))
    rk = np.zeros((Ttot, Hk))
    bo = np.zeros((Ttot, Hv))
    gc = np.zeros((Ttot, Hv))
    rc = _lib().oracle_gdn_prepass(_ptr(q), _ptr(k), _ptr(g), _ptr(beta), cup, B, T, Hk, Hv, dk,
                                   int(chunk), _ptr(rq), _ptr(rk), _ptr(bo), _ptr(gc))
    if rc != 0:
        raise ValueError("oracle_gdn_prepass rejected its arguments")
    return rq, rk, bo, gc


def gdn_decode_step(q, k, v, g, beta, state, threads=1):
    """One recurrent step for N independent sequences: a scan of length 1 each.

    q, k [N,Hk,dk]; v [N,Hv,dv]; g, beta [N,Hv]; state [N,Hv,dv,dk].
    Returns (out [N,Hv,dv], new_state [N,Hv,dv,dk]).
    """
    q = _f64(q)
    N = q.shape[0]
    return gdn_sequential(q, k, v, g, beta, state_in=state, B=N, threads=threads)


def cpu_threads() -> int:
    return os.cpu_count() or 1
