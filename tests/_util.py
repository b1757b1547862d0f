"""Shared helpers of the test-suite: oracle calls on head subsets, parity metrics.

Tolerances (written here, used by every parity test):

* prefill output: max |gpu - oracle| <= 2e-2 * RMS(oracle output), applied to
  the layer's computed value. The output is that value rounded once to the I/O
  dtype, which moves it by at most u*|value| (u = 2^-8 for bf16, 2^-24 for
  fp32), so the observable check is, element-wise,
      |out - ref| <= 2e-2 * RMS(ref) * (1 + u) + u * |ref|.
  (The exact fp64 result rounded to bf16 alone is already ~3e-2 * RMS away from
  it on these workloads: outputs are heavy-tailed, max|ref| ~ 12-16 RMS.)
* final state (prefill and decode): ||gpu - oracle||_F <= 1e-3 * ||oracle||_F;
* decode output: the layer's output is the fp32 result rounded once to the
  I/O dtype, so the oracle's fp64 output is rounded the same way (RNE) before
  comparing; then ||gpu - ref|| <= 1e-3 * ||ref||; element-wise, the same
  rounding-aware bound as prefill with 1e-3 in place of 2e-2.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

PREFILL_OUT_TOL = 2e-2   # x RMS of the oracle output, max-abs
STATE_TOL = 1e-3         # relative Frobenius
DECODE_TOL = 1e-3        # relative (2-norm)


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def head_subset(batch, key_heads):
    """Inputs restricted to the given key heads and the value heads that share them."""
    grp = batch.Hv // batch.Hk
    vh = [h for kh in key_heads for h in range(kh * grp, (kh + 1) * grp)]
    sl = lambda x, idx: None if x is None else x[:, idx]  # noqa: E731
    st = None if batch.state is None else batch.state[:, vh]
    return (sl(batch.q, key_heads), sl(batch.k, key_heads), sl(batch.v, vh), sl(batch.g, vh),
            sl(batch.b, vh), st), vh


def oracle_prefill(batch, key_heads=None, state=None):
    """fp64 oracle (token scan) on all heads or on a subset of key heads."""
    if key_heads is None:
        q, k, v, g, b, st = batch.q, batch.k, batch.v, batch.g, batch.b, batch.state
        vh = list(range(batch.Hv))
    else:
        (q, k, v, g, b, st), vh = head_subset(batch, key_heads)
    if state is not None:
        st = state if key_heads is None else state[:, vh]
    cu = batch.cu_seqlens
    out, s = oracle.gdn_sequential(q, k, v, g, b, st, cu, B=None if cu is not None else batch.B,
                                   threads=threads())
    return out, s, vh


def rms(x) -> float:
    return float(np.sqrt(np.mean(np.square(x)))) if np.size(x) else 0.0


UNIT_ROUNDOFF = {torch.bfloat16: 2.0 ** -8, torch.float32: 2.0 ** -24}


def prefill_out_err(gpu_out, ref) -> float:
    """max over elements of (|gpu - ref| - u|ref|) / (RMS(ref) (1 + u)): the computation's error
    in units of the output RMS, once the single rounding to the output dtype is allowed for."""
    if not ref.size:
        return 0.0
    u = UNIT_ROUNDOFF[gpu_out.dtype]
    g = gpu_out.detach().float().cpu().double().numpy()
    return float(np.max(np.abs(g - ref) - u * np.abs(ref)) / (max(rms(ref), 1e-30) * (1 + u)))


def prefill_out_raw_err(gpu_out, ref) -> float:
    """max |gpu - ref| / RMS(ref), rounding of the output included (reported, not asserted)."""
    g = gpu_out.detach().float().cpu().double().numpy()
    return float(np.max(np.abs(g - ref)) / max(rms(ref), 1e-30)) if ref.size else 0.0


def state_err(gpu_state, ref) -> float:
    g = gpu_state.detach().cpu().double().numpy()
    return float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))


def round_like(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Round fp64 values once (RNE) to `dtype` and back."""
    return torch.from_numpy(ref).to(dtype).double().numpy()


def decode_out_err(gpu_out, ref) -> tuple[float, float]:
    """(relative 2-norm error, max error in units of the I/O dtype's last place)."""
    dt = gpu_out.dtype
    r = round_like(ref, dt)
    g = gpu_out.detach().cpu().double().numpy()
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    mant = {torch.bfloat16: 7, torch.float32: 23}[dt]  # explicit mantissa bits
    _, ex = np.frexp(np.maximum(np.abs(r), np.finfo(np.float32).tiny))  # |r| = m 2^ex, m in [0.5, 1)
    ulp = np.ldexp(1.0, ex - 1 - mant)  # spacing of the format in [2^(ex-1), 2^ex)
    return rel, float(np.max(np.abs(g - r) / ulp)) if r.size else 0.0


def assert_outputs_close(a, b, tol):
    """Two outputs of the layer computed by different routes, each rounded once to its dtype:
    |a - b| <= tol * RMS(b) + 2u * max(|a|, |b|) element-wise."""
    u = UNIT_ROUNDOFF[a.dtype]
    x, y = a.detach().float(), b.detach().float()
    bound = tol * y.pow(2).mean().sqrt() + 2 * u * torch.maximum(x.abs(), y.abs())
    excess = ((x - y).abs() - bound).max().item()
    assert excess <= 0, f"outputs differ beyond the bound by {excess:.3e}"
