"""Prefill on inputs far from unit scale, through the C ABI, against the fp64 oracle.

The tensor-core kernels carry some operands in fp16 with power-of-two scales chosen at run time:
K (and, with key sharing, Q) as sigma K with sigma set by the tile's largest magnitude, and the
state's fp16 copy with one scale per row. Keys and queries scaled by 300 or 1e-3 move sigma far
from its unit-scale value (the layer normalises q and k, so the outputs barely change); values
and initial states scaled by 1e4 or 1e-4 put the state beyond fp16's range or into its
subnormals, where only the row scales keep it exact to fp16 precision. The parity bars are
relative (output max-abs / RMS, state relative Frobenius), so they hold at every scale.

The last cases draw nearly identical keys with beta close to 1, where A = beta e^{G_t-G_s} kh_t.kh_s
is close to a strictly lower matrix of ones, the triangular solve (I + A)^-1 does the most work and
W = T diag(beta e) Kh cancels to a small fraction of its terms. They run on the ring kernel (the
default tensor-core path), which carries T diag(beta e) as fp16 hi + lo for this reason.
"""
import dataclasses

import pytest
import torch

from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import PREFILL_OUT_TOL, STATE_TOL, oracle_prefill, prefill_out_err, state_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SCALES = [(300.0, 1.0), (1e-3, 1.0), (1.0, 1e4), (1.0, 1e-4)]  # (q and k, v and state)


def scaled(batch, qk, vs):
    """The batch with q, k times qk and v, the initial state times vs (rounded to the I/O type)."""
    def mul(x, s):
        return x if s == 1.0 else (x.float() * s).to(x.dtype)
    return dataclasses.replace(batch, q=mul(batch.q, qk), k=mul(batch.k, qk), v=mul(batch.v, vs),
                               state=None if batch.state is None else batch.state * vs)


def run_and_check(batch, key_heads=None):
    d = batch.to(DEV)
    out = torch.full(d.v.shape, float("nan"), dtype=d.v.dtype, device=DEV)
    so = torch.full((batch.B, batch.Hv, batch.dv, batch.dk), float("nan"), device=DEV)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state, so, out, d.cu_seqlens,
                    B=None if d.cu_seqlens is not None else batch.B, chunk=batch.chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    ro, rs, vh = oracle_prefill(batch, key_heads)
    o = out if key_heads is None else out[:, vh]
    s = so if key_heads is None else so[:, vh]
    assert torch.isfinite(o).all() and torch.isfinite(s).all()
    eo, es = prefill_out_err(o, ro), state_err(s, rs)
    assert eo <= PREFILL_OUT_TOL, f"output max-abs/RMS {eo:.3e}"
    assert es <= STATE_TOL, f"state rel-Frobenius {es:.3e}"


@pytest.mark.parametrize("qk,vs", SCALES)
def test_ring_kernel_one_sequence(qk, vs):
    b = inputs.make_batch(B=1, T=300, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=71,
                          init_state=True, slow_gate=True)
    run_and_check(scaled(b, qk, vs))


@pytest.mark.parametrize("qk,vs", SCALES)
def test_ring_kernel_key_sharing(qk, vs):
    """More chains than state CTAs: Q is scaled to fp16 as well, with its own sigma."""
    b = inputs.make_batch(Hk=20, Hv=40, dk=128, dv=128, dtype="bf16", chunk=64, seed=72, init_state=True,
                          lengths=[190, 64, 333])
    run_and_check(scaled(b, qk, vs), key_heads=[0, 11])


@pytest.mark.parametrize("qk,vs", SCALES)
def test_cluster_kernel(qk, vs, monkeypatch):
    monkeypatch.setenv("GDN_PREFILL_KERNEL", "cluster")
    b = inputs.make_batch(Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=73, init_state=True,
                          slow_gate=True, lengths=[65, 300])
    run_and_check(scaled(b, qk, vs))


def correlated_keys(batch, spread=0.05, beta_logit=4.0):
    """Every key of a key head is that head's first key plus spread x N(0, 1) noise; beta logits
    raised by beta_logit (beta near 1). Seeded from the batch's own seed."""
    gen = torch.Generator().manual_seed(int(batch.meta["seed"]) + 500)
    k = batch.k.float()
    k = k[:1].expand_as(k) + spread * torch.randn(k.shape, generator=gen)
    return dataclasses.replace(batch, k=k.to(batch.k.dtype), b=(batch.b.float() + beta_logit).to(batch.b.dtype))


def test_correlated_keys_ring_kernel():
    b = inputs.make_batch(B=1, T=700, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=74,
                          init_state=True, slow_gate=True)
    run_and_check(correlated_keys(b))


def test_correlated_keys_ring_kernel_key_sharing():
    b = inputs.make_batch(Hk=20, Hv=40, dk=128, dv=128, dtype="bf16", chunk=64, seed=75, init_state=True,
                          lengths=[190, 64, 333])
    run_and_check(correlated_keys(b), key_heads=[0, 11])
