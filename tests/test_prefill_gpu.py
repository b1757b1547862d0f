"""Chunked prefill on the GPU against the fp64 oracle, through the C ABI.

Small cases compare every output; the long workloads compare full sequences
on a sample of heads (the oracle runs each (sequence, value head) on its own,
so a head subset is an exact sample). Output buffers are filled with NaN
before each call, so an element the kernel fails to write fails the test.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import (PREFILL_OUT_TOL, STATE_TOL, assert_outputs_close, oracle_prefill, prefill_out_err,
                   state_err)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_prefill(batch, state_in="batch", in_place=False):
    d = batch.to(DEV)
    si = d.state if state_in == "batch" else state_in
    out = torch.full(d.v.shape, float("nan"), dtype=d.v.dtype, device=DEV)
    if in_place and si is not None:
        so = si.clone()
        si = so
    else:
        so = torch.full((batch.B, batch.Hv, batch.dv, batch.dk), float("nan"), device=DEV)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, si, so, out, d.cu_seqlens,
                    B=None if d.cu_seqlens is not None else batch.B, chunk=batch.chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    return out, so


def check(batch, out, so, key_heads=None):
    ro, rs, vh = oracle_prefill(batch, key_heads)
    o = out if key_heads is None else out[:, vh]
    s = so if key_heads is None else so[:, vh]
    eo, es = prefill_out_err(o, ro), state_err(s, rs)
    assert eo <= PREFILL_OUT_TOL, f"output max-abs/RMS {eo:.3e}"
    assert es <= STATE_TOL, f"state rel-Frobenius {es:.3e}"
    return eo, es


def test_tiny_fp32():
    """B=1, T=64, Hk=Hv=2, dk=dv=32, fp32, chunk 16, zero state, seed 0."""
    b = inputs.tiny_fp32()
    out, so = run_prefill(b, state_in=None)
    check(b, out, so)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv,chunk", [(32, 32, 16), (64, 64, 32), (128, 64, 64), (64, 128, 16),
                                         (128, 128, 32), (32, 128, 64)])
def test_shapes_ragged(dtype, dk, dv, chunk):
    b = inputs.make_batch(B=2, T=100, Hk=2, Hv=4, dk=dk, dv=dv, dtype=dtype, chunk=chunk, seed=dk + dv,
                          init_state=True)
    out, so = run_prefill(b)
    check(b, out, so)


@pytest.mark.parametrize("hk,hv", [(3, 3), (2, 8), (1, 8), (5, 10), (40, 80)])
def test_head_groups_on_the_tensor_core_kernel(hk, hv):
    """Value heads per key head r = 1, 4, 8, 2 (odd key-head count) and more chains than state
    CTAs (80 heads x 3 sequences): the state CTAs are dealt in groups of r, several chains each."""
    b = inputs.make_batch(Hk=hk, Hv=hv, dk=128, dv=128, dtype="bf16", chunk=64, seed=hk * 100 + hv,
                          init_state=True, lengths=[190, 64, 333] if hv < 80 else [65, 1, 130])
    assert gdn.gdn_prefill_path(3, 600, hk, hv, 128, 128, 64, gdn.GDN_BF16) == 1
    out, so = run_prefill(b)
    check(b, out, so, key_heads=None if hk <= 5 else [0, 17, 39])


@pytest.mark.parametrize("lengths", [[0, 1, 63, 64, 65, 130, 7], [200], [1], [64, 64, 64]])
def test_varlen_edges_qwen_heads(lengths):
    """Packed sequences with empty, single-token and partial-last-block members."""
    b = inputs.make_batch(Hk=4, Hv=8, dk=128, dv=128, dtype="bf16", chunk=64, seed=5, init_state=True,
                          lengths=lengths)
    out, so = run_prefill(b)
    check(b, out, so)
    if 0 in lengths:  # a zero-length sequence carries its state through unchanged
        n = lengths.index(0)
        assert torch.equal(so[n].cpu(), b.state[n])


@pytest.mark.parametrize("split", ["1,0", "2,0", "4,0", "4,1"])
def test_cluster_splits(split, monkeypatch):
    """With few heads, a cluster of P CTAs per value head prepares the blocks (ranks F..P-1 in
    turn) for the CTA that carries the state: every split gives the oracle's result."""
    monkeypatch.setenv("GDN_PREFILL_KERNEL", "cluster")
    monkeypatch.setenv("GDN_PREFILL_CLUSTER", split)
    b = inputs.make_batch(Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=21, init_state=True,
                          slow_gate=True, lengths=[0, 1, 63, 64, 65, 130, 7, 700])
    out, so = run_prefill(b)
    check(b, out, so)


def test_null_state_in_means_zeros():
    b = inputs.make_batch(B=1, T=130, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=6)
    out0, so0 = run_prefill(b, state_in=None)
    zeros = torch.zeros(1, 4, 128, 128, device=DEV)
    out1, so1 = run_prefill(b, state_in=zeros)
    assert torch.equal(out0, out1) and torch.equal(so0, so1)
    check(b, out0, so0)


def test_in_place_state():
    b = inputs.make_batch(B=3, T=150, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=7,
                          init_state=True)
    out, so = run_prefill(b, in_place=True)
    check(b, out, so)


@pytest.mark.parametrize("dtype,dk,dv,chunk", [("f32", 64, 64, 32), ("bf16", 32, 128, 16)])
def test_in_place_state_cuda_core_kernel(dtype, dk, dv, chunk):
    """state_in == state_out on the CUDA-core block kernel (sizes the tensor-core kernels do not
    take): each row is read before it is overwritten, so the aliased call equals the oracle."""
    b = inputs.make_batch(B=3, T=130, Hk=2, Hv=4, dk=dk, dv=dv, dtype=dtype, chunk=chunk, seed=8,
                          init_state=True)
    assert gdn.gdn_prefill_path(b.B, b.T, b.Hk, b.Hv, dk, dv, chunk,
                                gdn.GDN_F32 if dtype == "f32" else gdn.GDN_BF16) == 0
    out, so = run_prefill(b, in_place=True)
    check(b, out, so)


def test_split_call_equals_one_call():
    """Carrying the state across two calls gives the one-call result (prompt fragments)."""
    b = inputs.make_batch(B=1, T=300, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=8,
                          init_state=True, slow_gate=True)
    out, so = run_prefill(b)
    d = b.to(DEV)
    cut = 170  # not a multiple of the block length
    mid = torch.empty_like(d.state)
    o1 = torch.empty(cut, 4, 128, dtype=torch.bfloat16, device=DEV)
    o2 = torch.empty(300 - cut, 4, 128, dtype=torch.bfloat16, device=DEV)
    s2 = torch.empty_like(d.state)
    gdn.gdn_prefill(d.q[:cut], d.k[:cut], d.v[:cut], d.g[:cut], d.b[:cut], d.state, mid, o1, B=1, chunk=64)
    gdn.gdn_prefill(d.q[cut:].contiguous(), d.k[cut:].contiguous(), d.v[cut:].contiguous(),
                    d.g[cut:].contiguous(), d.b[cut:].contiguous(), mid, s2, o2, B=1, chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    assert_outputs_close(torch.cat([o1, o2]), out, 1e-2)
    # each route is within the oracle's state bar, so they are within twice it of each other
    assert (s2 - so).norm() <= 2 * STATE_TOL * so.norm()
    check(b, torch.cat([o1, o2]), s2)


def test_prefill_equals_decode_steps():
    b = inputs.make_batch(B=2, T=40, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=12,
                          init_state=True, slow_gate=True)
    out, so = run_prefill(b)
    d = b.to(DEV)
    st = d.state.clone()
    q, k, v, g, bb = (x.view(2, 40, *x.shape[1:]) for x in (d.q, d.k, d.v, d.g, d.b))
    outs = []
    for t in range(40):
        o = torch.empty(2, 4, 128, dtype=torch.bfloat16, device=DEV)
        gdn.gdn_decode_step(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                            g[:, t].contiguous(), bb[:, t].contiguous(), st, o)
        outs.append(o)
    torch.cuda.synchronize()
    dec = torch.stack(outs, 1).reshape(80, 4, 128)
    assert_outputs_close(dec, out, 2e-2)
    assert (st - so).norm() <= 1e-3 * so.norm()


def test_prefill_4k_all_heads():
    """One sequence of 4096 tokens, Hk=16, Hv=32, dk=dv=128, bf16, chunk 64, zero state."""
    b = inputs.prefill_4k()
    out, so = run_prefill(b, state_in=None)
    check(b, out, so)


def test_prefill_4k_slow_gate():
    """Slow gates keep the state alive across all 64 blocks, so carry errors would show."""
    b = inputs.make_batch(B=1, T=4096, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=1,
                          init_state=True, slow_gate=True)
    out, so = run_prefill(b)
    check(b, out, so, key_heads=[0, 7, 15])


@pytest.mark.parametrize("T,key_heads", [(32768, [3, 12]), (131072, [9])])
def test_prefill_long_sampled_heads(T, key_heads):
    b = inputs.prefill_long(T=T)
    out, so = run_prefill(b)
    check(b, out, so, key_heads=key_heads)


def test_prefill_varlen_16_sampled_heads():
    """16 packed sequences, lengths uniform in [256, 16384], each with its own state."""
    b = inputs.prefill_varlen()
    out, so = run_prefill(b)
    check(b, out, so, key_heads=[5])


def test_inconsistent_cu_seqlens_is_reported():
    b = inputs.make_batch(Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=13, lengths=[50, 30])
    d = b.to(DEV)
    bad = torch.tensor([0, 60, 40], dtype=torch.int32, device=DEV)  # decreasing
    out = torch.zeros(80, 4, 128, dtype=torch.bfloat16, device=DEV)
    so = torch.zeros(2, 4, 128, 128, device=DEV)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, None, so, out, bad, chunk=64)
    assert gdn.gdn_get_device_status() == gdn.GDN_ERR_DEVICE_CHECK
    assert gdn.gdn_get_device_status() == gdn.GDN_OK  # reading clears it
