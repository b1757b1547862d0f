"""Few-token prefill (at most 8 tokens per sequence, no cu_seqlens): gdn_prefill evaluates it as a
token scan, one pass over each state. Parity against the fp64 oracle with the decode bars (the
arithmetic is the decode step's, applied T times in fp32), and agreement with T decode steps and
with the block kernels (forced by passing cu_seqlens)."""
import pytest
import torch

import oracle
from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import (DECODE_TOL, STATE_TOL, assert_outputs_close, decode_out_err, prefill_out_err, state_err,
                   threads)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(batch, state_in, in_place=False, cu=None):
    d = batch.to(DEV)
    out = torch.full(d.v.shape, float("nan"), dtype=d.v.dtype, device=DEV)
    sin = None if state_in is None else state_in.to(DEV)
    sout = sin if in_place else torch.full((batch.B, batch.Hv, batch.dv, batch.dk), float("nan"), device=DEV)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, sin, sout, out, cu, B=batch.B, T=None if cu is not None else batch.T,
                    chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    return out, sout


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,Hk,Hv,dk,dv", [(3, 2, 4, 128, 128), (2, 1, 2, 32, 64), (1, 2, 2, 64, 32)])
def test_scan_parity(T, dtype, B, Hk, Hv, dk, dv):
    assert gdn.gdn_prefill_path(B, T, Hk, Hv, dk, dv, 64, gdn.GDN_BF16 if dtype == "bf16" else gdn.GDN_F32) == 2
    b = inputs.make_batch(B=B, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype=dtype, chunk=64, seed=40 + T,
                          init_state=True)
    out, st = _run(b, b.state)
    ro, rs = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, b.state, None, B=B, threads=threads())
    assert prefill_out_err(out, ro) <= DECODE_TOL
    assert decode_out_err(out, ro)[0] <= DECODE_TOL
    assert state_err(st, rs) <= STATE_TOL


@pytest.mark.parametrize("in_place,zero_state", [(True, False), (False, True)])
def test_scan_in_place_and_zero_state(in_place, zero_state):
    b = inputs.make_batch(B=4, T=4, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=51,
                          init_state=not zero_state)
    out, st = _run(b, b.state, in_place=in_place)
    ro, rs = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, b.state, None, B=4, threads=threads())
    assert prefill_out_err(out, ro) <= DECODE_TOL
    assert state_err(st, rs) <= STATE_TOL


def test_scan_qwen_shape_128_sequences_4_tokens():
    """The speculative-verify shape: 128 sequences x 4 tokens, Hk=16, Hv=32, dk=dv=128."""
    b = inputs.make_batch(B=128, T=4, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=52,
                          init_state=True)
    out, st = _run(b, b.state, in_place=True)
    for kh in (0, 7, 15):  # oracle on a few key heads (and the value heads that share them)
        vh = [2 * kh, 2 * kh + 1]
        ro, rs = oracle.gdn_sequential(b.q[:, [kh]], b.k[:, [kh]], b.v[:, vh], b.g[:, vh], b.b[:, vh],
                                       b.state[:, vh], None, B=128, threads=threads())
        assert prefill_out_err(out[:, vh], ro) <= DECODE_TOL
        assert state_err(st[:, vh], rs) <= STATE_TOL


def test_scan_equals_decode_steps_and_block_kernels():
    T, B = 6, 5
    b = inputs.make_batch(B=B, T=T, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=53, init_state=True)
    out_s, st_s = _run(b, b.state)
    # T decode steps on the GPU
    d = b.to(DEV)
    st_d = d.state.clone()
    out_d = torch.empty_like(out_s)
    for t in range(T):
        rows = torch.arange(B, device=DEV) * T + t
        o = torch.empty(B, 4, 128, dtype=torch.bfloat16, device=DEV)
        gdn.gdn_decode_step(d.q[rows].contiguous(), d.k[rows].contiguous(), d.v[rows].contiguous(),
                            d.g[rows].contiguous(), d.b[rows].contiguous(), st_d, o)
        out_d[rows] = o
    # the block kernels, forced by packing the same sequences with cu_seqlens
    cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device=DEV)
    out_b, st_b = _run(b, b.state, cu=cu)
    torch.cuda.synchronize()
    for other_out, other_st in ((out_d, st_d), (out_b, st_b)):
        assert (st_s - other_st).norm() <= 2 * STATE_TOL * st_s.norm()
        assert_outputs_close(out_s, other_out, 2 * 2e-2)
