"""Decode step on the GPU against the fp64 oracle (one step = a scan of length 1)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import (DECODE_TOL, STATE_TOL, assert_outputs_close, decode_out_err, prefill_out_err, state_err,
                   threads)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_decode(q, k, v, g, b, state):
    qd, kd, vd, gd, bd = (x.to(DEV) for x in (q, k, v, g, b))
    sd = state.to(DEV).clone()
    out = torch.full(vd.shape, float("nan"), dtype=vd.dtype, device=DEV)  # poisoned
    gdn.gdn_decode_step(qd, kd, vd, gd, bd, sd, out)
    torch.cuda.synchronize()
    return out, sd


def check(out, st, q, k, v, g, b, state):
    ro, rs = oracle.gdn_decode_step(q, k, v, g, b, state, threads=threads())
    rel, _ = decode_out_err(out, ro)
    assert rel <= DECODE_TOL, rel
    # element-wise: the fp32 value within 1e-3 RMS of the oracle, then one rounding to the output dtype
    assert prefill_out_err(out, ro) <= DECODE_TOL
    assert state_err(st, rs) <= DECODE_TOL
    return ro, rs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128), (32, 128)])
@pytest.mark.parametrize("N", [1, 5])
def test_decode_shapes(dtype, dk, dv, N):
    q, k, v, g, b, state = inputs.make_decode_inputs(N, Hk=2, Hv=4, dk=dk, dv=dv, dtype=dtype, seed=N)
    q, k, v, g, b = q[0], k[0], v[0], g[0], b[0]
    out, st = run_decode(q, k, v, g, b, state)
    check(out, st, q, k, v, g, b, state)


@pytest.mark.parametrize("N", [1, 8, 32, 128])
def test_decode_qwen_shape(N):
    """Hk=16, Hv=32, dk=dv=128, bf16 I/O, fp32 state ~N(0, 0.02)."""
    q, k, v, g, b, state = inputs.make_decode_inputs(N, seed=0)
    q, k, v, g, b = q[0], k[0], v[0], g[0], b[0]
    out, st = run_decode(q, k, v, g, b, state)
    check(out, st, q, k, v, g, b, state)


def test_decode_128_steps_16_states():
    """128 consecutive steps on 16 sequences, state carried in place on the GPU."""
    steps, N = 128, 16
    q, k, v, g, b, state = inputs.make_decode_inputs(N, seed=3, steps=steps)
    sd = state.to(DEV).clone()
    ref_s = state.double().numpy()
    outs = []
    for t in range(steps):
        out = torch.empty(N, 32, 128, dtype=torch.bfloat16, device=DEV)
        gdn.gdn_decode_step(q[t].to(DEV), k[t].to(DEV), v[t].to(DEV), g[t].to(DEV), b[t].to(DEV), sd, out)
        outs.append(out)
    torch.cuda.synchronize()
    for t in range(steps):
        ro, ref_s = oracle.gdn_decode_step(q[t], k[t], v[t], g[t], b[t], ref_s, threads=threads())
        rel, _ = decode_out_err(outs[t], ro)
        assert rel <= DECODE_TOL, (t, rel)
    assert state_err(sd, ref_s) <= STATE_TOL


def test_decode_is_in_place_and_touches_only_its_state():
    q, k, v, g, b, state = inputs.make_decode_inputs(3, Hk=2, Hv=4, seed=9)
    q, k, v, g, b = (x[0].to(DEV) for x in (q, k, v, g, b))
    big = torch.randn(5, 4, 128, 128, device=DEV)
    before = big.clone()
    out = torch.empty(3, 4, 128, dtype=torch.bfloat16, device=DEV)
    gdn.gdn_decode_step(q, k, v, g, b, big[1:4], out)  # a view: rows 1..3 only
    torch.cuda.synchronize()
    assert torch.equal(big[0], before[0]) and torch.equal(big[4], before[4])
    assert not torch.equal(big[1:4], before[1:4])


def test_decode_matches_prefill_of_one_token():
    q, k, v, g, b, state = inputs.make_decode_inputs(4, Hk=2, Hv=4, seed=11)
    q, k, v, g, b = (x[0].to(DEV) for x in (q, k, v, g, b))
    sd = state.to(DEV)
    out_d = torch.empty(4, 4, 128, dtype=torch.bfloat16, device=DEV)
    st_d = sd.clone()
    gdn.gdn_decode_step(q, k, v, g, b, st_d, out_d)
    out_p = torch.empty_like(out_d)
    st_p = torch.empty_like(sd)
    gdn.gdn_prefill(q, k, v, g, b, sd, st_p, out_p, B=4, T=1, chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    # each route is within the oracle's bars, so they are within twice those of each other
    assert (st_d - st_p).norm() <= 2 * STATE_TOL * st_d.norm()
    assert_outputs_close(out_p, out_d, 2 * 2e-2)
