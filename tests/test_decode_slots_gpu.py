"""Decode over a pool of resident states (slot-indexed), on the GPU, against the fp64 oracle.

Sequence n of a step updates pool entry slots[n]; the oracle runs the plain decode step on the
gathered states, and every entry that no sequence names must come back bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import DECODE_TOL, STATE_TOL, decode_out_err, prefill_out_err, state_err, threads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pool_case(N, num_slots, Hk, Hv, dk, dv, dtype, seed, n_pad):
    q, k, v, g, b, _ = inputs.make_decode_inputs(N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype=dtype, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1000)
    pool = torch.randn(num_slots, Hv, dv, dk, generator=gen) * 0.02
    slots = torch.randperm(num_slots, generator=gen)[:N].to(torch.int32)
    if n_pad:
        slots[torch.randperm(N, generator=gen)[:n_pad]] = -1
    return q[0], k[0], v[0], g[0], b[0], pool, slots


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,num_slots,n_pad", [(1, 1, 0), (5, 12, 2), (32, 96, 3), (128, 128, 0)])
def test_decode_slots_parity(dtype, N, num_slots, n_pad):
    Hk, Hv = (16, 32) if N >= 32 else (2, 4)
    q, k, v, g, b, pool, slots = _pool_case(N, num_slots, Hk, Hv, 128, 128, dtype, seed=N, n_pad=n_pad)
    pd = pool.to(DEV)
    out = torch.full(v.shape, float("nan"), dtype=v.dtype, device=DEV)  # poisoned
    gdn.gdn_decode_step_slots(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), b.to(DEV), pd, slots.to(DEV), out)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    live = [n for n in range(N) if slots[n] >= 0]
    idx = slots[live].long()
    ro, rs = oracle.gdn_decode_step(q[live], k[live], v[live], g[live], b[live], pool[idx], threads=threads())
    rel, _ = decode_out_err(out[live], ro)
    assert rel <= DECODE_TOL, rel
    assert prefill_out_err(out[live], ro) <= DECODE_TOL
    assert state_err(pd[idx], rs) <= STATE_TOL
    pad = [n for n in range(N) if slots[n] < 0]
    if pad:
        assert torch.count_nonzero(out[pad]).item() == 0
    untouched = sorted(set(range(num_slots)) - set(idx.tolist()))
    if untouched:
        assert torch.equal(pd[untouched].cpu(), pool[untouched])


def test_decode_slots_identity_equals_decode_step():
    """slots = 0..N-1 is the plain decode step, bit for bit (the same arithmetic per row)."""
    q, k, v, g, b, state = inputs.make_decode_inputs(8, seed=5)
    q, k, v, g, b = (x[0].to(DEV) for x in (q, k, v, g, b))
    s1, s2 = state.to(DEV), state.to(DEV).clone()
    o1 = torch.empty(8, 32, 128, dtype=torch.bfloat16, device=DEV)
    o2 = torch.empty_like(o1)
    gdn.gdn_decode_step(q, k, v, g, b, s1, o1)
    gdn.gdn_decode_step_slots(q, k, v, g, b, s2, torch.arange(8, dtype=torch.int32, device=DEV), o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_decode_slots_steps_carry_state_per_session():
    """Several steps over a changing subset of sessions: each session's state follows its own
    token stream, as if each had been decoded alone."""
    Hk, Hv, num_slots, steps = 2, 4, 6, 5
    gen = torch.Generator().manual_seed(17)
    pool0 = torch.randn(num_slots, Hv, 128, 128, generator=gen) * 0.02
    pd = pool0.to(DEV)
    ref = pool0.double().numpy().copy()
    for t in range(steps):
        sel = torch.randperm(num_slots, generator=gen)[:4].to(torch.int32)
        q, k, v, g, b, _ = inputs.make_decode_inputs(4, Hk=Hk, Hv=Hv, seed=100 + t)
        q, k, v, g, b = q[0], k[0], v[0], g[0], b[0]
        out = torch.empty(4, Hv, 128, dtype=torch.bfloat16, device=DEV)
        gdn.gdn_decode_step_slots(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), b.to(DEV), pd, sel.to(DEV), out)
        ro, rs = oracle.gdn_decode_step(q, k, v, g, b, ref[sel.long().numpy()], threads=threads())
        ref[sel.long().numpy()] = rs
        rel, _ = decode_out_err(out, ro)
        assert rel <= DECODE_TOL, (t, rel)
    torch.cuda.synchronize()
    assert state_err(pd, ref) <= STATE_TOL


def test_decode_slots_out_of_range_is_flagged_and_skipped():
    q, k, v, g, b, pool, slots = _pool_case(3, 4, 2, 4, 128, 128, "bf16", seed=21, n_pad=0)
    slots[1] = 4  # one past the pool
    pd = pool.to(DEV)
    out = torch.full(v.shape, float("nan"), dtype=v.dtype, device=DEV)
    gdn.gdn_decode_step_slots(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), b.to(DEV), pd, slots.to(DEV), out)
    assert gdn.gdn_get_device_status() == gdn.GDN_ERR_DEVICE_CHECK
    assert gdn.gdn_get_device_status() == gdn.GDN_OK  # read and cleared
    assert torch.count_nonzero(out[1]).item() == 0
    named = {int(slots[0]), int(slots[2])}
    for e in range(4):
        if e not in named:
            assert torch.equal(pd[e].cpu(), pool[e])
    assert not torch.isnan(out[[0, 2]].float()).any()
