"""Prefill from host memory with the copies overlapped fragment by fragment: bit-identical to
gdn_prefill on device buffers (fragments are whole blocks, the state is carried in fp32), and
within the oracle's bars."""
import pytest
import torch

import oracle
from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import PREFILL_OUT_TOL, STATE_TOL, prefill_out_err, state_err, threads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _host_run(b, fragment, init_state):
    host = {n: getattr(b, n).pin_memory() for n in ("q", "k", "v", "g", "b")}
    sin = b.state[0].pin_memory() if init_state else None
    sout = torch.empty(b.Hv, b.dv, b.dk).pin_memory()
    out = torch.empty(b.v.shape, dtype=b.v.dtype).pin_memory()
    dev = {n: torch.empty_like(t, device=DEV) for n, t in host.items()}
    dev["out"] = torch.empty(b.v.shape, dtype=b.v.dtype, device=DEV)
    dev["state"] = torch.empty(b.Hv, b.dv, b.dk, device=DEV)
    gdn.gdn_prefill_from_host(host["q"], host["k"], host["v"], host["g"], host["b"], sin, sout, out, dev,
                              chunk=64, fragment=fragment)
    torch.cuda.current_stream().synchronize()
    return out, sout


def _device_run(b, init_state):
    d = b.to(DEV)
    out = torch.empty(d.v.shape, dtype=d.v.dtype, device=DEV)
    so = torch.empty(1, b.Hv, b.dv, b.dk, device=DEV)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state if init_state else None, so, out, None, B=1, chunk=64)
    torch.cuda.synchronize()
    return out.cpu(), so[0].cpu()


@pytest.mark.parametrize("T,fragment,init_state", [(1000, 256, True), (4096, 1024, False), (640, 640, True)])
def test_from_host_equals_device_call(T, fragment, init_state):
    b = inputs.make_batch(B=1, T=T, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=60 + T,
                          init_state=True)
    out_h, st_h = _host_run(b, fragment, init_state)
    out_d, st_d = _device_run(b, init_state)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    assert torch.equal(out_h, out_d) and torch.equal(st_h, st_d)


def test_from_host_against_oracle():
    b = inputs.make_batch(B=1, T=700, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=70,
                          init_state=True, slow_gate=True)
    out_h, st_h = _host_run(b, 192, True)
    ro, rs = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, b.state, None, B=1, threads=threads())
    assert prefill_out_err(out_h, ro) <= PREFILL_OUT_TOL
    assert state_err(st_h, rs[0]) <= STATE_TOL


def test_from_host_empty_prompt_passes_state():
    b = inputs.make_batch(B=1, T=64, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=71,
                          init_state=True)
    e = lambda x: x[:0].contiguous()  # noqa: E731
    sin = b.state[0].pin_memory()
    sout = torch.full((4, 128, 128), float("nan")).pin_memory()
    dev = {"q": None, "k": None, "v": None, "g": None, "b": None, "out": None,
           "state": torch.empty(4, 128, 128, device=DEV)}
    gdn.gdn_prefill_from_host(e(b.q), e(b.k), e(b.v), e(b.g), e(b.b), sin, sout, e(b.v), dev, fragment=64)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(sout, b.state[0])


def test_from_host_pageable_memory_and_short_last_fragment():
    """Pageable host tensors work too (the copies then do not overlap), and a last fragment of a
    few tokens goes through the token scan: equal to the device call within the oracle's bars."""
    b = inputs.make_batch(B=1, T=64 * 5 + 3, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=72,
                          init_state=True)
    host = {n: getattr(b, n).clone() for n in ("q", "k", "v", "g", "b")}  # pageable
    sout = torch.empty(4, 128, 128)
    out = torch.empty(b.v.shape, dtype=b.v.dtype)
    dev = {n: torch.empty_like(t, device=DEV) for n, t in host.items()}
    dev["out"] = torch.empty(b.v.shape, dtype=b.v.dtype, device=DEV)
    dev["state"] = torch.empty(4, 128, 128, device=DEV)
    gdn.gdn_prefill_from_host(host["q"], host["k"], host["v"], host["g"], host["b"], b.state[0].clone(), sout, out,
                              dev, chunk=64, fragment=64)
    torch.cuda.current_stream().synchronize()
    ro, rs = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, b.state, None, B=1, threads=threads())
    assert prefill_out_err(out, ro) <= PREFILL_OUT_TOL
    assert state_err(sout, rs[0]) <= STATE_TOL
