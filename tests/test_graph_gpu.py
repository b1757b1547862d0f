"""Capture of the library's calls in CUDA graphs: a captured sequence of decode steps (plain and
slot-indexed) and a captured prefill, replayed, give bit-for-bit the results of the same calls
run eagerly. The graph replays the same kernels with the same arguments, so nothing may differ.

Calls that set up per-device state on first use (the device status word) are made once before
any capture, as a user of the library does.
"""
import pytest
import torch

from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _capture(fn, warm=2):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def test_graph_of_decode_steps_matches_eager():
    steps, N = 12, 8
    q, k, v, g, b, state = inputs.make_decode_inputs(N, seed=31, steps=steps)
    q, k, v, g, b = (x.to(DEV) for x in (q, k, v, g, b))
    st_graph = state.to(DEV)
    outs_graph = torch.empty(steps, N, 32, 128, dtype=torch.bfloat16, device=DEV)

    def run(st, outs):
        for t in range(steps):
            gdn.gdn_decode_step(q[t], k[t], v[t], g[t], b[t], st, outs[t])

    graph = _capture(lambda: run(st_graph, outs_graph))
    # replay from the initial state, twice: the state is carried in place through the captured steps
    st_graph.copy_(state.to(DEV))
    graph.replay()
    graph.replay()
    st_eager = state.to(DEV)
    outs_eager = torch.empty_like(outs_graph)
    run(st_eager, outs_eager)
    run(st_eager, outs_eager)
    torch.cuda.synchronize()
    assert torch.equal(st_graph, st_eager)
    assert torch.equal(outs_graph, outs_eager)


def test_graph_of_slot_decode_matches_eager():
    N, num_slots = 6, 10
    q, k, v, g, b, _ = inputs.make_decode_inputs(N, Hk=2, Hv=4, seed=33)
    q, k, v, g, b = (x[0].to(DEV) for x in (q, k, v, g, b))
    gen = torch.Generator().manual_seed(34)
    pool0 = (torch.randn(num_slots, 4, 128, 128, generator=gen) * 0.02).to(DEV)
    slots = torch.tensor([7, -1, 2, 9, 0, 4], dtype=torch.int32, device=DEV)
    out_g, out_e = (torch.empty(N, 4, 128, dtype=torch.bfloat16, device=DEV) for _ in range(2))
    pool_g = pool0.clone()
    gdn.gdn_decode_step_slots(q, k, v, g, b, pool0.clone(), slots, out_e)  # first call: per-device set-up
    graph = _capture(lambda: gdn.gdn_decode_step_slots(q, k, v, g, b, pool_g, slots, out_g))
    pool_g.copy_(pool0)
    graph.replay()
    pool_e = pool0.clone()
    gdn.gdn_decode_step_slots(q, k, v, g, b, pool_e, slots, out_e)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    assert torch.equal(pool_g, pool_e) and torch.equal(out_g, out_e)


def test_graph_of_prefill_matches_eager():
    batch = inputs.make_batch(B=1, T=640, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=35,
                              init_state=True)
    d = batch.to(DEV)
    outs = [torch.empty(640, 32, 128, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    sts = [torch.empty(1, 32, 128, 128, device=DEV) for _ in range(2)]
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state, sts[1], outs[1], None, B=1, chunk=64)  # set-up
    graph = _capture(lambda: gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state, sts[0], outs[0], None, B=1,
                                             chunk=64))
    outs[0].zero_()
    sts[0].zero_()
    graph.replay()
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state, sts[1], outs[1], None, B=1, chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(sts[0], sts[1])


def test_graph_of_few_token_prefill_matches_eager():
    """The few-token (token-scan) path, in place, captured and replayed."""
    b = inputs.make_batch(B=16, T=4, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=36,
                          init_state=True)
    d = b.to(DEV)
    out_g, out_e = torch.empty_like(d.v), torch.empty_like(d.v)
    st_g, st_e = d.state.clone(), d.state.clone()
    graph = _capture(lambda: gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, st_g, st_g, out_g, None, B=16, T=4))
    st_g.copy_(d.state)
    graph.replay()
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, st_e, st_e, out_e, None, B=16, T=4)
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e) and torch.equal(st_g, st_e)
