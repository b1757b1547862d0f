"""gdn_prefill_ws and gdn_prefill_workspace_size: the prefill with a caller-owned workspace.

The tensor-core kernel keeps its ring of prepared blocks and its per-call tables in the
workspace. The same inputs through gdn_prefill (the library's own workspace) and through
gdn_prefill_ws (the caller's) must give identical results; a workspace that is missing, too
small or misaligned is rejected before any device work; two calls on two streams with their
own workspaces may overlap.
"""
import ctypes

import pytest
import torch

from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import PREFILL_OUT_TOL, STATE_TOL, oracle_prefill, prefill_out_err, state_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bufs(b):
    out = torch.full((b.q.shape[0], b.Hv, b.dv), float("nan"), dtype=b.v.dtype, device=DEV)
    so = torch.full((b.B, b.Hv, b.dv, b.dk), float("nan"), device=DEV)
    return out, so


def _size(b):
    B = b.B if b.cu_seqlens is None else b.cu_seqlens.numel() - 1
    T = b.T if b.cu_seqlens is None else b.q.shape[0]
    return gdn.gdn_prefill_workspace_size(B, T, b.Hk, b.Hv, b.dk, b.dv, b.chunk, gdn.GDN_BF16)


CASES = {
    "B1_T700_seeded": lambda: inputs.make_batch(B=1, T=700, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64,
                                                seed=31, init_state=True),
    "varlen_6": lambda: inputs.make_batch(Hk=4, Hv=8, dk=128, dv=128, dtype="bf16", chunk=64, seed=32,
                                          init_state=True, lengths=[129, 0, 64, 1000, 5, 300]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_caller_workspace_equals_library_workspace(case):
    b = CASES[case]()
    d = b.to(DEV)
    nbytes = _size(b)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    ref_out, ref_so = _bufs(b)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state, ref_so, ref_out, d.cu_seqlens,
                    B=None if d.cu_seqlens is not None else b.B, chunk=64)
    out, so = _bufs(b)
    gdn.gdn_prefill_ws(d.q, d.k, d.v, d.g, d.b, d.state, so, out, ws, d.cu_seqlens,
                       B=None if d.cu_seqlens is not None else b.B, chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    assert torch.equal(out, ref_out) and torch.equal(so, ref_so)
    ro, rs, _ = oracle_prefill(b)
    assert prefill_out_err(out, ro) <= PREFILL_OUT_TOL
    assert state_err(so, rs) <= STATE_TOL


def test_bad_workspaces_are_rejected_before_any_work():
    b = CASES["B1_T700_seeded"]()
    d = b.to(DEV)
    nbytes = _size(b)
    big = torch.empty(nbytes + 512, dtype=torch.uint8, device=DEV)
    lib = gdn.library()
    out, so = _bufs(b)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(ptr, size):
        return lib.gdn_prefill_ws(P(d.q), P(d.k), P(d.v), P(d.g), P(d.b), P(d.state), P(so), P(out), None, 1,
                                  b.T, b.Hk, b.Hv, 128, 128, 64, gdn.GDN_BF16, ptr, size, stream)
    assert call(None, 0) == gdn.GDN_ERR_INVALID_ARG
    assert call(ctypes.c_void_p(big.data_ptr()), nbytes - 1) == gdn.GDN_ERR_INVALID_ARG
    assert call(ctypes.c_void_p(big.data_ptr() + 128), nbytes) == gdn.GDN_ERR_INVALID_ARG  # 128-byte aligned only
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and torch.isnan(so).all()
    assert call(ctypes.c_void_p(big.data_ptr()), nbytes) == gdn.GDN_OK
    torch.cuda.synchronize()
    assert not torch.isnan(so).any()
    # the size is the tensor-core kernel's even for sizes that run the token scan without
    # cu_seqlens (with cu_seqlens they take the block kernel); sizes it does not take need none
    assert gdn.gdn_prefill_workspace_size(4, 3, 16, 32, 128, 128, 64, gdn.GDN_BF16) > 0
    assert gdn.gdn_prefill_workspace_size(2, 100, 2, 4, 64, 64, 32, gdn.GDN_F32) == 0


def test_two_streams_with_their_own_workspaces():
    bs = [inputs.make_batch(B=1, T=900, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=40 + i,
                            init_state=True) for i in range(2)]
    ds = [b.to(DEV) for b in bs]
    wss = [torch.empty(_size(b), dtype=torch.uint8, device=DEV) for b in bs]
    bufs = [_bufs(b) for b in bs]
    streams = [torch.cuda.Stream() for _ in bs]
    torch.cuda.synchronize()
    for d, ws, (out, so), st in zip(ds, wss, bufs, streams):
        with torch.cuda.stream(st):
            gdn.gdn_prefill_ws(d.q, d.k, d.v, d.g, d.b, d.state, so, out, ws, None, B=1, chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    for b, (out, so) in zip(bs, bufs):
        ro, rs, vh = oracle_prefill(b, key_heads=[0, 9])
        assert prefill_out_err(out[:, vh], ro) <= PREFILL_OUT_TOL
        assert state_err(so[:, vh], rs) <= STATE_TOL
