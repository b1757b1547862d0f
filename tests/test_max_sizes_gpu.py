"""The largest sequence counts the C ABI accepts (B = 65535: one grid dimension per sequence),
through each kernel, against the fp64 oracle. Heads are small so that states and the oracle stay
cheap; the sequence lengths include empty ones."""
import pytest
import torch

import oracle
from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import (DECODE_TOL, PREFILL_OUT_TOL, STATE_TOL, decode_out_err, prefill_out_err, state_err,
                   threads)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
B_MAX = 65535


def _prefill(b, T=None):
    d = b.to(DEV)
    out = torch.full(d.v.shape, float("nan"), dtype=d.v.dtype, device=DEV)
    so = torch.full((b.B, b.Hv, b.dv, b.dk), float("nan"), device=DEV)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state, so, out, d.cu_seqlens, B=b.B, T=T, chunk=b.chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    return out, so


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_65535_packed_sequences_cuda_core_kernel(dtype):
    gen = torch.Generator().manual_seed(80)
    lengths = torch.randint(0, 4, (B_MAX,), generator=gen).tolist()  # 0..3 tokens, empty ones included
    b = inputs.make_batch(Hk=1, Hv=2, dk=32, dv=32, dtype=dtype, chunk=16, seed=81, init_state=True, lengths=lengths)
    # the path query takes tokens per sequence (no cu_seqlens); any T > 8 names the block kernel
    assert gdn.gdn_prefill_path(B_MAX, 9, 1, 2, 32, 32, 16, gdn.GDN_F32 if dtype == "f32" else gdn.GDN_BF16) == 0
    out, so = _prefill(b)
    ro, rs = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, b.state, b.cu_seqlens, threads=threads())
    assert prefill_out_err(out, ro) <= PREFILL_OUT_TOL
    assert state_err(so, rs) <= STATE_TOL
    empty = [n for n, L in enumerate(lengths) if L == 0]
    assert torch.equal(so[empty].cpu(), b.state[empty])  # an empty sequence passes its state through


def test_65535_sequences_of_two_tokens_token_scan():
    b = inputs.make_batch(B=B_MAX, T=2, Hk=1, Hv=2, dk=32, dv=64, dtype="bf16", chunk=16, seed=82, init_state=True)
    assert gdn.gdn_prefill_path(B_MAX, 2, 1, 2, 32, 64, 16, gdn.GDN_BF16) == 2
    out, so = _prefill(b, T=2)
    ro, rs = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, b.state, None, B=B_MAX, threads=threads())
    assert prefill_out_err(out, ro) <= DECODE_TOL
    assert state_err(so, rs) <= STATE_TOL


def test_4096_packed_sequences_tensor_core_kernel():
    """More sequences than the longest-first ordering ranks (it then keeps index order)."""
    gen = torch.Generator().manual_seed(83)
    lengths = torch.randint(0, 70, (4096,), generator=gen).tolist()
    b = inputs.make_batch(Hk=1, Hv=1, dk=128, dv=128, dtype="bf16", chunk=64, seed=84, init_state=True,
                          lengths=lengths)
    assert gdn.gdn_prefill_path(4096, 9, 1, 1, 128, 128, 64, gdn.GDN_BF16) == 1
    out, so = _prefill(b)
    ro, rs = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, b.state, b.cu_seqlens, threads=threads())
    assert prefill_out_err(out, ro) <= PREFILL_OUT_TOL
    assert state_err(so, rs) <= STATE_TOL


def test_decode_100000_sequences():
    q, k, v, g, bb, st = inputs.make_decode_inputs(100000, Hk=1, Hv=2, dk=32, dv=32, seed=85)
    q, k, v, g, bb = q[0], k[0], v[0], g[0], bb[0]
    sd = st.to(DEV)
    out = torch.full(v.shape, float("nan"), dtype=v.dtype, device=DEV)
    gdn.gdn_decode_step(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), bb.to(DEV), sd, out)
    torch.cuda.synchronize()
    ro, rs = oracle.gdn_decode_step(q, k, v, g, bb, st, threads=threads())
    assert decode_out_err(out, ro)[0] <= DECODE_TOL
    assert state_err(sd, rs) <= STATE_TOL
