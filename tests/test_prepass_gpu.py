"""The materialised pre-pass (inverse norms, beta, in-block cumulative gate) vs the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("chunk", [16, 64])
def test_prepass_varlen(dtype, chunk):
    b = inputs.make_batch(Hk=4, Hv=8, dk=128, dv=32, dtype=dtype, chunk=chunk, seed=21,
                          lengths=[0, 1, 70, 129, 5])
    d = b.to(DEV)
    T, Hk, Hv = b.tokens, b.Hk, b.Hv
    rq = torch.full((T, Hk), float("nan"), device=DEV)
    rk, beta, gc = torch.full_like(rq, float("nan")), torch.full((T, Hv), float("nan"), device=DEV), None
    gc = torch.full_like(beta, float("nan"))
    gdn.gdn_prepass(d.q, d.k, d.g, d.b, rq, rk, beta, gc, d.cu_seqlens, chunk=chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    erq, erk, ebeta, egc = oracle.gdn_prepass(b.q, b.k, b.g, b.b, b.cu_seqlens, chunk=chunk)
    np.testing.assert_allclose(rq.cpu().numpy(), erq, rtol=1e-5)
    np.testing.assert_allclose(rk.cpu().numpy(), erk, rtol=1e-5)
    np.testing.assert_allclose(beta.cpu().numpy(), ebeta, rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(gc.cpu().numpy(), egc, rtol=1e-5, atol=1e-5)


def test_prepass_fixed_length_batch():
    b = inputs.make_batch(B=3, T=100, Hk=2, Hv=4, dk=64, dv=32, dtype="bf16", chunk=32, seed=22)
    d = b.to(DEV)
    rq = torch.empty(300, 2, device=DEV)
    rk, beta, gc = torch.empty_like(rq), torch.empty(300, 4, device=DEV), torch.empty(300, 4, device=DEV)
    gdn.gdn_prepass(d.q, d.k, d.g, d.b, rq, rk, beta, gc, B=3, chunk=32)
    torch.cuda.synchronize()
    erq, erk, ebeta, egc = oracle.gdn_prepass(b.q, b.k, b.g, b.b, None, B=3, chunk=32)
    np.testing.assert_allclose(rq.cpu().numpy(), erq, rtol=1e-5)
    np.testing.assert_allclose(gc.cpu().numpy(), egc, rtol=1e-5, atol=1e-5)
