"""Prefill with fast gates, through the C ABI, against the fp64 oracle.

Inside a block the kernels form e^{G_t - G_s} (G the in-block cumulative log-decay) as the
product e^{G_t - gmin} e^{gmin - G_s} when the block's range gmax - gmin is below 80, and with
one exponential per element otherwise (the factors would overflow fp32). The standard gates
(g = -softplus(N(0,1))) span about 51 over a 64-token block, so only fast gates reach the second
form: at gate_scale 1.6 the blocks of one launch fall on both sides of the line, at 4 every full
block is beyond it, and decays of e^-200 underflow to zero inside a block. Each tensor-core
kernel (the ring kernel with and without key sharing, the cluster kernel) and the CUDA-core
kernel are run on such inputs.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import PREFILL_OUT_TOL, STATE_TOL, oracle_prefill, prefill_out_err, state_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
WIDE = 80.0  # the block range from which the kernels stop factoring e^{G_t - G_s}


def block_ranges(batch):
    """gmax - gmin of the in-block cumulative log-decay, for every (block, value head)."""
    g = batch.g.float().double().numpy()
    if batch.cu_seqlens is None:
        bounds = [(n * batch.T, (n + 1) * batch.T) for n in range(batch.B)]
    else:
        cu = batch.cu_seqlens.tolist()
        bounds = list(zip(cu[:-1], cu[1:]))
    out = []
    for lo, hi in bounds:
        for b0 in range(lo, hi, batch.chunk):
            G = np.cumsum(g[b0:min(b0 + batch.chunk, hi)], axis=0)
            out.extend(G.max(axis=0) - G.min(axis=0))
    return np.array(out)


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
    assert not torch.isnan(o).any() and not torch.isnan(s).any()
    eo, es = prefill_out_err(o, ro), state_err(s, rs)
    assert eo <= PREFILL_OUT_TOL, f"output max-abs/RMS {eo:.3e}"
    assert es <= STATE_TOL, f"state rel-Frobenius {es:.3e}"


def assert_ranges(batch, scale):
    r = block_ranges(batch)
    if scale < 2:  # both forms in one launch
        assert (r >= WIDE).any() and (r < WIDE).any(), (r.min(), r.max())
    else:  # every full block beyond the line
        assert np.median(r) >= 2 * WIDE, np.median(r)


@pytest.mark.parametrize("scale", [1.6, 4.0])
def test_ring_kernel_one_sequence(scale):
    """4 chains on as many state CTAs: the ring kernel without key sharing."""
    b = inputs.make_batch(B=1, T=700, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=61,
                          init_state=True, gate_scale=scale)
    assert gdn.gdn_prefill_path(1, 700, 2, 4, 128, 128, 64, gdn.GDN_BF16) == 1
    assert_ranges(b, scale)
    run_and_check(b)


@pytest.mark.parametrize("scale", [1.6, 4.0])
def test_ring_kernel_key_sharing(scale):
    """160 chains (4 sequences x 40 heads) on fewer state CTAs: the ring kernel with key sharing,
    whose later units of a key head take the Gram of the scaled fp16 tiles."""
    b = inputs.make_batch(Hk=20, Hv=40, dk=128, dv=128, dtype="bf16", chunk=64, seed=62, init_state=True,
                          lengths=[190, 64, 333, 500], gate_scale=scale)
    assert_ranges(b, scale)
    run_and_check(b, key_heads=[0, 7, 19])


@pytest.mark.parametrize("scale", [1.6, 4.0])
def test_cluster_kernel(scale, monkeypatch):
    monkeypatch.setenv("GDN_PREFILL_KERNEL", "cluster")
    b = inputs.make_batch(Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=63, init_state=True,
                          lengths=[0, 1, 65, 700], gate_scale=scale)
    assert_ranges(b, scale)
    run_and_check(b)


@pytest.mark.parametrize("scale", [1.6, 4.0])
def test_cuda_core_kernel(scale):
    """fp32, dk = dv = 64, blocks of 32 tokens: the CUDA-core block kernel."""
    b = inputs.make_batch(B=2, T=300, Hk=2, Hv=4, dk=64, dv=64, dtype="f32", chunk=32, seed=64, init_state=True,
                          gate_scale=scale * 2)
    assert gdn.gdn_prefill_path(2, 300, 2, 4, 64, 64, 32, gdn.GDN_F32) == 0
    run_and_check(b)
