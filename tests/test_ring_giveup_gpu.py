"""The tensor-core prefill's give-up path, exercised without any fault.

Every wait of the kernel (mbarrier phases, ring-slot flags, the consumer counter) is bounded;
when a wait runs out, the kernel raises the device status word and a launch-wide abort flag,
every role drains its own copies and MMAs, and the launch ends. GDN_TEST_WAIT_CYCLES shortens
the wait limit (a test hook read at each call) so that the first wait that is not already
satisfied gives up. The call must then report GDN_ERR_DEVICE_CHECK through the status word,
and the next call with the normal limit must run correctly on the same workspace.
"""
import pytest
import torch

from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import PREFILL_OUT_TOL, STATE_TOL, oracle_prefill, prefill_out_err, state_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _call(d, B):
    out = torch.full(d.v.shape, float("nan"), dtype=d.v.dtype, device=DEV)
    so = torch.full((B, d.Hv, d.dv, d.dk), float("nan"), device=DEV)
    gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, d.state, so, out, d.cu_seqlens,
                    B=None if d.cu_seqlens is not None else B, chunk=d.chunk)
    torch.cuda.synchronize()
    return out, so


@pytest.mark.parametrize("cycles", ["1", "3000"])
def test_wait_give_up_is_reported_and_next_call_passes(cycles, monkeypatch):
    b = inputs.make_batch(B=2, T=700, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", chunk=64, seed=21,
                          init_state=True)
    assert gdn.gdn_prefill_path(b.B, b.T, b.Hk, b.Hv, 128, 128, 64, gdn.GDN_BF16) == 1
    d = b.to(DEV)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    monkeypatch.setenv("GDN_TEST_WAIT_CYCLES", cycles)
    _call(d, b.B)
    assert gdn.gdn_get_device_status() == gdn.GDN_ERR_DEVICE_CHECK
    assert gdn.gdn_get_device_status() == gdn.GDN_OK  # reading clears it
    monkeypatch.delenv("GDN_TEST_WAIT_CYCLES")
    out, so = _call(d, b.B)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    ro, rs, _ = oracle_prefill(b)
    assert prefill_out_err(out, ro) <= PREFILL_OUT_TOL
    assert state_err(so, rs) <= STATE_TOL
