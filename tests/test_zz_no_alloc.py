"""gdn_prefill_static, the prefill entry point that allocates nothing at call time, through the
C ABI.

On the tensor-core sizes it runs the same kernels as gdn_prefill, with the scratch taken from a
fixed array in the library's device image and at most 8 state-carrying CTAs; on the other sizes
it runs gdn_prefill's scratch-free kernels. Its results are compared with gdn_prefill's on the
same inputs, on two consecutive calls (the second runs on the scratch the first one left), within
the parity tolerances of the suite. The file name sorts last, so in a full run these tests also
run after every other test of the suite; they pass alone in a fresh process too.
"""
import ctypes

import pytest
import torch

from gated_deltanet_linear_delta_gb300 import inputs
import gated_deltanet_linear_delta_gb300 as gdn

from _util import PREFILL_OUT_TOL, STATE_TOL, prefill_out_err, state_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call(entry, d, si, so, out):
    """One call of a gdn_prefill-shaped C entry point on the current stream; returns its status."""
    lib = gdn.library()
    fn = getattr(lib, entry)
    fn.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 8 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    B = d.B if d.cu_seqlens is None else d.cu_seqlens.numel() - 1
    T = d.T if d.cu_seqlens is None else d.q.shape[0]
    dtype = gdn.GDN_BF16 if d.q.dtype == torch.bfloat16 else gdn.GDN_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(_p(d.q), _p(d.k), _p(d.v), _p(d.g), _p(d.b), _p(si), _p(so), _p(out), _p(d.cu_seqlens),
              B, T, d.Hk, d.Hv, d.dk, d.dv, d.chunk, dtype, stream)


def buffers(batch):
    out = torch.full((batch.q.shape[0], batch.Hv, batch.dv), float("nan"), dtype=batch.v.dtype, device=DEV)
    so = torch.full((batch.B, batch.Hv, batch.dv, batch.dk), float("nan"), device=DEV)
    return out, so


CASES = {
    # tensor-core sizes: the fixed scratch is used
    "B1_T1000_seeded_state": lambda: inputs.make_batch(B=1, T=1000, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16",
                                                       chunk=64, seed=11, init_state=True),
    "varlen_5_seqs": lambda: inputs.make_batch(Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=12,
                                               init_state=True, lengths=[300, 1, 64, 777, 129]),
    "B3_T200_zero_state": lambda: inputs.make_batch(B=3, T=200, Hk=4, Hv=16, dk=128, dv=128, dtype="bf16",
                                                    chunk=64, seed=13),
    # scratch-free sizes (token scan; CUDA-core blocks)
    "scan_B4_T3": lambda: inputs.make_batch(B=4, T=3, Hk=16, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64,
                                            seed=14, init_state=True),
    "fp32_B2_T100": lambda: inputs.make_batch(B=2, T=100, Hk=2, Hv=4, dk=64, dv=64, dtype="f32", chunk=32,
                                              seed=15, init_state=True),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_matches_gdn_prefill_on_two_consecutive_calls(case):
    batch = CASES[case]()
    d = batch.to(DEV)
    ref_out, ref_so = buffers(batch)
    assert call("gdn_prefill", d, d.state, ref_so, ref_out) == gdn.GDN_OK
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    ro = ref_out.double().cpu().numpy()
    rs = ref_so.double().cpu().numpy()
    for _ in range(2):
        out, so = buffers(batch)
        assert call("gdn_prefill_static", d, d.state, so, out) == gdn.GDN_OK
        torch.cuda.synchronize()
        assert gdn.gdn_get_device_status() == gdn.GDN_OK
        eo, es = prefill_out_err(out, ro), state_err(so, rs)
        assert eo <= PREFILL_OUT_TOL, f"{case}: output max-abs/RMS {eo:.3e} against gdn_prefill"
        assert es <= STATE_TOL, f"{case}: state rel-Frobenius {es:.3e} against gdn_prefill"


def test_in_place_state_and_no_device_memory_taken():
    """The state updated in place (state_in == state_out); the device's free memory is the same
    before and after calls made once the first call has done its set-up."""
    batch = CASES["B1_T1000_seeded_state"]()
    d = batch.to(DEV)
    ref_out, ref_so = buffers(batch)
    assert call("gdn_prefill", d, d.state, ref_so, ref_out) == gdn.GDN_OK
    st = d.state.clone()
    out = torch.full_like(ref_out, float("nan"))
    assert call("gdn_prefill_static", d, st, st, out) == gdn.GDN_OK  # first call: set-up
    torch.cuda.synchronize()
    assert state_err(st, ref_so.double().cpu().numpy()) <= STATE_TOL
    st2 = d.state.clone()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        st2.copy_(d.state)
        assert call("gdn_prefill_static", d, st2, st2, out) == gdn.GDN_OK
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    assert state_err(st2, ref_so.double().cpu().numpy()) <= STATE_TOL


def test_sizes_over_the_fixed_scratch_are_rejected():
    """Hv/Hk = 16 needs 16 state-carrying CTAs (24 MiB of ring): GDN_ERR_UNSUPPORTED, and nothing
    is written."""
    batch = inputs.make_batch(B=1, T=256, Hk=2, Hv=32, dk=128, dv=128, dtype="bf16", chunk=64, seed=16)
    d = batch.to(DEV)
    out, so = buffers(batch)
    assert call("gdn_prefill_static", d, None, so, out) == gdn.GDN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and torch.isnan(so).all()
    # the same sizes through gdn_prefill still run
    assert call("gdn_prefill", d, None, so, out) == gdn.GDN_OK
    torch.cuda.synchronize()
    assert not torch.isnan(so).any()
