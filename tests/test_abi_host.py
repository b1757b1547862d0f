"""Host-side tests of the C ABI: the library loads, exports what gdn.h declares,
and rejects bad arguments with the documented status before any device work.

These calls never launch a kernel; they run without a GPU.
"""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc is needed to build the library")


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_delta_gb300 import _build
    import gated_deltanet_linear_delta_gb300 as gdn
    _build.build()
    return gdn.library()


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"^GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"gdn_prefill", "gdn_decode_step", "gdn_get_device_status", "gdn_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared in gdn.h but not exported"


def test_status_strings(lib):
    import gated_deltanet_linear_delta_gb300 as gdn
    assert gdn.gdn_status_string(0) == "GDN_OK"
    assert gdn.gdn_status_string(-1) == "GDN_ERR_INVALID_ARG"
    assert gdn.gdn_status_string(-2) == "GDN_ERR_UNSUPPORTED"
    assert gdn.gdn_status_string(-3) == "GDN_ERR_CUDA"
    assert gdn.gdn_status_string(-4) == "GDN_ERR_DEVICE_CHECK"
    assert gdn.gdn_status_string(7) == "GDN_UNKNOWN_STATUS"


A = 4096  # a 16-byte aligned fake address: validation never dereferences it


def prefill(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, si=None, so=A, out=A, cu=None, B=1, T=64, Hk=2, Hv=4,
                dk=128, dv=128, chunk=64, dtype=0)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gdn_prefill(p(args["q"]), p(args["k"]), p(args["v"]), p(args["g"]), p(args["b"]),
                           p(args["si"]), p(args["so"]), p(args["out"]), p(args["cu"]), args["B"],
                           args["T"], args["Hk"], args["Hv"], args["dk"], args["dv"], args["chunk"],
                           args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=48), -2), (dict(dv=256), -2), (dict(chunk=128), -2), (dict(chunk=0), -2),
    (dict(dtype=5), -2), (dict(Hk=3, Hv=4), -1), (dict(Hk=0), -1), (dict(B=-1), -1),
    (dict(T=-5), -1), (dict(q=A + 2), -1), (dict(out=A + 8), -1), (dict(cu=A + 4), -1),
    (dict(so=None), -1), (dict(v=None), -1), (dict(B=70000), -1),
])
def test_prefill_rejects(lib, kw, code):
    assert prefill(lib, **kw) == code


def test_prefill_zero_batch_is_a_noop(lib):
    assert prefill(lib, B=0) == 0


def prefill_static(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, si=None, so=A, out=A, cu=None, B=1, T=64, Hk=2, Hv=4,
                dk=128, dv=128, chunk=64, dtype=0)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gdn_prefill_static(p(args["q"]), p(args["k"]), p(args["v"]), p(args["g"]), p(args["b"]),
                                  p(args["si"]), p(args["so"]), p(args["out"]), p(args["cu"]), args["B"],
                                  args["T"], args["Hk"], args["Hv"], args["dk"], args["dv"], args["chunk"],
                                  args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=48), -2), (dict(chunk=128), -2), (dict(Hk=3, Hv=4), -1), (dict(B=-1), -1),
    (dict(q=A + 2), -1), (dict(so=None), -1),
])
def test_prefill_static_rejects(lib, kw, code):
    assert prefill_static(lib, **kw) == code


def test_prefill_static_zero_batch_is_a_noop(lib):
    assert prefill_static(lib, B=0) == 0


@pytest.mark.parametrize("sizes", [
    (1, 64, 2, 4, 48, 128, 64, 0), (1, 64, 3, 4, 128, 128, 64, 0), (-1, 64, 2, 4, 128, 128, 64, 0),
    (0, 64, 2, 4, 128, 128, 64, 0), (1, 64, 2, 4, 128, 128, 128, 0),
])
def test_workspace_size_is_zero_for_rejected_or_empty_sizes(lib, sizes):
    assert lib.gdn_prefill_workspace_size(*sizes) == 0


def decode(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, st=A, out=A, N=4, Hk=2, Hv=4, dk=128, dv=128, dtype=0)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gdn_decode_step(p(args["q"]), p(args["k"]), p(args["v"]), p(args["g"]), p(args["b"]),
                               p(args["st"]), p(args["out"]), args["N"], args["Hk"], args["Hv"],
                               args["dk"], args["dv"], args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=16), -2), (dict(dv=96), -2), (dict(dtype=2), -2), (dict(Hk=3, Hv=4), -1),
    (dict(N=-1), -1), (dict(st=None), -1), (dict(q=A + 4), -1), (dict(out=None), -1),
])
def test_decode_rejects(lib, kw, code):
    assert decode(lib, **kw) == code


def test_decode_zero_batch_is_a_noop(lib):
    assert decode(lib, N=0) == 0


def decode_slots(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, pool=A, slots=A, out=A, N=4, S=8, Hk=2, Hv=4, dk=128, dv=128,
                dtype=0)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gdn_decode_step_slots(p(args["q"]), p(args["k"]), p(args["v"]), p(args["g"]), p(args["b"]),
                                     p(args["pool"]), p(args["slots"]), p(args["out"]), args["N"], args["S"],
                                     args["Hk"], args["Hv"], args["dk"], args["dv"], args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=16), -2), (dict(dtype=2), -2), (dict(Hk=3, Hv=4), -1), (dict(N=-1), -1), (dict(S=-1), -1),
    (dict(slots=None), -1), (dict(slots=A + 4), -1), (dict(pool=None), -1), (dict(pool=A + 8), -1),
    (dict(out=None), -1),
])
def test_decode_slots_rejects(lib, kw, code):
    assert decode_slots(lib, **kw) == code


def test_decode_slots_zero_batch_is_a_noop(lib):
    assert decode_slots(lib, N=0) == 0


def from_host(lib, **kw):
    args = dict(T=256, fragment=128, chunk=64, dk=128, sd=A, so=A)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gdn_prefill_from_host(*([p(A)] * 5), None, p(args["so"]), p(A), *([p(A)] * 5), p(args["sd"]), p(A),
                                     args["T"], 2, 4, args["dk"], 128, args["chunk"], 0, args["fragment"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(fragment=0), -1), (dict(fragment=100), -1), (dict(T=-1), -1), (dict(so=None), -1),
    (dict(sd=None), -1), (dict(T=300 * 128), -1), (dict(dk=48), -2), (dict(chunk=48, fragment=96), -2),
])
def test_prefill_from_host_rejects(lib, kw, code):
    assert from_host(lib, **kw) == code


def test_prefill_path_selection(lib):
    import gated_deltanet_linear_delta_gb300 as gdn
    for T in (1, 4, 8):  # a few tokens per sequence: token scan
        assert gdn.gdn_prefill_path(16, T, 16, 32, 128, 128, 64, 0) == 2
    assert gdn.gdn_prefill_path(16, 9, 16, 32, 128, 128, 64, 0) == 1
    assert gdn.gdn_prefill_path(1, 64, 2, 4, 48, 128, 64, 0) == -2
    assert gdn.gdn_prefill_path(1, 64, 2, 4, 32, 32, 16, 1) == 0  # tiny fp32: CUDA-core kernel
    assert gdn.gdn_prefill_path(1, 4096, 16, 32, 128, 128, 64, 0) in (0, 1)


def test_valid_call_without_a_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert prefill(lib) == -3
