"""The allocation-free BatchNorm forward entry point.

`gbn_bn_forward_train_noalloc` serves callers that cannot allocate device
memory (inside a graph capture, a real-time loop, or a host framework that
owns every allocation): its scratch is a fixed device array inside the
library instead of a caller-provided workspace.  This file calls it through
the C ABI twice in a row, on two different workloads, and checks each
result against the ordinary `gbn_bn_forward_train` (which takes a
workspace) within the fp32 / bf16 parity tolerances of the other tests.

It is named so that pytest collects it last."""

import ctypes

import pytest
import torch

from bwd_bn_pass_gb300 import synth

from . import tolerances as tol

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["auto", "persistent"])
def _bn_path(request, gbn):
    """Every test runs twice: with the library's default size threshold for
    the single-launch persistent kernel, and with the threshold at 0 so that
    the persistent kernel takes every eligible shape, small ones included."""
    if request.param == "persistent":
        prev = gbn.bn_set_persistent_min_bytes(0)
        yield
        gbn.bn_set_persistent_min_bytes(prev)
    else:
        yield


DEV = "cuda:0"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _run(gbn, case, noalloc):
    inp = synth.bn_inputs(case)
    x = inp["x"].to(DEV)
    B, C = x.shape[:2]
    HW = x.numel() // (B * C)
    g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    rm, rv = inp["running_mean"].to(DEV), inp["running_var"].to(DEV)
    y = torch.empty_like(x)
    stats = torch.empty(8 * C, dtype=torch.float32, device=DEV)
    code = 0 if x.dtype == torch.float32 else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    L = gbn.lib()
    if noalloc:
        st = L.gbn_bn_forward_train_noalloc(_ptr(x), code, B, C, HW, _ptr(g), _ptr(b), _ptr(rm),
                                            _ptr(rv), case.momentum, case.eps, _ptr(y),
                                            _ptr(stats), stream)
    else:
        ws = torch.empty(L.gbn_bn_workspace_bytes(B, C, HW, -1), dtype=torch.uint8, device=DEV)
        st = L.gbn_bn_forward_train(_ptr(x), code, B, C, HW, _ptr(g), _ptr(b), _ptr(rm),
                                    _ptr(rv), case.momentum, case.eps, _ptr(y), _ptr(stats),
                                    _ptr(ws), ws.numel(), stream)
    assert st == 0, L.gbn_status_string(st)
    torch.cuda.synchronize()
    return {"y": y.cpu(), "stats": stats[:4 * C].cpu(), "rm": rm.cpu(), "rv": rv.cpu()}


def _compare(got, ref, dtype, what):
    for k in ("stats", "rm", "rv"):
        tol.check_f32(got[k], ref[k].double(), f"{what} {k}")
    if dtype == "f32":
        tol.check_f32(got["y"], ref["y"].double(), f"{what} y")
    else:
        r = ref["y"].double()
        B, C = r.shape[:2]
        r3 = r.reshape(B, C, -1)
        tol.check_bf16(got["y"].reshape(B, C, -1), r3, f"{what} y",
                       tol.tau_of(r3.numpy(), axis=(0, 2)))


def test_noalloc_forward_matches_workspace_forward_twice(gbn):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = [synth.CASES["bn_ragged_f32"],
             synth.BNCase("noalloc_bf16", (16, 64, 28, 28), "bf16", mu_range=(-100, 100),
                          sigma_range=(0.01, 10), seed=7),
             # many channels: the single-launch kernel's scratch would not fit
             # the fixed array, so the call runs the two-launch kernels
             synth.BNCase("noalloc_wide_f32", (64, 3000, 8, 8), "f32", mu_range=(-10, 10),
                          seed=8)]
    refs = [_run(gbn, c, noalloc=False) for c in cases]
    for c, ref in zip(cases, refs):          # two calls in a row
        got = _run(gbn, c, noalloc=True)
        _compare(got, ref, c.dtype, c.name)
