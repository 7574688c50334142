"""The allocation-free BatchNorm forward entry point.

`gbn_bn_forward_train_noalloc` serves callers that cannot allocate device
memory (inside a graph capture, a real-time loop, or a host framework that
owns every allocation): its scratch is a fixed device array inside the
library instead of a caller-provided workspace.

This file calls it through the C ABI twice in a row per workload and checks
each result three ways:
  * against the float64 oracle at the parity tolerances of the other tests;
  * bit for bit against the ordinary `gbn_bn_forward_train` (which takes a
    workspace) run on the same kernel path -- the entry point runs the same
    deterministic kernels: the small-channel single launch, the two-launch
    pair or, when its scratch fits, the single-launch persistent kernel;
  * bit for bit between its own two calls.
It also checks the size limit (more channels than the fixed array can hold
is GBN_EWORKSPACE, rejected before any launch) and that the device status
word stays clean.

It is named so that pytest collects it last."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
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
HUGE = 1 << 62  # a size threshold no tensor reaches: two-launch kernels only
GBN_EWORKSPACE = -4


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(gbn, inp, case, noalloc):
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


def _workspace_forms(gbn, inp, case):
    """gbn_bn_forward_train on each kernel path it can take: the
    small-channel single launch, the two-launch pair, and the persistent
    kernel wherever the shape is eligible."""
    prev = gbn.bn_set_persistent_min_bytes(HUGE)
    prev_small = gbn.bn_set_small_max_elems(0)
    try:
        forms = [_call(gbn, inp, case, noalloc=False)]       # two launches
        gbn.bn_set_small_max_elems(prev_small)
        forms.append(_call(gbn, inp, case, noalloc=False))  # small channels: one launch
        gbn.bn_set_persistent_min_bytes(0)
        forms.append(_call(gbn, inp, case, noalloc=False))  # persistent
    finally:
        gbn.bn_set_persistent_min_bytes(prev)
        gbn.bn_set_small_max_elems(prev_small)
    return forms


def _bit_equal(a, b):
    return all(torch.equal(a[k], b[k]) for k in ("y", "stats", "rm", "rv"))


def _check_oracle(got, inp, case):
    x = inp["x"].double().numpy()
    f = oracle.batch_norm_forward_train(
        x, inp["gamma"].double().numpy(), inp["beta"].double().numpy(),
        inp["running_mean"].double().numpy(), inp["running_var"].double().numpy(),
        case.momentum, case.eps)
    C = x.shape[1]
    s = got["stats"]
    for i, k in enumerate(("mean", "var", "inv_std", "scale")):
        tol.check_f32(s[i * C:(i + 1) * C], f[k], f"{case.name} {k}")
    tol.check_f32(got["rm"], f["running_mean"], f"{case.name} running_mean")
    tol.check_f32(got["rv"], f["running_var"], f"{case.name} running_var")
    if case.dtype == "f32":
        tol.check_f32(got["y"], f["y"], f"{case.name} y")
    else:
        B = x.shape[0]
        r3 = f["y"].reshape(B, C, -1)
        tol.check_bf16(got["y"].reshape(B, C, -1), r3, f"{case.name} y",
                       tol.tau_of(r3, axis=(0, 2)))


CASES = [
    synth.CASES["bn_ragged_f32"],
    synth.BNCase("noalloc_bf16", (16, 64, 28, 28), "bf16", mu_range=(-100, 100),
                 sigma_range=(0.01, 10), seed=7),
    # many channels: the single-launch kernel's scratch would not fit the
    # fixed array, so the call runs the two-launch kernels
    synth.BNCase("noalloc_wide_f32", (16, 3000, 8, 8), "f32", mu_range=(-10, 10), seed=8),
]


@pytest.mark.parametrize("case", CASES, ids=[c.name for c in CASES])
def test_noalloc_forward_two_calls_in_a_row(gbn, case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    inp = synth.bn_inputs(case)
    forms = _workspace_forms(gbn, inp, case)
    gbn.get_device_status(clear=True)
    first = _call(gbn, inp, case, noalloc=True)
    second = _call(gbn, inp, case, noalloc=True)   # the same inputs, right after
    assert _bit_equal(first, second), f"{case.name}: two calls differ"
    for got in (first, second):
        assert any(_bit_equal(got, f) for f in forms), (
            f"{case.name}: matches no kernel path of the workspace forward bit for bit")
        _check_oracle(got, inp, case)
    assert gbn.get_device_status() == 0, "device status word reports an error"


def test_noalloc_rejects_channels_beyond_the_fixed_array(gbn):
    """C = 5000 needs 16 * 5000 bytes of partials (one block per channel),
    more than the 64 KiB array: GBN_EWORKSPACE, and y is left untouched."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, C, HW = 2, 5000, 4
    gen = torch.Generator(device=DEV).manual_seed(20241209)
    x = torch.randn(B, C, HW, device=DEV, generator=gen)
    y = torch.full_like(x, 7.0)
    stats = torch.zeros(8 * C, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    L = gbn.lib()
    st = L.gbn_bn_forward_train_noalloc(_ptr(x), 0, B, C, HW, None, None, None, None, 0.1, 1e-5,
                                        _ptr(y), _ptr(stats), stream)
    torch.cuda.synchronize()
    assert st == GBN_EWORKSPACE, L.gbn_status_string(st)
    assert bool((y == 7.0).all()) and bool((stats == 0).all())
    # the largest channel count the array holds still runs
    C = 4096
    x = torch.randn(B, C, HW, device=DEV, generator=gen)
    y = torch.empty_like(x)
    stats = torch.empty(8 * C, device=DEV)
    st = L.gbn_bn_forward_train_noalloc(_ptr(x), 0, B, C, HW, None, None, None, None, 0.1, 1e-5,
                                        _ptr(y), _ptr(stats), stream)
    torch.cuda.synchronize()
    assert st == 0, L.gbn_status_string(st)
    f = oracle.batch_norm_forward_train(x.double().cpu().numpy(), np.ones(C), np.zeros(C),
                                        np.zeros(C), np.ones(C), 0.1, 1e-5)
    tol.check_f32(y.cpu(), f["y"], "C=4096 y")
