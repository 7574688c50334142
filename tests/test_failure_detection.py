"""Failure detection without a GPU fault.

Every cross-CTA and ring wait of the library is bounded: after its limit it
records GBN_DEV_WAIT_TIMEOUT in the device status word and the kernel
returns.  The self-test entry point makes one such wait run out (a barrier
nothing completes); the host then reads the status, clears it, and the
context keeps working.  Nothing here faults, traps or hangs the GPU."""

import pytest
import torch

from bwd_bn_pass_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_expired_wait_reports_status_and_context_stays_usable(gbn):
    gbn.init(0)
    torch.cuda.synchronize()
    assert gbn.get_device_status(clear=True) == 0
    gbn.selftest_bounded_wait(50_000_000)  # 50 ms
    torch.cuda.synchronize()
    st = gbn.get_device_status(clear=True)
    assert st & gbn.GBN_DEV_WAIT_TIMEOUT
    assert gbn.get_device_status() == 0  # cleared
    # the context still runs kernels, and they leave the status clean
    inp = synth.bn_inputs(synth.CASES["bn_tiny_f32"])
    x = inp["x"].to(DEV)
    y, stats = gbn.bn_forward_train(x, None, None, None, None, 0.1, 1e-5)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    assert gbn.get_device_status() == 0


def test_selftest_argument_errors(gbn):
    L = gbn.lib()
    assert L.gbn_selftest_bounded_wait(0, None) == -1
    assert L.gbn_selftest_bounded_wait(3_000_000_000, None) == -1
