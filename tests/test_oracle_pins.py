"""The float64 oracle against independent references (no GPU needed)."""

import numpy as np
import pytest

import oracle
from oracle import bn as obn, rmsnorm as orms, layernorm as oln

from . import pins
from .tolerances import check_f32, f32_violations


@pytest.mark.parametrize("pin", pins.BN_PINS, ids=lambda f: f.__name__)
def test_bn_pins(pin):
    if pin is pins.pin_bn_exact_rational:
        pytest.importorskip("sympy")
    pin(obn)


@pytest.mark.parametrize("pin", pins.RMS_PINS, ids=lambda f: f.__name__)
def test_rms_pins(pin):
    if pin is pins.pin_rms_exact_rational:
        pytest.importorskip("sympy")
    pin(orms)


@pytest.mark.parametrize("pin", pins.LN_PINS, ids=lambda f: f.__name__)
def test_ln_pins(pin):
    pin(oln)


def test_package_exports():
    for name in oracle.__all__:
        assert callable(getattr(oracle, name))


# ---------------------------------------------------------------------------
# Negative control (Aether-ML PR #18, "Testing": the large-offset test fails
# on a naive E[x^2] - E[x]^2).  The fp32 tolerance used by the GPU parity
# tests must reject a naive single-precision variance on large-offset data,
# and accept a single-precision one-pass sum that is shifted by one sample of
# the channel.  Both emulations live here, in the test, not in the oracle.

def _naive_f32_var(x):
    x = x.astype(np.float32)
    m = x.mean(axis=(0, 2), dtype=np.float32)
    m2 = (x * x).mean(axis=(0, 2), dtype=np.float32)
    return (m2 - m * m).astype(np.float64)


def _shifted_f32_var(x):
    x = x.astype(np.float32)
    shift = x[0, :, 0][None, :, None]
    d = x - shift
    s1 = d.sum(axis=(0, 2), dtype=np.float32).astype(np.float64)
    s2 = (d * d).sum(axis=(0, 2), dtype=np.float32).astype(np.float64)
    M = x.shape[0] * x.shape[2]
    return s2 / M - (s1 / M) ** 2


@pytest.mark.parametrize("mu,sigma,shape", [
    (1e4, 0.01, (16, 3, 256)),          # Aether-ML PR #18 "Testing": mean 1e4, std 0.01
    (None, 1.0, (64, 8, 1024)),         # the large-offset BN workload's law
])
def test_negative_control_naive_variance(mu, sigma, shape):
    r = np.random.default_rng(7)
    C = shape[1]
    mus = (np.full(C, mu) if mu is not None
           else r.uniform(-1000, 1000, C))
    x = (mus[None, :, None] + sigma * r.standard_normal(shape))
    x = x.astype(np.float32).astype(np.float64)   # stored values
    ref = oracle.batch_norm_forward_train(
        x, np.ones(C), np.zeros(C), np.zeros(C), np.ones(C), 0.1, 1e-5)["var"]
    naive = _naive_f32_var(x)
    assert f32_violations(naive, ref) > 0, "naive variance must fail"
    check_f32(_shifted_f32_var(x), ref, "shifted one-pass variance")
