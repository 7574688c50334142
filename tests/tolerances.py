"""Parity tolerances between the CUDA path and the float64 oracle.

fp32 outputs:  |got - ref| <= 1e-6 + 2e-5 * |ref|           (element-wise)

bf16 outputs:  |got - ref| <= 2 * ulp_bf16(max(|ref|, tau))  (element-wise)
               ulp_bf16(v) = 2 ** (floor(log2 v) - 7)
               tau = 2**-12 * RMS(ref) over the comparison group (per
               channel for BatchNorm y/dx, per tensor otherwise).

The floor tau exists because a bf16 ulp of a value that is near zero only
through cancellation is smaller than the fp32 rounding of the terms that
cancelled; without it a correct fp32-accumulating kernel would fail on
rounding alone.  ``bf16_report`` counts how many elements relied on it.
"""

import numpy as np

F32_ATOL = 1e-6
F32_RTOL = 2e-5
BF16_ULPS = 2.0
TAU_FACTOR = 2.0 ** -12


def _f64(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float64)


def f32_violations(got, ref):
    g, r = _f64(got), _f64(ref)
    assert g.shape == r.shape, f"shape {g.shape} vs {r.shape}"
    bad = ~(np.abs(g - r) <= F32_ATOL + F32_RTOL * np.abs(r))
    return int(bad.sum())


def check_f32(got, ref, name):
    g, r = _f64(got), _f64(ref)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    err = np.abs(g - r)
    bound = F32_ATOL + F32_RTOL * np.abs(r)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argmax(np.where(bad, err / bound, 0))
        raise AssertionError(
            f"{name}: {int(bad.sum())}/{g.size} outside fp32 tolerance; "
            f"worst at flat {i}: got {g.flat[i]!r} ref {r.flat[i]!r}")


def ulp_bf16(v):
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    return np.where(v > 0, np.exp2(e - 7), 0.0)


def tau_of(ref, axis=None):
    r = _f64(ref)
    return TAU_FACTOR * np.sqrt(np.mean(r * r, axis=axis, keepdims=True))


def bf16_report(got, ref, tau):
    g, r = _f64(got), _f64(ref)
    assert g.shape == r.shape, f"shape {g.shape} vs {r.shape}"
    tau = np.broadcast_to(np.asarray(tau, dtype=np.float64), r.shape)
    mag = np.maximum(np.abs(r), tau)
    bound = BF16_ULPS * ulp_bf16(mag)
    err = np.abs(g - r)
    bad = ~(err <= bound)
    return {"bad": int(bad.sum()), "tau_floor": int((np.abs(r) < tau).sum()),
            "err": err, "bound": bound, "g": g, "r": r, "badmask": bad}


# (check name, elements whose bound came from the floor tau, elements
# checked) of every bf16 comparison in this process; the test session prints
# the totals at its end.
TAU_FLOOR_LOG = []


def check_bf16(got, ref, name, tau=None):
    if tau is None:
        tau = tau_of(ref)
    rep = bf16_report(got, ref, tau)
    TAU_FLOOR_LOG.append((name, rep["tau_floor"], rep["g"].size))
    if rep["bad"]:
        bad = rep["badmask"]
        ratio = np.where(bad, rep["err"] / np.maximum(rep["bound"], 1e-300), 0)
        i = np.argmax(ratio)
        raise AssertionError(
            f"{name}: {rep['bad']}/{bad.size} outside 2 bf16 ulps; worst at "
            f"flat {i}: got {rep['g'].flat[i]!r} ref {rep['r'].flat[i]!r}")
    return rep


def check(got, ref, name, dtype, tau=None):
    """Dispatch on the output's storage dtype ("f32" or "bf16")."""
    if dtype == "f32":
        check_f32(got, ref, name)
        return None
    return check_bf16(got, ref, name, tau)
