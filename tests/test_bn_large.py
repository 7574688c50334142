"""BatchNorm beyond 32-bit element offsets, and the 64-bit offset form of the
two-launch kernels.

* A bf16 [512, 64, 256, 256] tensor holds 2^31 elements (4 GiB per tensor),
  so offsets past 2^31 - 1 are exercised in both BatchNorm paths (the
  persistent kernel, which takes this size by default, and the two-launch
  kernels).  The oracle checks three channels element by element; the
  statistics and dbeta of every channel are checked against their
  definitions (float64 mean, biased variance and sum over the channel,
  computed by torch from the same data).  The inputs follow the bf16
  BatchNorm workload's law (mu_c ~ U(-100, 100), sigma_c ~ U(0.01, 10)),
  drawn on the device from a seeded generator because 2^31 host-side draws
  would take minutes.
* The two-launch kernels switch from 32-bit to 64-bit vector offsets only
  past 2^32 vectors (64 GiB of bf16).  A test hook forces the 64-bit form on
  small tensors; it must give exactly the bits of the 32-bit form, and the
  oracle's results."""

import numpy as np
import pytest
import torch

import oracle
from bwd_bn_pass_gb300 import synth

from . import tolerances as tol

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _f64(t):
    return t.detach().cpu().double().numpy()


def _bn_law_on_device(shape, seed):
    """x = mu_c + sigma_c * N(0, 1) and dy ~ N(0, 1), both rounded to bf16;
    gamma ~ U(0.5, 1.5), beta ~ N(0, 0.1) (fp32)."""
    B, C = shape[:2]
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    mu = torch.rand(C, 1, 1, device=DEV, generator=gen) * 200.0 - 100.0
    sigma = torch.rand(C, 1, 1, device=DEV, generator=gen) * 9.99 + 0.01
    gamma = torch.rand(C, device=DEV, generator=gen) + 0.5
    beta = torch.randn(C, device=DEV, generator=gen) * 0.1
    x = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    dy = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    step = 32
    for b0 in range(0, B, step):
        n = min(step, B - b0)
        z = torch.randn((n,) + tuple(shape[1:]), device=DEV, generator=gen)
        x[b0:b0 + n] = (mu + sigma * z).to(torch.bfloat16)
        dy[b0:b0 + n] = torch.randn((n,) + tuple(shape[1:]), device=DEV,
                                    generator=gen).to(torch.bfloat16)
        del z
    return x, dy, gamma, beta


def test_bn_beyond_int32_elements(gbn):
    shape = (512, 64, 256, 256)  # 2^31 elements
    B, C = shape[:2]
    eps, momentum = 1e-5, 0.1
    x, dy, gamma, beta = _bn_law_on_device(shape, seed=20241207)
    assert x.numel() == 2 ** 31

    # definitions over every channel, in float64 from the same data
    mean64 = torch.empty(C, dtype=torch.float64)
    var64 = torch.empty(C, dtype=torch.float64)
    dbeta64 = torch.empty(C, dtype=torch.float64)
    for c in range(C):
        xc = x[:, c].double()
        mean64[c] = xc.mean().cpu()
        var64[c] = ((xc - xc.mean()) ** 2).mean().cpu()
        dbeta64[c] = dy[:, c].double().sum().cpu()
        del xc

    channels = [0, 31, C - 1]
    xs, dys = _f64(x[:, channels]), _f64(dy[:, channels])
    g, b = _f64(gamma[channels]), _f64(beta[channels])
    ref = oracle.batch_norm_forward_train(xs, g, b, np.zeros(len(channels)),
                                          np.ones(len(channels)), momentum, eps)
    ref.update(oracle.batch_norm_backward(xs, dys, g, eps))
    del xs, dys

    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    for path, threshold in (("persistent", None), ("two-launch", 1 << 62)):
        prev = gbn.bn_set_persistent_min_bytes(threshold) if threshold is not None else None
        try:
            rm = torch.zeros(C, device=DEV)
            rv = torch.ones(C, device=DEV)
            _, stats = gbn.bn_forward_train(x, gamma, beta, rm, rv, momentum, eps, y=y)
            _, grads = gbn.bn_backward(x, dy, stats, dx=dx)
            torch.cuda.synchronize()
        finally:
            if prev is not None:
                gbn.bn_set_persistent_min_bytes(prev)
        s, gr = stats.cpu(), grads.cpu()
        what = f"2^31 elements, {path}"
        tol.check_f32(s[:C], mean64.numpy(), f"{what} mean (all channels)")
        tol.check_f32(s[C:2 * C], var64.numpy(), f"{what} var (all channels)")
        tol.check_f32(gr[C:2 * C], dbeta64.numpy(), f"{what} dbeta (all channels)")
        got = {"mean": s[:C], "var": s[C:2 * C], "inv_std": s[2 * C:3 * C],
               "scale": s[3 * C:4 * C], "running_mean": rm.cpu(), "running_var": rv.cpu(),
               "dgamma": gr[:C], "dbeta": gr[C:2 * C], "k1": gr[2 * C:3 * C],
               "k2": gr[3 * C:]}
        for k, v in got.items():
            tol.check_f32(v[channels], ref[k], f"{what} {k}")
        for k, t in (("y", y), ("dx", dx)):
            g_ = t[:, channels].cpu().reshape(B, len(channels), -1)
            r = ref[k].reshape(B, len(channels), -1)
            tau = tol.tau_of(r, axis=(0, 2))
            tol.check_bf16(g_, r, f"{what} {k}", tau)


WIDE_CASES = [
    ("bn_ragged_f32", None),                                   # fp32, 40-wide planes
    ("wide_bf16_vec4", synth.BNCase("wide_bf16_vec4", (16, 48, 14, 14), "bf16",
                                    mu_range=(-100.0, 100.0), seed=1301)),
    ("wide_bf16_vec8", synth.BNCase("wide_bf16_vec8", (8, 16, 28, 28), "bf16", seed=1303)),
    ("wide_bf16_vec1", synth.BNCase("wide_bf16_vec1", (5, 19, 7, 9), "bf16", seed=1305)),
]


@pytest.mark.parametrize("name,case", WIDE_CASES, ids=[c[0] for c in WIDE_CASES])
@pytest.mark.parametrize("act", [None, "relu"])
def test_bn_wide_offsets_match_narrow(gbn, name, case, act):
    case = case if case is not None else synth.CASES[name]
    inp = synth.bn_inputs(case)
    x, dy = inp["x"].to(DEV), inp["dy"].to(DEV)
    g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    prev_t = gbn.bn_set_persistent_min_bytes(1 << 62)  # the two-launch kernels
    outs = []
    try:
        for wide in (False, True):
            prev_w = gbn.bn_set_wide_offsets(wide)
            try:
                y, stats = gbn.bn_forward_train(x, g, b, None, None, 0.1, 1e-5, act=act)
                dx, grads = gbn.bn_backward(x, dy, stats, beta=b, act=act)
                torch.cuda.synchronize()
            finally:
                gbn.bn_set_wide_offsets(prev_w)
            outs.append((y.cpu(), stats.cpu(), dx.cpu(), grads.cpu()))
    finally:
        gbn.bn_set_persistent_min_bytes(prev_t)
    for a, w, k in zip(outs[0], outs[1], ("y", "stats", "dx", "grads")):
        assert torch.equal(a, w), f"{name}: {k} differs between 32- and 64-bit offsets"
    if act is None:
        C = x.shape[1]
        xs, dys = _f64(inp["x"]), _f64(inp["dy"])
        ref = oracle.batch_norm_forward_train(xs, _f64(inp["gamma"]), _f64(inp["beta"]),
                                              np.zeros(C), np.ones(C), 0.1, 1e-5)
        ref.update(oracle.batch_norm_backward(xs, dys, _f64(inp["gamma"]), 1e-5))
        y, stats, dx, grads = outs[1]
        tol.check(y.double().numpy(), ref["y"], f"{name} y (64-bit)", case.dtype,
                  tau=tol.tau_of(ref["y"].reshape(x.shape[0], C, -1), axis=(0, 2))
                  .reshape(1, C, 1, 1) if case.dtype == "bf16" else None)
        tol.check_f32(grads[C:2 * C], ref["dbeta"], f"{name} dbeta (64-bit)")
        tol.check_f32(grads[:C], ref["dgamma"], f"{name} dgamma (64-bit)")
