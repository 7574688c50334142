"""BatchNorm2d training forward/backward: CUDA path vs the float64 oracle.

Element-by-element on the fp32 workloads ([8,4,8,8], [256,32,32,32] with
|mean| up to 1000, ragged [3,37,41,40]); on sampled channels for the full
bf16 [128,256,56,56] workload in the same launch configuration bench.py
times; plus edge cases, bit-determinism and the phase entry points."""

import numpy as np
import pytest
import torch

import oracle
from bwd_bn_pass_gb300 import synth

from . import tolerances as tol

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["auto", "persistent", "two_launch"])
def _bn_path(request, gbn):
    """Every test runs three times: with the library's defaults (the
    single-launch small-channel kernels for channels of at most 2048
    elements, the two-launch kernels, the persistent kernel from 128 MiB of
    input); with the persistent kernel's threshold at 0, so that it takes
    every eligible shape, small ones included; and with the small-channel
    kernels off and the threshold out of reach, so that the two-launch
    kernels take every shape."""
    if request.param == "persistent":
        prev = gbn.bn_set_persistent_min_bytes(0)
        yield
        gbn.bn_set_persistent_min_bytes(prev)
    elif request.param == "two_launch":
        prev = gbn.bn_set_persistent_min_bytes(1 << 62)
        prev_small = gbn.bn_set_small_max_elems(0)
        yield
        gbn.bn_set_persistent_min_bytes(prev)
        gbn.bn_set_small_max_elems(prev_small)
    else:
        yield


DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _f64(t):
    return t.detach().cpu().double().numpy()


def run_gpu(gbn, inp, *, gamma=True, beta=True):
    x = inp["x"].to(DEV)
    dy = inp["dy"].to(DEV)
    g = inp["gamma"].to(DEV) if gamma else None
    b = inp["beta"].to(DEV) if beta else None
    rm = inp["running_mean"].to(DEV)
    rv = inp["running_var"].to(DEV)
    y, stats = gbn.bn_forward_train(x, g, b, rm, rv, inp["momentum"], inp["eps"])
    dx, grads = gbn.bn_backward(x, dy, stats)
    torch.cuda.synchronize()
    C = x.shape[1]
    s, gr = stats.cpu(), grads.cpu()
    return {"y": y.cpu(), "dx": dx.cpu(), "mean": s[:C], "var": s[C:2 * C],
            "inv_std": s[2 * C:3 * C], "scale": s[3 * C:4 * C], "running_mean": rm.cpu(),
            "running_var": rv.cpu(), "dgamma": gr[:C], "dbeta": gr[C:2 * C],
            "k1": gr[2 * C:3 * C], "k2": gr[3 * C:]}


def run_oracle(inp, channels=None, *, gamma=True, beta=True):
    x, dy = inp["x"], inp["dy"]
    C = x.shape[1]
    g = inp["gamma"] if gamma else torch.ones(C)
    b = inp["beta"] if beta else torch.zeros(C)
    rm, rv = inp["running_mean"], inp["running_var"]
    if channels is not None:
        idx = torch.tensor(channels)
        x, dy = x.index_select(1, idx), dy.index_select(1, idx)
        g, b, rm, rv = g[idx], b[idx], rm[idx], rv[idx]
    x, dy, g, b, rm, rv = map(_f64, (x, dy, g, b, rm, rv))
    f = oracle.batch_norm_forward_train(x, g, b, rm, rv, inp["momentum"], inp["eps"])
    bw = oracle.batch_norm_backward(x, dy, g, inp["eps"])
    out = dict(f)
    out.update(bw)
    return out


def compare(got, ref, dtype, channels=None, what=""):
    sel = (lambda t: t) if channels is None else (lambda t: t[:, channels])
    vsel = (lambda t: t) if channels is None else (lambda t: t[channels])
    for k in ("mean", "var", "inv_std", "scale", "running_mean", "running_var", "dgamma",
              "dbeta", "k1", "k2"):
        tol.check_f32(vsel(got[k]), ref[k], f"{what} {k}")
    for k in ("y", "dx"):
        g = sel(got[k])
        r = ref[k]
        if dtype == "f32":
            tol.check_f32(g, r, f"{what} {k}")
        else:
            B, C = r.shape[:2]
            tau = tol.tau_of(r.reshape(B, C, -1), axis=(0, 2))
            tol.check_bf16(g.reshape(B, C, -1), r.reshape(B, C, -1), f"{what} {k}", tau)


@pytest.mark.parametrize("name", ["bn_tiny_f32", "bn_offset_f32", "bn_ragged_f32"])
def test_bn_parity_full(gbn, name):
    case = synth.CASES[name]
    inp = synth.bn_inputs(case)
    compare(run_gpu(gbn, inp), run_oracle(inp), case.dtype, what=name)


def test_bn_offset_bf16_full_size_all_channels(gbn):
    """The bf16 [128,256,56,56] workload at full size, in the launch
    configuration bench.py times: every channel element by element against
    the oracle (run 32 channels at a time to bound host memory)."""
    case = synth.CASES["bn_offset_bf16"]
    inp = synth.bn_inputs(case)
    got = run_gpu(gbn, inp)
    C = inp["x"].shape[1]
    for c0 in range(0, C, 32):
        channels = list(range(c0, min(C, c0 + 32)))
        ref = run_oracle(inp, channels)
        compare(got, ref, "bf16", channels, what=f"bn_offset_bf16 channels {c0}..")
    # property over every channel: sum_{b,hw} dx ~ 0 relative to sum |dx|
    x = inp["x"]
    dx = got["dx"].float().reshape(x.shape[0], C, -1)
    s = dx.double().sum(dim=(0, 2))
    a = dx.double().abs().sum(dim=(0, 2))
    assert torch.all(s.abs() <= 2e-3 * a + 1e-6), "sum dx per channel not ~0"


def test_bn_offset_bf16_full_size_bit_deterministic(gbn):
    """Two forward + backward runs of the full bf16 [128,256,56,56] workload
    (the single-launch persistent kernel) give identical bits."""
    inp = synth.bn_inputs(synth.CASES["bn_offset_bf16"])
    a = run_gpu(gbn, inp)
    b = run_gpu(gbn, inp)
    for k in a:
        assert torch.equal(a[k], b[k]), f"{k} differs between two runs"


TMEM_CASES = [
    synth.CASES["bn_offset_bf16"],
    synth.CASES["bn_offset_f32"],
    synth.BNCase("segs_bf16", (16, 2048, 8, 8), "bf16", mu_range=(-100, 100),
                 sigma_range=(0.01, 10), seed=91),
    synth.BNCase("mid_bf16", (64, 96, 28, 28), "bf16", mu_range=(-100, 100),
                 sigma_range=(0.01, 10), seed=92),
]


@pytest.mark.parametrize("case", TMEM_CASES, ids=lambda c: c.name)
def test_bn_persistent_tmem_bit_identical(gbn, case):
    """The persistent kernel with and without its tensor-memory tier (five
    stages per SM kept in TMEM between the passes) and its end-of-pass work
    stealing gives the same bits: full bf16 [128,256,56,56] (where stealing
    is used), fp32 [256,32,32,32], a range of 16 one-stage channel segments
    per CTA ([16,2048,8,8]) and a short range ([64,96,28,28]).  Runs on the
    persistent-everywhere setting only."""
    if gbn.bn_persistent_min_bytes() != 0:
        pytest.skip("checked once, with the persistent kernel taking every shape")
    inp = synth.bn_inputs(case)
    prev = gbn.bn_set_persistent_tmem(False)
    prev_s = gbn.bn_set_persistent_steal(False)
    try:
        plain = run_gpu(gbn, inp)
        gbn.bn_set_persistent_tmem(True)
        tmem = run_gpu(gbn, inp)
    finally:
        gbn.bn_set_persistent_tmem(prev)
        gbn.bn_set_persistent_steal(prev_s)
    full = run_gpu(gbn, inp)  # the defaults: TMEM tier and work stealing
    for k in full:
        assert torch.equal(tmem[k], plain[k]), f"{k} differs with the TMEM tier"
        assert torch.equal(full[k], plain[k]), f"{k} differs with work stealing"


@pytest.mark.parametrize("name", ["bn_offset_f32", "bn_ragged_f32"])
def test_bn_bit_deterministic(gbn, name):
    inp = synth.bn_inputs(synth.CASES[name])
    a = run_gpu(gbn, inp)
    b = run_gpu(gbn, inp)
    for k in a:
        assert torch.equal(a[k], b[k]), f"{k} differs between two runs"


def test_bn_many_channels(gbn):
    """3000 channels of 64 elements per plane: every CTA of the single-launch
    kernel spans ~20 channel segments (one per-segment reduction, partial and
    finalize each)."""
    case = synth.BNCase("bn_wide_f32", (64, 3000, 8, 8), "f32", mu_range=(-50.0, 50.0),
                        seed=97)
    inp = synth.bn_inputs(case)
    compare(run_gpu(gbn, inp), run_oracle(inp), case.dtype, what="bn 3000 channels")


def test_bn_bf16_bit_deterministic(gbn):
    case = synth.BNCase("det_bf16", (32, 64, 28, 28), "bf16", mu_range=(-100, 100),
                        sigma_range=(0.01, 10), seed=99)
    inp = synth.bn_inputs(case)
    a, b = run_gpu(gbn, inp), run_gpu(gbn, inp)
    for k in a:
        assert torch.equal(a[k], b[k]), f"{k} differs between two runs"


EDGE = [
    synth.BNCase("c1", (7, 1, 5, 9), "f32", mu_range=(-50, 50)),
    synth.BNCase("hw1", (64, 5, 1, 1), "f32", mu_range=(-3, 3)),
    synth.BNCase("m2", (2, 3, 1, 1), "f32"),
    synth.BNCase("odd_hw", (5, 6, 7, 7), "f32", mu_range=(-100, 100)),
    synth.BNCase("odd_hw_bf16", (9, 6, 7, 7), "bf16", mu_range=(-10, 10),
                 sigma_range=(0.1, 3)),
    synth.BNCase("hw196_bf16", (4, 16, 14, 14), "bf16", sigma_range=(0.5, 2)),
    synth.BNCase("b1_big_plane", (1, 3, 160, 160), "f32", mu_range=(-1000, 1000)),
    synth.BNCase("many_c", (2, 1500, 3, 3), "f32", mu_range=(-5, 5)),
    synth.BNCase("wide_bf16", (3, 37, 41, 40), "bf16", mu_range=(-100, 100),
                 sigma_range=(0.01, 10)),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: c.name)
def test_bn_edge_shapes(gbn, case):
    inp = synth.bn_inputs(case)
    compare(run_gpu(gbn, inp), run_oracle(inp), case.dtype, what=case.name)


def test_bn_no_affine(gbn):
    inp = synth.bn_inputs(synth.CASES["bn_ragged_f32"])
    got = run_gpu(gbn, inp, gamma=False, beta=False)
    compare(got, run_oracle(inp, gamma=False, beta=False), "f32", what="no affine")


def test_bn_constant_channel(gbn):
    case = synth.BNCase("const", (4, 3, 6, 6), "f32")
    inp = synth.bn_inputs(case)
    inp["x"][:, 1] = 123.5
    compare(run_gpu(gbn, inp), run_oracle(inp), "f32", what="constant channel")


def test_bn_misaligned_views(gbn):
    """Device views offset by one element: the vector width falls back to 1."""
    inp = synth.bn_inputs(synth.CASES["bn_ragged_f32"])
    ref = run_oracle(inp)

    def misaligned(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
        buf[1:] = t.to(DEV).reshape(-1)
        return buf[1:].view(t.shape)

    xm, dym = misaligned(inp["x"]), misaligned(inp["dy"])
    assert xm.data_ptr() % 16 != 0
    rm, rv = inp["running_mean"].to(DEV), inp["running_var"].to(DEV)
    y, stats = gbn.bn_forward_train(xm, inp["gamma"].to(DEV), inp["beta"].to(DEV), rm, rv,
                                    inp["momentum"], inp["eps"])
    dx, grads = gbn.bn_backward(xm, dym, stats)
    C = xm.shape[1]
    tol.check_f32(y, ref["y"], "misaligned y")
    tol.check_f32(dx, ref["dx"], "misaligned dx")
    tol.check_f32(grads[:C], ref["dgamma"], "misaligned dgamma")
    tol.check_f32(stats[C:2 * C], ref["var"], "misaligned var")


def _run_phases(gbn, inp):
    x, dy = inp["x"].to(DEV), inp["dy"].to(DEV)
    g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    rm, rv = inp["running_mean"].to(DEV), inp["running_var"].to(DEV)
    ws = gbn.bn_workspace(x)
    y = torch.empty_like(x)
    stats = gbn.bn_stats_tensor(x.shape[1], x.device)
    gbn.bn_stats(x, ws)
    gbn.bn_finalize_apply(x, g, b, rm, rv, inp["momentum"], inp["eps"], y, stats, ws)
    dx = torch.empty_like(x)
    grads = torch.empty(4 * x.shape[1], dtype=torch.float32, device=DEV)
    gbn.bn_grad_sums(x, dy, stats, ws)
    gbn.bn_finalize_dx(x, dy, stats, dx, grads, ws)
    torch.cuda.synchronize()
    C = x.shape[1]
    s, gr = stats.cpu(), grads.cpu()
    return {"y": y.cpu(), "dx": dx.cpu(), "mean": s[:C], "var": s[C:2 * C],
            "inv_std": s[2 * C:3 * C], "scale": s[3 * C:4 * C], "running_mean": rm.cpu(),
            "running_var": rv.cpu(), "dgamma": gr[:C], "dbeta": gr[C:2 * C],
            "k1": gr[2 * C:3 * C], "k2": gr[3 * C:]}


@pytest.mark.parametrize("name", ["bn_offset_f32", "bn_ragged_f32"])
def test_bn_phase_entry_points(gbn, name):
    """The four phase entry points chained by hand (the two-launch kernels)
    match the oracle and are bit-deterministic.  The composite calls may take
    the single-launch persistent kernel, whose per-CTA split of the channel
    sums differs, so the two paths agree within the parity tolerance (each is
    checked against the oracle) rather than bit for bit."""
    case = synth.CASES[name]
    inp = synth.bn_inputs(case)
    a = _run_phases(gbn, inp)
    compare(a, run_oracle(inp), case.dtype, what=f"{name} phases")
    b = _run_phases(gbn, inp)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    compare(run_gpu(gbn, inp), run_oracle(inp), case.dtype, what=f"{name} composite")


def _constant_dy_inputs(dtype, centred):
    """dy constant per channel (the gradient of a plain sum of the outputs):
    sum dy*(x - mean) is then exactly 0, so dgamma and k1 are 0 and only the
    fp32 tolerance's absolute floor remains.  The constants are exact in
    bf16; 0.30078125 has a full 8-bit significand.  Channels with a large
    offset have few significant bits in x - shift; zero-mean channels span
    many binades, where a channel sum of x - shift rounded in plain fp32
    would miss that floor."""
    mu = None if centred else ((-1000.0, 1000.0) if dtype == "f32" else (-100.0, 100.0))
    sigma = None if dtype == "f32" else (0.01, 10.0)
    case = synth.BNCase(f"const_dy_{dtype}", (64, 8, 56, 56), dtype, mu_range=mu,
                        sigma_range=sigma, seed=881 + 2 * centred + (dtype == "bf16"))
    inp = synth.bn_inputs(case)
    c = torch.tensor([1.0, 0.30078125, -2.5, 7.0, -0.0078125, 1.0, 3.0, -1.0])
    inp["dy"] = c.view(1, 8, 1, 1).expand(inp["x"].shape).to(inp["x"].dtype).contiguous()
    return case, inp


@pytest.mark.parametrize("centred", [False, True], ids=["offset", "centred"])
@pytest.mark.parametrize("path", ["composite", "phases", "misaligned"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bn_constant_dy_cancels(gbn, dtype, path, centred):
    """The channel sums cancel to the last bit: dgamma, dbeta, k1, k2 within
    the fp32 tolerance of the oracle (dgamma = 0 exactly there), on the
    single-launch kernel, the two-launch kernels and their scalar form.  dx
    is dy*scale + k2 plus rounding: within a few fp32 ulps of dy*scale."""
    case, inp = _constant_dy_inputs(dtype, centred)
    if path == "composite":
        got = run_gpu(gbn, inp)
    elif path == "phases":
        got = _run_phases(gbn, inp)
    else:
        def misaligned(t):
            buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
            buf[1:] = t.to(DEV).reshape(-1)
            return buf[1:].view(t.shape)
        xm, dym = misaligned(inp["x"]), misaligned(inp["dy"])
        y, stats = gbn.bn_forward_train(xm, inp["gamma"].to(DEV), inp["beta"].to(DEV), None,
                                        None, inp["momentum"], inp["eps"])
        dx, grads = gbn.bn_backward(xm, dym, stats)
        C = xm.shape[1]
        gr = grads.cpu()
        got = {"dx": dx.cpu(), "dgamma": gr[:C], "dbeta": gr[C:2 * C], "k1": gr[2 * C:3 * C],
               "k2": gr[3 * C:]}
    ref = run_oracle(inp)
    assert np.max(np.abs(ref["dgamma"])) < 1e-7   # 0 up to the oracle's own float64 rounding
    for k in ("dgamma", "dbeta", "k1", "k2"):
        tol.check_f32(got[k], ref[k], f"constant dy {dtype} {path} {k}")
    C = inp["x"].shape[1]
    term = np.abs(_f64(inp["dy"][0, :, 0, 0]) * ref["scale"]).reshape(1, C, 1, 1)
    err = np.abs(_f64(got["dx"]) - ref["dx"])
    assert np.all(err <= 2.0 ** -20 * term + 1e-30), f"dx off by {err.max()}"


def test_bn_apply_modes(gbn):
    case = synth.CASES["bn_ragged_f32"]
    inp = synth.bn_inputs(case)
    x = inp["x"].to(DEV)
    g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    y, stats = gbn.bn_forward_train(x, g, b, None, None, 0.1, 1e-5)
    y2 = gbn.bn_apply(x, b, stats=stats)
    assert torch.equal(y, y2), "apply from stats must equal the training apply"
    # inference: running stats -> (mean, scale)
    r = np.random.default_rng(3)
    C = x.shape[1]
    rmean = torch.tensor(r.uniform(-1000, 1000, C), dtype=torch.float32)
    rvar = torch.tensor(r.uniform(0.5, 2.0, C), dtype=torch.float32)
    scale = (inp["gamma"].double() / torch.sqrt(rvar.double() + 1e-5)).float()
    yi = gbn.bn_apply(x, b, mean=rmean.to(DEV), scale=scale.to(DEV))
    ref = oracle.batch_norm_apply(_f64(inp["x"]), _f64(rmean), _f64(scale), _f64(inp["beta"]))
    tol.check_f32(yi, ref, "inference apply")


def test_bn_in_place(gbn):
    inp = synth.bn_inputs(synth.CASES["bn_ragged_f32"])
    ref = run_gpu(gbn, inp)
    x = inp["x"].to(DEV)
    dy = inp["dy"].to(DEV)
    y, stats = gbn.bn_forward_train(x.clone(), inp["gamma"].to(DEV), inp["beta"].to(DEV),
                                    None, None, 0.1, 1e-5)
    xi = x.clone()
    gbn.bn_forward_train(xi, inp["gamma"].to(DEV), inp["beta"].to(DEV), None, None, 0.1,
                         1e-5, y=xi)
    assert torch.equal(xi.cpu(), ref["y"])
    dyi = dy.clone()
    gbn.bn_backward(x, dyi, stats, dx=dyi)
    assert torch.equal(dyi.cpu(), ref["dx"])


def test_bn_rejects_non_fp32_running_stats(gbn):
    x = torch.randn(4, 3, 5, device=DEV)
    rm = torch.zeros(3, dtype=torch.float64, device=DEV)
    rv = torch.ones(3, dtype=torch.float64, device=DEV)
    with pytest.raises(TypeError):
        gbn.bn_forward_train(x, None, None, rm, rv)


def test_bn_running_stats_ema_over_steps(gbn):
    case = synth.CASES["bn_tiny_f32"]
    inp = synth.bn_inputs(case)
    x = inp["x"].to(DEV)
    rm = torch.zeros(4, device=DEV)
    rv = torch.ones(4, device=DEV)
    rm_o, rv_o = np.zeros(4), np.ones(4)
    for _ in range(5):
        gbn.bn_forward_train(x, None, None, rm, rv, 0.1, 1e-5)
        f = oracle.batch_norm_forward_train(_f64(inp["x"]), np.ones(4), np.zeros(4), rm_o,
                                            rv_o, 0.1, 1e-5)
        rm_o, rv_o = f["running_mean"], f["running_var"]
    tol.check_f32(rm, rm_o, "running_mean after 5 steps")
    tol.check_f32(rv, rv_o, "running_var after 5 steps")


def test_device_status_clean(gbn):
    torch.cuda.synchronize()
    assert gbn.get_device_status() == 0
