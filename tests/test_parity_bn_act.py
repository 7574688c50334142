"""BatchNorm2d with a fused ReLU / LeakyReLU: CUDA path vs the float64 oracle.

The activation's kink turns a floating-point value into a decision (is
pre = (x - mean)*scale + beta above 0?).  The kernels decide on their fp32
pre, the oracle on its float64 pre; the inputs are therefore first moved
away from the kink: every element whose oracle pre lies within
1e-4 * (|gamma| + |beta|) of 0 is shifted to the nearest storage value at
least twice that far out on the same side, which is over a hundred times
the fp32 error of the kernels' pre.  The decision is then unique and the
comparison is the usual element-by-element one.  Exact zeros (a constant
channel with beta = 0) are decided identically on both sides and are
tested as such."""

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
ACTS = {"relu": (oracle.ACT_RELU, 0.0), "leaky_relu": (oracle.ACT_LEAKY_RELU, 0.1)}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _f64(t):
    return t.detach().cpu().double().numpy()


def _ulp(v, dtype):
    a = np.maximum(np.abs(v), 1e-30)
    if dtype == torch.bfloat16:
        return np.exp2(np.floor(np.log2(a)) - 7)
    return np.spacing(a.astype(np.float32)).astype(np.float64)


def nudge_off_kink(inp, channels=None, use_beta=True):
    """Move the elements of x (in place, storage dtype) whose oracle pre is
    within 1e-4*(|gamma|+|beta|) of 0 to at least twice that distance."""
    x = inp["x"]
    C = x.shape[1]
    chs = list(range(C)) if channels is None else list(channels)
    n = len(chs)
    bshape = (1, n) + (1,) * (x.dim() - 2)
    g = _f64(inp["gamma"][chs])
    b = _f64(inp["beta"][chs]) if use_beta else np.zeros(n)
    assert np.all(g > 0)
    delta = (1e-4 * (np.abs(g) + np.abs(b))).reshape(bshape)
    for _ in range(4):
        xs = x[:, chs]
        x64 = _f64(xs)
        f = oracle.batch_norm_forward_train(x64, g, b, np.zeros(n), np.ones(n), 0.0, inp["eps"])
        pre = f["y"]
        close = np.abs(pre) < delta
        if not close.any():
            return
        mean = f["mean"].reshape(bshape)
        scale = f["scale"].reshape(bshape)
        bb = b.reshape(bshape)
        s = np.where(pre >= 0, 1.0, -1.0)
        target = np.broadcast_to(mean + (s * 4.0 * delta - bb) / scale, x64.shape)
        new = np.where(close, target, x64)
        for _ in range(16):
            newt = torch.from_numpy(new).to(x.dtype)
            v = _f64(newt)
            short = close & (s * ((v - mean) * scale + bb) < 2.0 * delta)
            if not short.any():
                break
            new = np.where(short, v + s * _ulp(v, x.dtype), v)
        x[:, chs] = newt
    raise AssertionError("could not move x off the activation's kink")


def run_gpu(gbn, inp, act, slope, *, beta=True, x=None, dy=None):
    x = inp["x"].to(DEV) if x is None else x
    dy = inp["dy"].to(DEV) if dy is None else dy
    g = inp["gamma"].to(DEV)
    b = inp["beta"].to(DEV) if beta else None
    rm = inp["running_mean"].to(DEV)
    rv = inp["running_var"].to(DEV)
    y, stats = gbn.bn_forward_train(x, g, b, rm, rv, inp["momentum"], inp["eps"], act=act,
                                    slope=slope)
    dx, grads = gbn.bn_backward(x, dy, stats, beta=b, act=act, slope=slope)
    torch.cuda.synchronize()
    C = x.shape[1]
    s, gr = stats.cpu(), grads.cpu()
    return {"y": y.cpu(), "dx": dx.cpu(), "mean": s[:C], "var": s[C:2 * C],
            "inv_std": s[2 * C:3 * C], "scale": s[3 * C:4 * C], "running_mean": rm.cpu(),
            "running_var": rv.cpu(), "dgamma": gr[:C], "dbeta": gr[C:2 * C],
            "k1": gr[2 * C:3 * C], "k2": gr[3 * C:]}


def run_oracle(inp, act, slope, channels=None, *, beta=True):
    x, dy = inp["x"], inp["dy"]
    C = x.shape[1]
    g = inp["gamma"]
    b = inp["beta"] if beta else torch.zeros(C)
    rm, rv = inp["running_mean"], inp["running_var"]
    if channels is not None:
        idx = torch.tensor(channels)
        x, dy = x.index_select(1, idx), dy.index_select(1, idx)
        g, b, rm, rv = g[idx], b[idx], rm[idx], rv[idx]
    x, dy, g, b, rm, rv = map(_f64, (x, dy, g, b, rm, rv))
    code, _ = ACTS[act]
    f = oracle.batch_norm_act_forward_train(x, g, b, rm, rv, inp["momentum"], inp["eps"], code,
                                            slope)
    bw = oracle.batch_norm_act_backward(x, dy, g, b, inp["eps"], code, slope)
    out = dict(f)
    out.update({k: v for k, v in bw.items() if k != "pre"})
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


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
@pytest.mark.parametrize("name", ["bn_tiny_f32", "bn_offset_f32", "bn_ragged_f32"])
def test_bn_act_parity(gbn, name, act):
    case = synth.CASES[name]
    inp = synth.bn_inputs(case)
    nudge_off_kink(inp)
    slope = ACTS[act][1]
    compare(run_gpu(gbn, inp, act, slope), run_oracle(inp, act, slope), case.dtype,
            what=f"{name} {act}")


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
def test_bn_act_bf16(gbn, act):
    case = synth.BNCase("bn_act_bf16", (16, 96, 28, 28), "bf16", mu_range=(-10.0, 10.0),
                        sigma_range=(0.1, 4.0), seed=4201)
    inp = synth.bn_inputs(case)
    nudge_off_kink(inp)
    slope = ACTS[act][1]
    compare(run_gpu(gbn, inp, act, slope), run_oracle(inp, act, slope), "bf16",
            what=f"bf16 {act}")


def test_bn_relu_full_size_sampled_channels(gbn):
    """The bf16 [128,256,56,56] workload with ReLU, 10 channels checked
    element by element against the oracle."""
    case = synth.CASES["bn_offset_bf16"]
    inp = synth.bn_inputs(case)
    C = inp["x"].shape[1]
    channels = sorted({0, C - 1} | set(range(13, C, 31)))[:10]
    nudge_off_kink(inp, channels)
    got = run_gpu(gbn, inp, "relu", 0.0)
    compare(got, run_oracle(inp, "relu", 0.0, channels), "bf16", channels, what="full relu")


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
def test_bn_act_two_launch_path(gbn, act):
    """Views offset by one element take the two-launch kernels (vector
    width 1); they match the oracle like the single-launch kernel."""
    inp = synth.bn_inputs(synth.CASES["bn_ragged_f32"])
    nudge_off_kink(inp)
    slope = ACTS[act][1]

    def misaligned(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
        buf[1:] = t.to(DEV).reshape(-1)
        return buf[1:].view(t.shape)

    xm, dym = misaligned(inp["x"]), misaligned(inp["dy"])
    assert xm.data_ptr() % 16 != 0
    got = run_gpu(gbn, inp, act, slope, x=xm, dy=dym)
    compare(got, run_oracle(inp, act, slope), "f32", what=f"two-launch {act}")


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
def test_bn_act_without_beta(gbn, act):
    inp = synth.bn_inputs(synth.CASES["bn_ragged_f32"])
    nudge_off_kink(inp, use_beta=False)
    slope = ACTS[act][1]
    compare(run_gpu(gbn, inp, act, slope, beta=False),
            run_oracle(inp, act, slope, beta=False), "f32", what=f"no beta {act}")


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
def test_bn_act_zero_channel_at_kink(gbn, act):
    """An all-zero channel with beta = 0 has pre = 0 exactly on both sides:
    ReLU gives y = 0 and gates dy to 0, LeakyReLU gates it by the slope."""
    case = synth.BNCase("act_zero", (4, 3, 6, 6), "f32")
    inp = synth.bn_inputs(case)
    nudge_off_kink(inp, [0, 2])
    inp["x"][:, 1] = 0.0
    inp["beta"][1] = 0.0
    slope = ACTS[act][1]
    got = run_gpu(gbn, inp, act, slope)
    ref = run_oracle(inp, act, slope)
    compare(got, ref, "f32", what=f"zero channel {act}")
    assert torch.all(got["y"][:, 1] == 0)
    expect_dbeta = 0.0 if act == "relu" else slope * float(inp["dy"][:, 1].double().sum())
    assert abs(float(got["dbeta"][1]) - expect_dbeta) <= 1e-5 * (1 + abs(expect_dbeta))


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
def test_bn_act_bit_deterministic_and_in_place(gbn, act):
    inp = synth.bn_inputs(synth.CASES["bn_offset_f32"])
    slope = ACTS[act][1]
    a = run_gpu(gbn, inp, act, slope)
    b = run_gpu(gbn, inp, act, slope)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    x = inp["x"].to(DEV)
    g, be = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    _, stats = gbn.bn_forward_train(x, g, be, None, None, 0.1, inp["eps"], act=act, slope=slope)
    xi = x.clone()
    gbn.bn_forward_train(xi, g, be, None, None, 0.1, inp["eps"], y=xi, act=act, slope=slope)
    assert torch.equal(xi.cpu(), a["y"])
    dyi = inp["dy"].to(DEV)
    gbn.bn_backward(x, dyi, stats, dx=dyi, beta=be, act=act, slope=slope)
    assert torch.equal(dyi.cpu(), a["dx"])


def test_bn_act_none_matches_plain(gbn):
    """Through the _act entry points, GBN_ACT_NONE is the plain BatchNorm
    bit for bit."""
    import ctypes
    from bwd_bn_pass_gb300 import gbnorm as G
    inp = synth.bn_inputs(synth.CASES["bn_ragged_f32"])
    x, dy = inp["x"].to(DEV), inp["dy"].to(DEV)
    g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    y0, s0 = gbn.bn_forward_train(x, g, b, None, None, 0.1, inp["eps"])
    dx0, gr0 = gbn.bn_backward(x, dy, s0)
    B, C, HW = x.shape[0], x.shape[1], x[0, 0].numel()
    ws = gbn.bn_workspace(x)
    y1, s1 = torch.empty_like(x), gbn.bn_stats_tensor(C, x.device)
    dx1, gr1 = torch.empty_like(x), torch.empty(4 * C, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    nb = ws.numel() * ws.element_size()
    L = G.lib()
    assert L.gbn_bn_forward_train_act(p(x), 0, B, C, HW, p(g), p(b), None, None, 0.1,
                                      inp["eps"], 0, 0.0, p(y1), p(s1), p(ws), nb, st) == 0
    assert L.gbn_bn_backward_act(p(x), p(dy), 0, B, C, HW, p(s1), p(b), 0, 0.0, p(dx1),
                                 p(gr1), p(ws), nb, st) == 0
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(s0, s1)
    assert torch.equal(dx0, dx1) and torch.equal(gr0, gr1)


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
def test_bn_apply_act(gbn, act):
    case = synth.CASES["bn_ragged_f32"]
    inp = synth.bn_inputs(case)
    slope = ACTS[act][1]
    x = inp["x"].to(DEV)
    g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    y, stats = gbn.bn_forward_train(x, g, b, None, None, 0.1, 1e-5, act=act, slope=slope)
    y2 = gbn.bn_apply(x, b, stats=stats, act=act, slope=slope)
    assert torch.equal(y, y2), "apply from stats must equal the training apply"
    r = np.random.default_rng(5)
    C = x.shape[1]
    rmean = torch.tensor(r.uniform(-1000, 1000, C), dtype=torch.float32)
    rvar = torch.tensor(r.uniform(0.5, 2.0, C), dtype=torch.float32)
    scale = (inp["gamma"].double() / torch.sqrt(rvar.double() + 1e-5)).float()
    yi = gbn.bn_apply(x, b, mean=rmean.to(DEV), scale=scale.to(DEV), act=act, slope=slope)
    pre = oracle.batch_norm_apply(_f64(inp["x"]), _f64(rmean), _f64(scale), _f64(inp["beta"]))
    ref = oracle.activation(pre, ACTS[act][0], slope)
    # y is continuous at the kink, so no decision needs moving off it here.
    tol.check_f32(yi, ref, f"inference apply {act}")


def test_bn_act_rejects_bad_arguments(gbn):
    x = torch.randn(2, 3, 4, device=DEV)
    with pytest.raises(ValueError):
        gbn.bn_forward_train(x, act="gelu")
    with pytest.raises(RuntimeError):
        gbn.bn_forward_train(x, act="leaky_relu", slope=float("nan"))
