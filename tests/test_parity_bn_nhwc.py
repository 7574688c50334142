"""Channels-last (NHWC) BatchNorm2d: CUDA path vs the float64 oracle.

The inputs are the NCHW workloads' seeded tensors permuted to [N, H, W, C]
(contiguous), so the channel statistics are the same as in the NCHW tests;
the oracle is the channels-last wrapper of the pinned NCHW oracle.  Covers
every vector width (C divisible by 8, 4, 2 or odd, and a misaligned view),
narrow and wide C, large offsets, the fused activations, a constant dy, the
[128, 56, 56, 256] bf16 workload on sampled channels, and bit-determinism."""

import numpy as np
import pytest
import torch

import oracle
from bwd_bn_pass_gb300 import synth

from . import tolerances as tol
from .test_parity_bn_act import nudge_off_kink

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ACTS = {None: (oracle.ACT_NONE, 0.0), "relu": (oracle.ACT_RELU, 0.0),
        "leaky_relu": (oracle.ACT_LEAKY_RELU, 0.1)}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _f64(t):
    return t.detach().cpu().double().numpy()


def _nhwc(t):
    return t.permute(0, 2, 3, 1).contiguous()


def nhwc_inputs(case, act=None):
    """The NCHW case's tensors (moved off the activation's kink when act is
    set), then x and dy permuted to channels-last."""
    inp = synth.bn_inputs(case)
    if act is not None:
        nudge_off_kink(inp)
    inp["x"] = _nhwc(inp["x"])
    inp["dy"] = _nhwc(inp["dy"])
    return inp


def run_gpu(gbn, inp, act=None, *, x=None, dy=None, beta=True):
    x = inp["x"].to(DEV) if x is None else x
    dy = inp["dy"].to(DEV) if dy is None else dy
    g = inp["gamma"].to(DEV)
    b = inp["beta"].to(DEV) if beta else None
    rm, rv = inp["running_mean"].to(DEV), inp["running_var"].to(DEV)
    slope = ACTS[act][1]
    y, stats = gbn.bn_nhwc_forward_train(x, g, b, rm, rv, inp["momentum"], inp["eps"], act=act,
                                         slope=slope)
    dx, grads = gbn.bn_nhwc_backward(x, dy, stats, beta=b, act=act, slope=slope)
    torch.cuda.synchronize()
    C = x.shape[-1]
    s, gr = stats.cpu(), grads.cpu()
    return {"y": y.cpu(), "dx": dx.cpu(), "mean": s[:C], "var": s[C:2 * C],
            "inv_std": s[2 * C:3 * C], "scale": s[3 * C:4 * C], "running_mean": rm.cpu(),
            "running_var": rv.cpu(), "dgamma": gr[:C], "dbeta": gr[C:2 * C],
            "k1": gr[2 * C:3 * C], "k2": gr[3 * C:]}


def run_oracle(inp, act=None, channels=None, *, beta=True):
    x, dy = inp["x"], inp["dy"]
    C = x.shape[-1]
    g = inp["gamma"]
    b = inp["beta"] if beta else torch.zeros(C)
    rm, rv = inp["running_mean"], inp["running_var"]
    if channels is not None:
        idx = torch.tensor(channels)
        x, dy = x.index_select(-1, idx), dy.index_select(-1, idx)
        g, b, rm, rv = g[idx], b[idx], rm[idx], rv[idx]
    x, dy, g, b, rm, rv = map(_f64, (x, dy, g, b, rm, rv))
    code, slope = ACTS[act]
    f = oracle.batch_norm_nhwc_forward_train(x, g, b, rm, rv, inp["momentum"], inp["eps"], code,
                                             slope)
    bw = oracle.batch_norm_nhwc_backward(x, dy, g, b, inp["eps"], code, slope)
    out = dict(f)
    out.update({k: v for k, v in bw.items() if k != "pre"})
    return out


def compare(got, ref, dtype, channels=None, what=""):
    sel = (lambda t: t) if channels is None else (lambda t: t[..., channels])
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
            C = r.shape[-1]
            tau = tol.tau_of(r.reshape(-1, C), axis=0)  # per channel
            tol.check_bf16(g.reshape(-1, C), r.reshape(-1, C), f"{what} {k}", tau)


SHAPES = [
    ("f32", (4, 64, 7, 9), None),            # C % 4 == 0: 16-byte vectors
    ("f32", (3, 37, 11, 13), (-1000.0, 1000.0)),  # odd C: scalar lanes, large offsets
    ("bf16", (8, 256, 28, 28), (-10.0, 10.0)),    # C % 8 == 0, TX = 32
    ("bf16", (16, 6, 10, 10), None),         # C = 6: 4-byte vectors
    ("bf16", (2, 3000, 5, 3), (-5.0, 5.0)),  # wide C: many column tiles, few rows
    ("bf16", (64, 8, 56, 56), None),         # one vector per row, many rows
]


@pytest.mark.parametrize("dtype,shape,mu", SHAPES, ids=lambda v: str(v))
def test_nhwc_parity(gbn, dtype, shape, mu):
    case = synth.BNCase(f"nhwc_{shape}", shape, dtype, mu_range=mu, seed=901 + shape[1])
    inp = nhwc_inputs(case)
    compare(run_gpu(gbn, inp), run_oracle(inp), dtype, what=f"nhwc {dtype} {shape}")


@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
@pytest.mark.parametrize("dtype,shape", [("f32", (4, 64, 7, 9)), ("bf16", (8, 96, 14, 14)),
                                         ("bf16", (5, 37, 6, 6))])
def test_nhwc_act(gbn, dtype, shape, act):
    case = synth.BNCase(f"nhwc_act_{shape}", shape, dtype, mu_range=(-3.0, 3.0),
                        seed=951 + shape[1])
    inp = nhwc_inputs(case, act)
    compare(run_gpu(gbn, inp, act), run_oracle(inp, act), dtype, what=f"nhwc {act} {shape}")


def test_nhwc_without_beta(gbn):
    case = synth.BNCase("nhwc_nobeta", (3, 40, 9, 9), "f32", seed=971)
    inp = nhwc_inputs(case)
    compare(run_gpu(gbn, inp, None, beta=False), run_oracle(inp, None, beta=False), "f32",
            what="nhwc no beta")


def test_nhwc_full_size_sampled_channels(gbn):
    """The bf16 [128, 256, 56, 56] workload channels-last; 10 channels
    checked element by element."""
    inp = nhwc_inputs(synth.CASES["bn_offset_bf16"])
    C = inp["x"].shape[-1]
    channels = sorted({0, C - 1} | set(range(11, C, 29)))[:10]
    got = run_gpu(gbn, inp)
    compare(got, run_oracle(inp, None, channels), "bf16", channels, what="nhwc full")


def test_nhwc_misaligned_view(gbn):
    case = synth.BNCase("nhwc_mis", (3, 32, 5, 7), "f32", mu_range=(-50.0, 50.0), seed=977)
    inp = nhwc_inputs(case)

    def misaligned(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
        buf[1:] = t.to(DEV).reshape(-1)
        return buf[1:].view(t.shape)

    xm, dym = misaligned(inp["x"]), misaligned(inp["dy"])
    assert xm.data_ptr() % 16 != 0
    compare(run_gpu(gbn, inp, x=xm, dy=dym), run_oracle(inp), "f32", what="nhwc misaligned")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nhwc_constant_dy_cancels(gbn, dtype):
    """A constant dy per channel on zero-mean channels: dgamma and k1 are 0
    to within the fp32 tolerance's absolute floor."""
    case = synth.BNCase(f"nhwc_const_{dtype}", (32, 16, 28, 28), dtype, seed=983)
    inp = nhwc_inputs(case)
    c = torch.tensor([1.0, 0.30078125, -2.5, 7.0] * 4)
    inp["dy"] = c.expand(inp["x"].shape).to(inp["x"].dtype).contiguous()
    got = run_gpu(gbn, inp)
    ref = run_oracle(inp)
    for k in ("dgamma", "dbeta", "k1", "k2"):
        tol.check_f32(got[k], ref[k], f"nhwc constant dy {dtype} {k}")


def test_nhwc_bit_deterministic_and_in_place(gbn):
    case = synth.BNCase("nhwc_det", (8, 64, 14, 14), "bf16", mu_range=(-20.0, 20.0), seed=991)
    inp = nhwc_inputs(case)
    a = run_gpu(gbn, inp)
    b = run_gpu(gbn, inp)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    x = inp["x"].to(DEV)
    g, be = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    _, stats = gbn.bn_nhwc_forward_train(x, g, be, None, None, 0.1, inp["eps"])
    xi = x.clone()
    gbn.bn_nhwc_forward_train(xi, g, be, None, None, 0.1, inp["eps"], y=xi)
    assert torch.equal(xi.cpu(), a["y"])
    dyi = inp["dy"].to(DEV)
    gbn.bn_nhwc_backward(x, dyi, stats, dx=dyi)
    assert torch.equal(dyi.cpu(), a["dx"])


def test_nhwc_matches_nchw_statistics(gbn):
    """The same data through the NCHW and NHWC entry points: the statistics
    agree within the fp32 tolerance (different kernels, different orders)."""
    case = synth.BNCase("nhwc_vs_nchw", (16, 32, 12, 12), "f32", mu_range=(-100.0, 100.0),
                        seed=997)
    inp = synth.bn_inputs(case)
    x = inp["x"].to(DEV)
    _, s1 = gbn.bn_forward_train(x, None, None, None, None, 0.1, inp["eps"])
    _, s2 = gbn.bn_nhwc_forward_train(_nhwc(x), None, None, None, None, 0.1, inp["eps"])
    C = x.shape[1]
    tol.check_f32(s2[:4 * C].cpu(), _f64(s1[:4 * C]), "nhwc vs nchw stats")


@pytest.mark.parametrize("act", [None, "relu", "leaky_relu"])
def test_nhwc_apply_modes(gbn, act):
    """Apply from a training stats buffer equals the training forward's y
    bit for bit; the inference form matches the oracle's apply."""
    case = synth.BNCase("nhwc_apply", (6, 48, 9, 11), "f32", mu_range=(-100.0, 100.0),
                        seed=1009)
    inp = nhwc_inputs(case)
    slope = ACTS[act][1]
    x = inp["x"].to(DEV)
    g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
    y, stats = gbn.bn_nhwc_forward_train(x, g, b, None, None, 0.1, 1e-5, act=act, slope=slope)
    y2 = gbn.bn_nhwc_apply(x, b, stats=stats, act=act, slope=slope)
    assert torch.equal(y, y2)
    r = np.random.default_rng(9)
    C = x.shape[-1]
    rmean = torch.tensor(r.uniform(-100, 100, C), dtype=torch.float32)
    rvar = torch.tensor(r.uniform(0.5, 2.0, C), dtype=torch.float32)
    scale = (inp["gamma"].double() / torch.sqrt(rvar.double() + 1e-5)).float()
    yi = gbn.bn_nhwc_apply(x, b, mean=rmean.to(DEV), scale=scale.to(DEV), act=act, slope=slope)
    x64 = np.moveaxis(_f64(inp["x"]), -1, 1)
    pre = oracle.batch_norm_apply(x64, _f64(rmean), _f64(scale), _f64(inp["beta"]))
    ref = np.moveaxis(oracle.activation(pre, ACTS[act][0], slope), 1, -1)
    tol.check_f32(yi, ref, f"nhwc inference apply {act}")


@pytest.mark.parametrize("dtype,shape", [("f32", (2, 1, 1, 1)), ("bf16", (1, 1, 2, 3)),
                                         ("bf16", (3, 5000, 1, 2)), ("f32", (2, 7, 1, 1))])
def test_nhwc_edge_shapes(gbn, dtype, shape):
    """Two rows only, one channel, 5000 channels (20 column tiles of 32
    vectors), a 1x1 image."""
    case = synth.BNCase(f"nhwc_edge_{shape}", shape, dtype, seed=1013 + shape[1])
    inp = nhwc_inputs(case)
    compare(run_gpu(gbn, inp), run_oracle(inp), dtype, what=f"nhwc edge {shape}")
