"""RMSNorm and (fused) LayerNorm training forwards: CUDA path vs the float64
oracle.

The row workloads of the backward tests (RMSNorm [2048, 8192] bf16 / fp32,
fused bias+dropout+add LayerNorm [8192, 1600] bf16) element by element, all
three kernel forms (a warp per row, a block per row, the streaming form for
long or unaligned rows), rows with a large offset, optional inputs, edge
sizes, bit-determinism, and the forward's saved statistics feeding the
backward."""

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
    return None if t is None else t.detach().cpu().double().numpy()


def _dev(t):
    return None if t is None else t.to(DEV)


# ------------------------------------------------------------------ RMSNorm

def _rms_check(gbn, x, w, eps, what):
    y, rstd = gbn.rmsnorm_forward(_dev(x), _dev(w), eps)
    torch.cuda.synchronize()
    ref = oracle.rms_norm_forward(_f64(x), _f64(w), eps)
    tol.check(y.cpu(), ref["y"], f"{what} y", "f32" if x.dtype == torch.float32 else "bf16")
    tol.check_f32(rstd.cpu(), ref["rstd"], f"{what} rstd")
    return y, rstd


@pytest.mark.parametrize("name", ["rms_bf16", "rms_f32"])
def test_rms_forward_full_size(gbn, name):
    inp = synth.rms_inputs(synth.CASES[name])
    _rms_check(gbn, inp["x"], inp["w"], inp["eps"], name)


@pytest.mark.parametrize("R,H,dtype", [
    (37, 64, "bf16"),      # a warp per row, one vector per lane
    (19, 1600, "f32"),     # a block per row (400 vectors)
    (5, 20000, "bf16"),    # streaming form (2500 vectors)
    (6, 1001, "f32"),      # streaming form (not a whole number of vectors)
    (3, 4, "f32"),         # one vector per row
])
def test_rms_forward_shapes(gbn, R, H, dtype):
    inp = synth.rms_inputs(synth.RMSCase(f"rmsf_{R}x{H}", R, H, dtype, seed=31 + H))
    _rms_check(gbn, inp["x"], inp["w"], inp["eps"], f"rms fwd {R}x{H} {dtype}")


def test_rms_forward_without_weight_and_zero_rows(gbn):
    inp = synth.rms_inputs(synth.RMSCase("rmsf_now", 9, 512, "bf16", seed=41))
    _rms_check(gbn, inp["x"], None, inp["eps"], "rms fwd w=None")
    x = torch.empty(0, 512, dtype=torch.bfloat16, device=DEV)
    y, rstd = gbn.rmsnorm_forward(x, None, 1e-5)
    assert y.numel() == 0 and rstd.numel() == 0


def test_rms_forward_misaligned_view(gbn):
    inp = synth.rms_inputs(synth.RMSCase("rmsf_mis", 4, 256, "f32", seed=43))
    big = torch.zeros(4 * 256 + 1, dtype=torch.float32)
    big[1:] = inp["x"].reshape(-1)
    xv = big.to(DEV)[1:].view(4, 256)           # 4-byte aligned, not 16
    y, rstd = gbn.rmsnorm_forward(xv, _dev(inp["w"]), inp["eps"])
    ref = oracle.rms_norm_forward(_f64(inp["x"]), _f64(inp["w"]), inp["eps"])
    tol.check_f32(y.cpu(), ref["y"], "misaligned y")
    tol.check_f32(rstd.cpu(), ref["rstd"], "misaligned rstd")


# ---------------------------------------------------------------- LayerNorm

def _ln_fused(gbn, inp, eps, **kw):
    out = gbn.layernorm_forward(_dev(inp["inp"]), _dev(inp["gamma"]), _dev(inp["beta"]), eps,
                                residual=_dev(inp["residual"]), bias=_dev(inp["bias"]),
                                mask=_dev(inp["mask"]), dropout_scale=inp["dropout_scale"], **kw)
    torch.cuda.synchronize()
    return out


def _ln_fused_ref(inp, eps):
    mask = None if inp["mask"] is None else _f64(inp["mask"].to(torch.uint8))
    return oracle.fused_bias_dropout_add_layer_norm_forward(
        _f64(inp["inp"]), _f64(inp["residual"]), _f64(inp["bias"]), mask,
        inp["dropout_scale"], _f64(inp["gamma"]), _f64(inp["beta"]), eps)


def _ln_compare(out, ref, dtype, what):
    tol.check(out["y"].cpu(), ref["y"], f"{what} y", dtype)
    if out.get("z") is not None:
        tol.check(out["z"].cpu(), ref["z"], f"{what} z", dtype)
    tol.check_f32(out["mean"].cpu(), ref["mean"], f"{what} mean")
    tol.check_f32(out["rstd"].cpu(), ref["rstd"], f"{what} rstd")


def test_ln_fused_forward_full_size(gbn):
    case = synth.CASES["ln_fused_bf16"]
    inp = synth.ln_inputs(case)
    _ln_compare(_ln_fused(gbn, inp, case.eps), _ln_fused_ref(inp, case.eps), "bf16",
                "fused LN fwd")


@pytest.mark.parametrize("R,H,dtype", [
    (33, 1600, "f32"),     # a block per row (400 vectors)
    (70, 256, "bf16"),     # a warp per row
    (4, 20000, "bf16"),    # streaming form
    (9, 1000, "f32"),      # streaming form with a mask (H % 16 != 0)
])
def test_ln_fused_forward_shapes(gbn, R, H, dtype):
    case = synth.LNCase(f"lnf_{R}x{H}", R, H, dtype, seed=53 + H)
    inp = synth.ln_inputs(case)
    _ln_compare(_ln_fused(gbn, inp, case.eps), _ln_fused_ref(inp, case.eps), dtype,
                f"fused LN fwd {R}x{H} {dtype}")


@pytest.mark.parametrize("R,H,dtype", [(64, 1600, "f32"), (50, 96, "bf16"), (7, 3000, "f32")])
def test_ln_plain_forward_large_offset(gbn, R, H, dtype):
    """Rows with |mean| up to 1000 and unit spread: the shifted form keeps y
    and the statistics within the strict fp32 bound."""
    g = torch.Generator().manual_seed(61 + H)
    mu = torch.empty(R, 1, dtype=torch.float64).uniform_(-1000, 1000, generator=g)
    x = (mu + torch.randn(R, H, generator=g, dtype=torch.float64)).to(synth.DTYPES[dtype])
    gamma = torch.empty(H, dtype=torch.float64).uniform_(0.5, 1.5, generator=g).to(x.dtype)
    beta = (0.1 * torch.randn(H, generator=g, dtype=torch.float64)).to(x.dtype)
    out = gbn.layernorm_forward(_dev(x), _dev(gamma), _dev(beta), 1e-5)
    torch.cuda.synchronize()
    ref = oracle.layer_norm_forward(_f64(x), _f64(gamma), _f64(beta), 1e-5)
    _ln_compare(out, ref, dtype, f"plain LN fwd offset {R}x{H} {dtype}")


def test_ln_forward_optional_inputs(gbn):
    case = synth.LNCase("lnf_opt", 16, 512, "bf16", seed=67)
    inp = synth.ln_inputs(case)
    # fused without bias, without mask, without the z output
    inp2 = dict(inp, bias=None, mask=None)
    out = _ln_fused(gbn, inp2, case.eps, want_z=False)
    assert out["z"] is None
    _ln_compare(out, _ln_fused_ref(inp2, case.eps), "bf16", "fused, no bias/mask")
    # plain without gamma / beta
    out = gbn.layernorm_forward(_dev(inp["inp"]), None, None, case.eps)
    torch.cuda.synchronize()
    ref = oracle.layer_norm_forward(_f64(inp["inp"]), None, None, case.eps)
    _ln_compare(out, ref, "bf16", "plain, no affine")


def test_forwards_bit_deterministic(gbn):
    inp = synth.ln_inputs(synth.LNCase("lnf_det", 256, 1600, "bf16", seed=71))
    a = _ln_fused(gbn, inp, 1e-5)
    b = _ln_fused(gbn, inp, 1e-5)
    for k in ("y", "z", "mean", "rstd"):
        assert torch.equal(a[k], b[k]), k
    r = synth.rms_inputs(synth.RMSCase("rmsf_det", 64, 8192, "bf16", seed=73))
    y1, s1 = gbn.rmsnorm_forward(_dev(r["x"]), _dev(r["w"]), 1e-5)
    y2, s2 = gbn.rmsnorm_forward(_dev(r["x"]), _dev(r["w"]), 1e-5)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)


def test_ln_forward_statistics_feed_the_backward(gbn):
    """The saved mean / rstd of the forward drive the fused backward; the
    backward then matches the oracle backward given the same statistics."""
    case = synth.LNCase("lnf_rt", 128, 1600, "bf16", seed=79)
    inp = synth.ln_inputs(case)
    out = _ln_fused(gbn, inp, case.eps)
    bw = gbn.layernorm_backward(_dev(inp["dy"]), _dev(inp["inp"]), out["mean"], out["rstd"],
                                _dev(inp["gamma"]), residual=_dev(inp["residual"]),
                                bias=_dev(inp["bias"]), mask=_dev(inp["mask"]),
                                dropout_scale=inp["dropout_scale"])
    torch.cuda.synchronize()
    mask = _f64(inp["mask"].to(torch.uint8))
    ref = oracle.fused_bias_dropout_add_layer_norm_backward(
        _f64(inp["dy"]), _f64(inp["inp"]), _f64(inp["residual"]), _f64(inp["bias"]), mask,
        inp["dropout_scale"], _f64(out["mean"]), _f64(out["rstd"]), _f64(inp["gamma"]))
    for k in ("dx", "dresidual", "dgamma", "dbeta", "dbias"):
        tol.check(bw[k].cpu(), ref[k], f"round trip {k}", "bf16")
