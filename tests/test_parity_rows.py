"""RMSNorm and (fused) LayerNorm backward: CUDA path vs the float64 oracle.

Full-size workloads element by element (RMSNorm [2048, 8192] in bf16 and
fp32, fused LayerNorm [8192, 1600] bf16), both the bulk-copy fast path and
the generic path (ragged / unaligned H), all optional inputs, edge sizes and
bit-determinism."""

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


def _check(got, ref, dtype, name):
    tol.check(got, ref, name, dtype)


# ------------------------------------------------------------------ RMSNorm

def rms_case(R, H, dtype, seed=5):
    case = synth.RMSCase(f"rms_{R}x{H}_{dtype}", R, H, dtype, seed=seed)
    inp = synth.rms_inputs(case)
    rstd = oracle.rms_norm_rstd(_f64(inp["x"]), inp["eps"])
    inp["rstd"] = torch.tensor(rstd, dtype=torch.float32)
    return inp


def rms_gpu(gbn, inp, **kw):
    dx, dw = gbn.rmsnorm_backward(inp["dy"].to(DEV), inp["x"].to(DEV), inp["w"].to(DEV),
                                  inp["rstd"].to(DEV), **kw)
    torch.cuda.synchronize()
    return dx.cpu(), dw.cpu()


def rms_ref(inp):
    return oracle.rms_norm_backward(_f64(inp["x"]), _f64(inp["dy"]), _f64(inp["w"]),
                                    _f64(inp["rstd"]))


@pytest.mark.parametrize("name", ["rms_bf16", "rms_f32"])
def test_rms_full_size(gbn, name):
    case = synth.CASES[name]
    inp = synth.rms_inputs(case)
    inp["rstd"] = torch.tensor(oracle.rms_norm_rstd(_f64(inp["x"]), case.eps),
                               dtype=torch.float32)
    dx, dw = rms_gpu(gbn, inp)
    ref = rms_ref(inp)
    _check(dx, ref["dx"], case.dtype, f"{name} dx")
    _check(dw, ref["dw"], case.dtype, f"{name} dw")


RMS_SHAPES = [
    (1, 8, "bf16"), (3, 64, "f32"), (37, 1000, "bf16"), (37, 1000, "f32"),
    (200, 512, "bf16"), (150, 5000, "bf16"), (64, 3000, "f32"), (70, 8192, "bf16"),
    (33, 6144, "f32"),
    # generic path: H*esize not a multiple of 16, or rows larger than the fast path
    (41, 1001, "bf16"), (41, 777, "f32"), (20, 9000, "f32"), (12, 20000, "bf16"),
    (5, 3, "f32"),
]


@pytest.mark.parametrize("R,H,dtype", RMS_SHAPES)
def test_rms_shapes(gbn, R, H, dtype):
    inp = rms_case(R, H, dtype)
    dx, dw = rms_gpu(gbn, inp)
    ref = rms_ref(inp)
    _check(dx, ref["dx"], dtype, f"rms {R}x{H} dx")
    _check(dw, ref["dw"], dtype, f"rms {R}x{H} dw")


def test_rms_zero_rows_gives_zero_dweight(gbn):
    w = torch.rand(256, device=DEV)
    x = torch.empty(0, 256, device=DEV)
    dx, dw = gbn.rmsnorm_backward(x, x, w, torch.empty(0, device=DEV))
    torch.cuda.synchronize()
    assert dx.numel() == 0 and torch.all(dw == 0)


def test_rms_misaligned_uses_generic_path(gbn):
    inp = rms_case(40, 1024, "bf16")
    ref = rms_ref(inp)

    def mis(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
        buf[1:] = t.to(DEV).reshape(-1)
        return buf[1:].view(t.shape)

    dx, dw = gbn.rmsnorm_backward(mis(inp["dy"]), mis(inp["x"]), inp["w"].to(DEV),
                                  inp["rstd"].to(DEV))
    _check(dx, ref["dx"], "bf16", "rms misaligned dx")
    _check(dw, ref["dw"], "bf16", "rms misaligned dw")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_rms_bit_deterministic(gbn, dtype):
    inp = rms_case(2048, 8192, dtype, seed=11)
    a = rms_gpu(gbn, inp)
    b = rms_gpu(gbn, inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ---------------------------------------------------------------- LayerNorm

def ln_case(R, H, dtype, fused=True, with_dz_extra=False, seed=9):
    case = synth.LNCase(f"ln_{R}x{H}", R, H, dtype, fused=fused, with_dz_extra=with_dz_extra,
                        seed=seed)
    return prepare_ln(synth.ln_inputs(case))


def prepare_ln(inp):
    if inp["residual"] is not None:
        z = oracle.dropout_add(_f64(inp["inp"]), _f64(inp["residual"]), _f64(inp["bias"]),
                               _f64(inp["mask"]), inp["dropout_scale"])
    else:
        z = _f64(inp["inp"])
    mu, rs = oracle.layer_norm_saved_stats(z, inp["eps"])
    inp["mean"] = torch.tensor(mu, dtype=torch.float32)
    inp["rstd"] = torch.tensor(rs, dtype=torch.float32)
    return inp


def ln_gpu(gbn, inp, drop=()):
    d = {k: (None if (v is None or k in drop) else (v.to(DEV) if torch.is_tensor(v) else v))
         for k, v in inp.items()}
    out = gbn.layernorm_backward(d["dy"], d["inp"], d["mean"], d["rstd"], d["gamma"],
                                 residual=d["residual"], bias=d["bias"], mask=d["mask"],
                                 dropout_scale=inp["dropout_scale"], dz_extra=d["dz_extra"])
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu()) for k, v in out.items()}


def ln_ref(inp, drop=()):
    g = {k: (None if k in drop else v) for k, v in inp.items()}
    if g["residual"] is not None:
        return oracle.fused_bias_dropout_add_layer_norm_backward(
            _f64(g["dy"]), _f64(g["inp"]), _f64(g["residual"]), _f64(g["bias"]),
            _f64(g["mask"]), inp["dropout_scale"], _f64(g["mean"]), _f64(g["rstd"]),
            _f64(g["gamma"]), dz_extra=_f64(g["dz_extra"]))
    return oracle.layer_norm_backward(_f64(g["dy"]), _f64(g["inp"]), _f64(g["mean"]),
                                      _f64(g["rstd"]), _f64(g["gamma"]),
                                      dz_extra=_f64(g["dz_extra"]))


def ln_compare(got, ref, dtype, what):
    for k, r in ref.items():
        if r is None:
            continue
        _check(got[k], r, dtype, f"{what} {k}")


def test_ln_fused_full_size(gbn):
    case = synth.CASES["ln_fused_bf16"]
    inp = prepare_ln(synth.ln_inputs(case))
    ln_compare(ln_gpu(gbn, inp), ln_ref(inp), "bf16", "ln_fused_bf16")


LN_SHAPES = [
    (1, 1600, "bf16", True), (37, 1600, "bf16", True), (129, 1024, "f32", True),
    (64, 4096, "bf16", True), (50, 8192, "bf16", False), (33, 4096, "f32", False),
    (100, 320, "bf16", False), (31, 2048, "f32", True),
    # generic path: unaligned rows, mask with H % 16 != 0, or rows too wide
    (23, 1000, "bf16", True), (23, 777, "f32", False), (9, 12288, "bf16", True),
    (7, 5000, "f32", True), (4, 3, "bf16", True),
]


@pytest.mark.parametrize("R,H,dtype,fused", LN_SHAPES)
def test_ln_shapes(gbn, R, H, dtype, fused):
    inp = ln_case(R, H, dtype, fused=fused)
    ln_compare(ln_gpu(gbn, inp), ln_ref(inp), dtype, f"ln {R}x{H} fused={fused}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fused", [True, False])
def test_ln_with_dz_extra(gbn, dtype, fused):
    inp = ln_case(96, 1600, dtype, fused=fused, with_dz_extra=True)
    ln_compare(ln_gpu(gbn, inp), ln_ref(inp), dtype, f"ln dz_extra fused={fused}")


@pytest.mark.parametrize("drop", [("mask",), ("bias",), ("mask", "bias")])
def test_ln_fused_optional_inputs(gbn, drop):
    inp = ln_case(80, 1600, "bf16")
    got = ln_gpu(gbn, inp, drop)
    ref = ln_ref(inp, drop)
    ln_compare(got, ref, "bf16", f"ln without {drop}")


def test_ln_dropped_positions_have_zero_dx(gbn):
    inp = ln_case(64, 1600, "bf16")
    got = ln_gpu(gbn, inp)
    assert torch.all(got["dx"][inp["mask"] == 0] == 0)


def test_ln_bit_deterministic(gbn):
    inp = ln_case(4096, 1600, "bf16", seed=13)
    a, b = ln_gpu(gbn, inp), ln_gpu(gbn, inp)
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k


def test_device_status_clean(gbn):
    torch.cuda.synchronize()
    assert gbn.get_device_status() == 0


# ------------------------------------------- LayerNorm backward variants --

def saved_z_case(R, H, dtype, seed=13, with_dz_extra=False):
    """A fused case whose LayerNorm input z is stored in `dtype` (as the
    forward writes it) and handed to the backward instead of the operands."""
    inp = synth.ln_inputs(synth.LNCase(f"lnz_{R}x{H}", R, H, dtype, seed=seed,
                                       with_dz_extra=with_dz_extra))
    z = oracle.dropout_add(_f64(inp["inp"]), _f64(inp["residual"]), _f64(inp["bias"]),
                           _f64(inp["mask"]), inp["dropout_scale"])
    inp["z"] = torch.tensor(z).to(inp["inp"].dtype)
    mu, rs = oracle.layer_norm_saved_stats(_f64(inp["z"]), inp["eps"])
    inp["mean"] = torch.tensor(mu, dtype=torch.float32)
    inp["rstd"] = torch.tensor(rs, dtype=torch.float32)
    return inp


def saved_z_gpu(gbn, inp, dres_f32=False):
    d = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
    out = gbn.layernorm_backward(d["dy"], d["z"], d["mean"], d["rstd"], d["gamma"],
                                 mask=d["mask"], dropout_scale=inp["dropout_scale"],
                                 dz_extra=d["dz_extra"], saved_z=True, dres_f32=dres_f32)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu()) for k, v in out.items()}


def saved_z_ref(inp):
    return oracle.layer_norm_backward_saved_z(
        _f64(inp["dy"]), _f64(inp["z"]), _f64(inp["mask"]), inp["dropout_scale"],
        _f64(inp["mean"]), _f64(inp["rstd"]), _f64(inp["gamma"]), dz_extra=_f64(inp["dz_extra"]))


@pytest.mark.parametrize("R,H,dtype", [(8192, 1600, "bf16"), (129, 1024, "f32"),
                                       (23, 1000, "bf16"), (7, 5000, "f32")])
def test_ln_backward_from_saved_z(gbn, R, H, dtype):
    """The fused outputs from the saved z match the oracle (bulk-copy path for
    the aligned shapes, the generic kernel for H % 16 != 0 or wide rows)."""
    inp = saved_z_case(R, H, dtype)
    ln_compare(saved_z_gpu(gbn, inp), saved_z_ref(inp), dtype, f"saved z {R}x{H}")


def test_ln_backward_saved_z_with_dz_extra_and_fp32_dresidual(gbn):
    inp = saved_z_case(96, 1600, "bf16", with_dz_extra=True)
    got = saved_z_gpu(gbn, inp, dres_f32=True)
    ref = saved_z_ref(inp)
    assert got["dresidual"].dtype == torch.float32
    tol.check_f32(got["dresidual"], ref["dresidual"], "saved z fp32 dresidual")
    for k in ("dx", "dbias", "dgamma", "dbeta"):
        _check(got[k], ref[k], "bf16", f"saved z {k}")


@pytest.mark.parametrize("R,H", [(256, 1600), (23, 1000)])
def test_ln_fused_backward_fp32_dresidual(gbn, R, H):
    """dresidual in fp32 (the residual gradient the fused repro emits in fp32)
    from bf16 operands, on the bulk-copy
    and the generic kernel; the other outputs are unchanged."""
    inp = ln_case(R, H, "bf16")
    d = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
    out = gbn.layernorm_backward(d["dy"], d["inp"], d["mean"], d["rstd"], d["gamma"],
                                 residual=d["residual"], bias=d["bias"], mask=d["mask"],
                                 dropout_scale=inp["dropout_scale"], dres_f32=True)
    torch.cuda.synchronize()
    ref = ln_ref(inp)
    assert out["dresidual"].dtype == torch.float32
    tol.check_f32(out["dresidual"].cpu(), ref["dresidual"], "fp32 dresidual")
    for k in ("dx", "dbias", "dgamma", "dbeta"):
        _check(out[k].cpu(), ref[k], "bf16", f"fp32-dres run {k}")
