"""No kernel writes outside its outputs or workspace.

Every output and workspace of a call is carved out of a larger device
buffer whose bands before and after it hold a byte pattern; after the call
the bands must be unchanged.  The shapes are ragged (row or plane lengths
that are not a multiple of the vector width, a tail of rows or planes that
leaves a block or CTA part-filled) and run through every kernel path:
persistent and two-launch BatchNorm, channels-last BatchNorm, RMSNorm and
LayerNorm forward and backward.  (Out-of-bounds reads are not visible this
way; the parity tests would see their effect on the results.)"""

import pytest
import torch

from bwd_bn_pass_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BAND = 4096  # bytes of pattern on each side
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class Guarded:
    """Device tensors inside patterned byte buffers; `check()` asserts the
    bands are intact."""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        raw = torch.full((BAND + nbytes + BAND,), PATTERN, dtype=torch.uint8, device=DEV)
        t = raw[BAND:BAND + nbytes].view(dtype).view(shape)
        t.zero_()
        self.bufs.append((raw, nbytes))
        return t

    def like(self, t):
        return self.empty(tuple(t.shape), t.dtype)

    def bytes(self, nbytes):
        return self.empty((max(nbytes, 1),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for raw, nbytes in self.bufs:
            assert torch.all(raw[:BAND] == PATTERN), "band before an output was written"
            assert torch.all(raw[BAND + nbytes:] == PATTERN), "band after an output was written"


@pytest.mark.parametrize("path", ["two-launch", "small-channel", "persistent"])
@pytest.mark.parametrize("dtype,shape", [("f32", (3, 37, 41, 40)), ("bf16", (5, 19, 7, 9)),
                                         ("bf16", (2, 300, 8, 8)), ("f32", (4, 3, 5, 5))])
def test_batchnorm_writes_stay_inside(gbn, dtype, shape, path):
    prev = gbn.bn_set_persistent_min_bytes(0 if path == "persistent" else 1 << 62)
    prev_small = gbn.bn_set_small_max_elems(0 if path == "two-launch" else 2048)
    try:
        inp = synth.bn_inputs(synth.BNCase("guard_bn", shape, dtype, seed=1201))
        x, dy = inp["x"].to(DEV), inp["dy"].to(DEV)
        G = Guarded()
        C = shape[1]
        y, dx = G.like(x), G.like(x)
        stats, grads = G.empty((8 * C,), torch.float32), G.empty((4 * C,), torch.float32)
        rm, rv = G.empty((C,), torch.float32), G.empty((C,), torch.float32)
        rv.fill_(1.0)
        ws = G.bytes(gbn.bn_workspace_bytes(shape[0], C, shape[2] * shape[3]))
        gbn.bn_forward_train(x, inp["gamma"].to(DEV), inp["beta"].to(DEV), rm, rv, 0.1, 1e-5,
                             y=y, stats=stats, ws=ws, act="relu")
        gbn.bn_backward(x, dy, stats, dx=dx, grads=grads, ws=ws, beta=inp["beta"].to(DEV),
                        act="relu")
        G.check()
    finally:
        gbn.bn_set_persistent_min_bytes(prev)
        gbn.bn_set_small_max_elems(prev_small)


@pytest.mark.parametrize("dtype,shape", [("f32", (3, 37, 5, 3)), ("bf16", (4, 24, 3, 7)),
                                         ("bf16", (2, 6, 9, 1))])
def test_channels_last_writes_stay_inside(gbn, dtype, shape):
    inp = synth.bn_inputs(synth.BNCase("guard_nhwc", shape, dtype, seed=1203))
    x = inp["x"].permute(0, 2, 3, 1).contiguous().to(DEV)
    dy = inp["dy"].permute(0, 2, 3, 1).contiguous().to(DEV)
    C = x.shape[-1]
    G = Guarded()
    y, dx = G.like(x), G.like(x)
    stats, grads = G.empty((8 * C,), torch.float32), G.empty((4 * C,), torch.float32)
    ws = G.bytes(gbn.lib().gbn_bn_nhwc_workspace_bytes(x.numel() // C, C, -1))
    gbn.bn_nhwc_forward_train(x, None, None, None, None, 0.1, 1e-5, y=y, stats=stats, ws=ws)
    gbn.bn_nhwc_backward(x, dy, stats, dx=dx, grads=grads, ws=ws)
    G.check()


@pytest.mark.parametrize("R,H,dtype", [(37, 1000, "bf16"), (33, 6144, "f32"), (70, 8192, "bf16"),
                                       (41, 1001, "bf16"), (5, 3, "f32")])
def test_rmsnorm_writes_stay_inside(gbn, R, H, dtype):
    inp = synth.rms_inputs(synth.RMSCase("guard_rms", R, H, dtype, seed=1205))
    x, dy, w = inp["x"].to(DEV), inp["dy"].to(DEV), inp["w"].to(DEV)
    G = Guarded()
    y, rstd = G.like(x), G.empty((R,), torch.float32)
    gbn.rmsnorm_forward(x, w, 1e-5, y=y, rstd=rstd)
    dx, dw = G.like(x), G.like(w)
    kind = gbn.GBN_ROW_RMS
    ws = G.bytes(gbn.rowwise_workspace_bytes(R, H, kind, x.dtype))
    gbn.rmsnorm_backward(dy, x, w, rstd, dx=dx, dw=dw, ws=ws)
    G.check()


@pytest.mark.parametrize("R,H,dtype", [(33, 1600, "bf16"), (9, 1000, "f32"), (70, 256, "bf16"),
                                       (4, 20000, "bf16")])
def test_layernorm_writes_stay_inside(gbn, R, H, dtype):
    case = synth.LNCase("guard_ln", R, H, dtype, seed=1207 + H)
    inp = synth.ln_inputs(case)
    d = {k: v.to(DEV) for k, v in inp.items() if torch.is_tensor(v)}
    G = Guarded()
    y, z = G.like(d["inp"]), G.like(d["inp"])
    mean, rstd = G.empty((R,), torch.float32), G.empty((R,), torch.float32)
    gbn.layernorm_forward(d["inp"], d["gamma"], d["beta"], case.eps, residual=d["residual"],
                          bias=d["bias"], mask=d["mask"], dropout_scale=inp["dropout_scale"],
                          y=y, z=z, mean=mean, rstd=rstd)
    dx, dres = G.like(d["inp"]), G.like(d["inp"])
    dg, db, dbias = G.like(d["gamma"]), G.like(d["gamma"]), G.like(d["gamma"])
    ws = G.bytes(gbn.rowwise_workspace_bytes(R, H, gbn.GBN_ROW_LN_FUSED, d["inp"].dtype))
    gbn.layernorm_backward(d["dy"], d["inp"], mean, rstd, d["gamma"], residual=d["residual"],
                           bias=d["bias"], mask=d["mask"], dropout_scale=inp["dropout_scale"],
                           dx=dx, dresidual=dres, dgamma=dg, dbeta=db, dbias=dbias, ws=ws)
    G.check()
