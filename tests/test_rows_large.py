"""RMSNorm and fused LayerNorm backward at 2^31 elements per tensor.

Row offsets past 2^31 - 1 are exercised: RMSNorm bf16 [2^18, 8192] and the
bias+dropout+add LayerNorm bf16 [1342178, 1600].  Rows are independent, so
the oracle checks sampled rows (first, middle, last) element by element; the
column sums run over every row, so dweight (RMSNorm) and dgamma / dbeta
(LayerNorm) are checked against their definitions -- float64 sums over all
rows of dy*x*rstd, dy*xhat and dy, computed by torch from the same data.
Inputs follow the workloads' laws, drawn on the device from a seeded
generator (2^31 host-side draws would take minutes); the saved statistics
are computed by torch from the same stored values."""

import numpy as np
import pytest
import torch

import oracle

from . import tolerances as tol

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CHUNK = 1 << 14  # rows per float64 chunk (at most ~1 GB per temporary)


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _f64(t):
    return t.detach().cpu().double().numpy()


def _randn_bf16(R, H, gen):
    out = torch.empty(R, H, dtype=torch.bfloat16, device=DEV)
    for r0 in range(0, R, CHUNK):
        n = min(CHUNK, R - r0)
        out[r0:r0 + n] = torch.randn(n, H, device=DEV, generator=gen).to(torch.bfloat16)
    return out


def _rows(R):
    return [0, 1, R // 2 + 3, R - 2, R - 1]


def test_rms_backward_beyond_int32_elements(gbn):
    R, H, eps = 1 << 18, 8192, 1e-5
    gen = torch.Generator(device=DEV)
    gen.manual_seed(20241208)
    x = _randn_bf16(R, H, gen)
    dy = _randn_bf16(R, H, gen)
    w = (torch.rand(H, device=DEV, generator=gen) + 0.5).to(torch.bfloat16)
    assert x.numel() == 2 ** 31
    rstd = torch.empty(R, device=DEV)
    for r0 in range(0, R, CHUNK):
        xs = x[r0:r0 + CHUNK].double()
        rstd[r0:r0 + CHUNK] = torch.rsqrt((xs * xs).mean(dim=1) + eps).float()
    dx, dw = gbn.rmsnorm_backward(dy, x, w, rstd)
    torch.cuda.synchronize()

    rows = _rows(R)
    ref = oracle.rms_norm_backward(_f64(x[rows]), _f64(dy[rows]), _f64(w), _f64(rstd[rows]))
    tol.check_bf16(dx[rows].cpu(), ref["dx"], "2^31 elements RMSNorm dx (sampled rows)")

    dw64 = torch.zeros(H, dtype=torch.float64, device=DEV)
    for r0 in range(0, R, CHUNK):
        dw64 += (dy[r0:r0 + CHUNK].double() * x[r0:r0 + CHUNK].double()
                 * rstd[r0:r0 + CHUNK].double()[:, None]).sum(dim=0)
    tol.check_bf16(dw.cpu(), dw64.cpu().numpy(), "2^31 elements RMSNorm dweight (all rows)")


def test_fused_layernorm_backward_beyond_int32_elements(gbn):
    H, eps, keep_prob = 1600, 1e-5, 0.9
    R = (2 ** 31 + H - 1) // H  # 1342178 rows: 2^31 + 800 elements
    scale = float(np.float32(1.0 / 0.9))
    gen = torch.Generator(device=DEV)
    gen.manual_seed(20241209)
    inp = _randn_bf16(R, H, gen)
    res = _randn_bf16(R, H, gen)
    dy = _randn_bf16(R, H, gen)
    mask = torch.empty(R, H, dtype=torch.uint8, device=DEV)
    for r0 in range(0, R, CHUNK):
        n = min(CHUNK, R - r0)
        mask[r0:r0 + n] = (torch.rand(n, H, device=DEV, generator=gen) < keep_prob).to(torch.uint8)
    bias = torch.randn(H, device=DEV, generator=gen).to(torch.bfloat16)
    gamma = (torch.rand(H, device=DEV, generator=gen) + 0.5).to(torch.bfloat16)
    assert inp.numel() > 2 ** 31

    def z_chunk(r0, n):
        return (res[r0:r0 + n].double()
                + mask[r0:r0 + n].double() * scale * (inp[r0:r0 + n].double() + bias.double()))

    mean = torch.empty(R, device=DEV)
    rstd = torch.empty(R, device=DEV)
    for r0 in range(0, R, CHUNK):
        n = min(CHUNK, R - r0)
        z = z_chunk(r0, n)
        mu = z.mean(dim=1)
        mean[r0:r0 + n] = mu.float()
        rstd[r0:r0 + n] = torch.rsqrt(((z - mu[:, None]) ** 2).mean(dim=1) + eps).float()
        del z

    out = gbn.layernorm_backward(dy, inp, mean, rstd, gamma, residual=res, bias=bias, mask=mask,
                                 dropout_scale=scale)
    torch.cuda.synchronize()
    dx, dres, dgamma, dbeta, dbias = (out[k] for k in ("dx", "dresidual", "dgamma", "dbeta",
                                                       "dbias"))

    rows = _rows(R)
    ref = oracle.fused_bias_dropout_add_layer_norm_backward(
        _f64(dy[rows]), _f64(inp[rows]), _f64(res[rows]), _f64(bias), _f64(mask[rows]), scale,
        _f64(mean[rows]), _f64(rstd[rows]), _f64(gamma))
    tol.check_bf16(dx[rows].cpu(), ref["dx"], "2^31 elements LayerNorm dx (sampled rows)")
    tol.check_bf16(dres[rows].cpu(), ref["dresidual"],
                   "2^31 elements LayerNorm dresidual (sampled rows)")

    dg64 = torch.zeros(H, dtype=torch.float64, device=DEV)
    db64 = torch.zeros(H, dtype=torch.float64, device=DEV)
    for r0 in range(0, R, CHUNK):
        n = min(CHUNK, R - r0)
        xhat = (z_chunk(r0, n) - mean[r0:r0 + n].double()[:, None]) * rstd[r0:r0 + n].double()[:, None]
        d = dy[r0:r0 + n].double()
        dg64 += (d * xhat).sum(dim=0)
        db64 += d.sum(dim=0)
        del xhat, d
    tol.check_bf16(dgamma.cpu(), dg64.cpu().numpy(), "2^31 elements LayerNorm dgamma (all rows)")
    tol.check_bf16(dbeta.cpu(), db64.cpu().numpy(), "2^31 elements LayerNorm dbeta (all rows)")
    assert torch.isfinite(dbias.float()).all()
