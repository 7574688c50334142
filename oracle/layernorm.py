"""LayerNorm backward, plain and fused with bias+dropout+add (oracle).

Test infrastructure only; see ``oracle/__init__.py``.

Source: nvFuser issue #1473, "Why is LayerNorm Backward Segmenting?".

* "A repro of the 3-Kernel layer_norm backward fusion" (nvfuser_fusion_id14)
  is the plain LayerNorm backward.
* "A repro of the 1-Kernel bias+dropout+add+layer_norm backward fusion"
  (nvfuser_fusion_id9) is the same backward followed by the gradient of a
  bias+dropout+add that produced the LayerNorm input.

What is computed, per row of length H with the saved mean mu and saved
rstd rho = 1/sqrt(var + eps) (both inputs of the repros), written out by the
chain rule.  The forward is y = xhat * gamma + beta with xhat = (z - mu) * rho,
where mu and var (biased) are functions of the whole row z.  With
g = dL/dxhat = dy * gamma, the loss reaches z directly through xhat, and
through mu and var:

    dL/dvar  = sum_j g_j * (z_j - mu) * d(rho)/d(var)
             = -1/2 * rho^3 * sum_j g_j * (z_j - mu)
    dL/dmu   = -rho * sum_j g_j          (the var path adds
               dL/dvar * (-2/H) * sum_j (z_j - mu) = 0)
    dz_j     = g_j * rho + dL/dvar * 2 * (z_j - mu) / H + dL/dmu / H
    dz      += dz_extra                  (an optional fp32 gradient that
                                          reaches z by another path)
    dgamma   = sum_rows dy * xhat,   dbeta = sum_rows dy

and, for the fused form where z = residual + dropout(input + bias), the
derivative of that sum and of the dropout's elementwise scale:

    dresidual = dz
    dinput    = dz * scale * mask
    dbias     = sum_rows dinput

Readings where the pages are silent (the fusion definitions show the
backward only): the forward is ``z = residual + mask * scale * (input +
bias)``, the post-attention bias-dropout-add; ``dz_extra`` is optional.
"""

import numpy as np


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def dropout_add(inp, residual, bias, mask, scale):
    """z = residual + mask * scale * (inp + bias), in float64.

    bias may be None (no bias); mask may be None (everything kept).
    """
    inp = _f64(inp)
    t = inp if bias is None else inp + _f64(bias)[None, :]
    if mask is not None:
        t = t * np.asarray(mask, dtype=np.float64)
    return _f64(residual) + float(scale) * t


def layer_norm_saved_stats(z, eps):
    """Setup helper: per-row mean and rstd = 1/sqrt(biased var + eps)."""
    z = _f64(z)
    mu = z.mean(axis=1)
    c = z - mu[:, None]
    var = (c * c).mean(axis=1)
    return mu, 1.0 / np.sqrt(var + eps)


def layer_norm_forward(z, gamma, beta, eps):
    """Training forward whose saved statistics (mean, rstd) the backward takes:
    ``y = (z - mean) * rstd * gamma + beta`` per row, with the biased
    variance.  gamma / beta may be None (ones / zeros).  Returns dict
    y [R, H], mean [R], rstd [R]."""
    z = _f64(z)
    H = z.shape[1]
    mu, rstd = layer_norm_saved_stats(z, eps)
    g = np.ones(H) if gamma is None else _f64(gamma)
    b = np.zeros(H) if beta is None else _f64(beta)
    centred = z - mu[:, None]
    y = centred * rstd[:, None] * g[None, :] + b[None, :]
    return {"y": y, "mean": mu, "rstd": rstd}


def fused_bias_dropout_add_layer_norm_forward(inp, residual, bias, mask, scale, gamma, beta,
                                              eps):
    """The forward whose backward is ``nvfuser_fusion_id9``: z = residual +
    mask * scale * (inp + bias) (the residual-stream output), then the
    LayerNorm of z.  Returns dict z, y [R, H], mean, rstd [R]."""
    z = dropout_add(inp, residual, bias, mask, scale)
    out = layer_norm_forward(z, gamma, beta, eps)
    out["z"] = z
    return out


def _ln_core(dy, z, mean, rstd, gamma, dz_extra):
    dy = _f64(dy)
    z = _f64(z)
    mu = _f64(mean)[:, None]
    rho = _f64(rstd)[:, None]
    gamma = _f64(gamma)[None, :]
    H = z.shape[1]

    centred = z - mu
    xhat = centred * rho
    g = dy * gamma
    dvar = -0.5 * (g * centred).sum(axis=1, keepdims=True) * rho * rho * rho
    dmean = -(g * rho).sum(axis=1, keepdims=True)
    dz = g * rho + 2.0 * dvar * centred / H + dmean / H
    if dz_extra is not None:
        dz = dz + _f64(dz_extra)
    dgamma = (dy * xhat).sum(axis=0)
    dbeta = dy.sum(axis=0)
    return dz, dgamma, dbeta


def layer_norm_backward(dy, x, mean, rstd, gamma, dz_extra=None):
    """Plain LayerNorm backward (nvfuser_fusion_id14).

    Returns dict dx [R, H] (includes dz_extra when given), dgamma, dbeta [H].
    """
    dz, dgamma, dbeta = _ln_core(dy, x, mean, rstd, gamma, dz_extra)
    return {"dx": dz, "dgamma": dgamma, "dbeta": dbeta}


def fused_bias_dropout_add_layer_norm_backward(dy, inp, residual, bias, mask,
                                               scale, mean, rstd, gamma,
                                               dz_extra=None):
    """Backward of LayerNorm(residual + dropout(inp + bias)) (fusion_id9).

    The LayerNorm input z is recomputed from (inp, residual, bias, mask,
    scale).  Returns dict dx (gradient of inp), dresidual, dbias, dgamma,
    dbeta.  bias may be None (then dbias is returned as None); mask may be
    None (everything kept).
    """
    z = dropout_add(inp, residual, bias, mask, scale)
    dz, dgamma, dbeta = _ln_core(dy, z, mean, rstd, gamma, dz_extra)
    dresidual = dz
    keep = 1.0 if mask is None else np.asarray(mask, dtype=np.float64)
    dx = dresidual * float(scale) * keep
    dbias = None if bias is None else dx.sum(axis=0)
    return {"dx": dx, "dresidual": dresidual, "dbias": dbias,
            "dgamma": dgamma, "dbeta": dbeta}


def layer_norm_backward_saved_z(dy, z, mask, scale, mean, rstd, gamma, dz_extra=None,
                                with_dbias=True):
    """The fused backward given the saved LayerNorm input z (the
    residual-stream output of the forward) instead of the operands that
    produced it: the same dz, dresidual = dz, dx = dz * scale * mask and
    dbias = sum_rows dx (nvfuser_fusion_id9 with the LayerNorm input read,
    not recomputed).
    mask may be None (everything kept).  Returns dict dx, dresidual, dbias
    (None unless with_dbias), dgamma, dbeta."""
    dz, dgamma, dbeta = _ln_core(dy, z, mean, rstd, gamma, dz_extra)
    keep = 1.0 if mask is None else np.asarray(mask, dtype=np.float64)
    dx = dz * float(scale) * keep
    return {"dx": dx, "dresidual": dz, "dbias": dx.sum(axis=0) if with_dbias else None,
            "dgamma": dgamma, "dbeta": dbeta}
