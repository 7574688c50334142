"""RMSNorm backward in float64 (oracle).

Test infrastructure only; see ``oracle/__init__.py``.

Source: nvFuser issue #3629, "Performance gap between manual nvfuser
definition and thunder.jit for rmsnorm".

* Forward (section with ``rmsnorm_prims`` / ``F.rms_norm``):
  ``y = w * x / sqrt(mean(x^2, dim=1) + eps)`` (``rms_norm_forward``).
* Backward (section "nvfuser pre-generated definition", ``rmsnorm_bwd_fusion``):
  with the saved per-row statistic, ``dx = dy*w/rms - x * sum(dy*w*x) /
  (H * rms^3)`` and ``dweight = sum over rows of dy * x / rms``.

The pages save either rms (the nvFuser benchmark definition) or 1/rms (the
Thunder definition).  This oracle, like the library, takes the reciprocal
``rstd = 1/rms`` as its input, so the backward reads

    S_r    = sum_j w_j * dy_rj * x_rj
    dx_rj  = rstd_r * w_j * dy_rj - x_rj * rstd_r^3 * S_r / H
    dw_j   = sum_r dy_rj * x_rj * rstd_r
"""

import numpy as np


def rms_norm_rstd(x, eps):
    """Setup helper: the saved statistic rstd = 1/sqrt(mean(x^2) + eps) per row."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt((x * x).mean(axis=1) + eps)


def rms_norm_forward(x, w, eps):
    """Training forward (the ``rmsnorm_prims`` / ``F.rms_norm`` section):
    ``y = w * x * rstd`` with ``rstd = 1/sqrt(mean(x^2) + eps)`` per row.

    x: [R, H]; w: [H] or None (all ones).  Returns dict y [R, H], rstd [R]
    (the statistic the backward takes)."""
    x = np.asarray(x, dtype=np.float64)
    rstd = rms_norm_rstd(x, eps)
    wv = np.ones(x.shape[1]) if w is None else np.asarray(w, dtype=np.float64)
    y = x * rstd[:, None] * wv[None, :]
    return {"y": y, "rstd": rstd}


def rms_norm_backward(x, dy, w, rstd):
    """x, dy: [R, H]; w: [H]; rstd: [R].  Returns dict dx [R, H], dw [H]."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    rstd = np.asarray(rstd, dtype=np.float64)
    H = x.shape[1]

    row_sum = (w[None, :] * dy * x).sum(axis=1)
    rstd3 = rstd * rstd * rstd
    dx = rstd[:, None] * w[None, :] * dy - x * (rstd3 * row_sum / H)[:, None]
    dw = (dy * x * rstd[:, None]).sum(axis=0)
    return {"dx": dx, "dw": dw}
