"""BatchNorm2d training forward / apply / backward in float64 (oracle).

Test infrastructure only; see ``oracle/__init__.py``.

Sources
-------
Aether-ML PR #18, "perf(batchnorm): device-sized grid, one-pass statistics,
finalize kernels":

* section "One-pass statistics": the forward finalize writes per channel
  (mean, var, inv_std, gamma * inv_std) and updates running_mean and
  running_var in place; the apply is ``out = (x - mean) * scale + beta`` and
  is shared by training and inference.
* section "Backward finalize": grads = (dgamma, dbeta, k1, k2) with
  ``k1 = -scale * inv_std^2 * sum(dy * (x - mean)) / N``,
  ``k2 = -scale * dbeta / N`` and ``dx = dy * scale + (x - mean) * k1 + k2``.

The one-pass shifted sums and the partials are how the GPU reaches these
numbers; the quantities themselves have plain definitions, so this file
writes the definitions out (two-pass variance, float64, no shift).

Readings where the pages are silent
-----------------------------------
* ``N`` in k1/k2 is the per-channel element count ``M = B * H * W``.
* The batch variance is biased (divides by M), as in the test of Aether-ML
  PR #18 ("Testing") that compares it with "the float64 variance of the same data".
* running_var takes the unbiased ``var * M / (M - 1)``; momentum follows
  ``new = (1 - m) * old + m * batch`` (the PyTorch BatchNorm2d convention).
* Fusing ReLU / LeakyReLU into BatchNorm is "Part 2" of Aether-ML PR #18
  (section "Context"; "Follow-ups": ReLU costs more per step than the BatchNorm
  forward).  That page gives no definition beyond the names, so the reading
  here is the composition: y = act(pre) with pre the BatchNorm output, and
  the backward gates dy by d act / d pre -- 1 where pre > 0, else 0 (ReLU)
  or the negative slope (LeakyReLU) -- before the BatchNorm backward.
"""

import numpy as np


def _bcs(x):
    """View an NC... array as float64 [B, C, S] with S = product of the rest."""
    x = np.asarray(x, dtype=np.float64)
    if x.ndim < 2:
        raise ValueError("batch norm input needs at least 2 dims (N, C, ...)")
    return x.reshape(x.shape[0], x.shape[1], -1)


def _channel(v):
    """Broadcast a per-channel vector [C] against [B, C, S]."""
    return np.asarray(v, dtype=np.float64)[None, :, None]


def batch_norm_forward_train(x, gamma, beta, running_mean, running_var,
                             momentum, eps):
    """Training-mode forward.  Returns a dict of float64 arrays.

    x: [B, C, ...]; gamma, beta, running_mean, running_var: [C].
    Keys: y (shape of x), mean, var, inv_std, scale, running_mean,
    running_var (all [C]).
    """
    x3 = _bcs(x)
    B, C, S = x3.shape
    M = B * S
    gamma = np.asarray(gamma, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)

    mean = x3.sum(axis=(0, 2)) / M
    centred = x3 - _channel(mean)
    var = (centred * centred).sum(axis=(0, 2)) / M
    inv_std = 1.0 / np.sqrt(var + eps)
    scale = gamma * inv_std
    y = centred * _channel(scale) + _channel(beta)

    m = float(momentum)
    new_rm = (1.0 - m) * np.asarray(running_mean, np.float64) + m * mean
    new_rv = (1.0 - m) * np.asarray(running_var, np.float64) \
        + m * var * (M / (M - 1.0))
    return {
        "y": y.reshape(np.shape(x)),
        "mean": mean,
        "var": var,
        "inv_std": inv_std,
        "scale": scale,
        "running_mean": new_rm,
        "running_var": new_rv,
    }


def batch_norm_apply(x, mean, scale, beta):
    """Centred apply ``(x - mean) * scale + beta`` (inference form)."""
    x3 = _bcs(x)
    y = (x3 - _channel(mean)) * _channel(scale) + _channel(beta)
    return y.reshape(np.shape(x))


def batch_norm_backward(x, dy, gamma, eps):
    """Training-mode backward given the forward's input.

    mean and inv_std are recomputed from x in float64.  Returns a dict:
    dx (shape of x), dgamma, dbeta, k1, k2 (all [C]).
    """
    x3 = _bcs(x)
    dy3 = _bcs(dy)
    B, C, S = x3.shape
    M = B * S
    gamma = np.asarray(gamma, dtype=np.float64)

    mean = x3.sum(axis=(0, 2)) / M
    centred = x3 - _channel(mean)
    var = (centred * centred).sum(axis=(0, 2)) / M
    inv_std = 1.0 / np.sqrt(var + eps)
    scale = gamma * inv_std

    dbeta = dy3.sum(axis=(0, 2))
    sum_dy_xc = (dy3 * centred).sum(axis=(0, 2))
    dgamma = sum_dy_xc * inv_std
    k1 = -scale * inv_std * inv_std * sum_dy_xc / M
    k2 = -scale * dbeta / M
    dx = dy3 * _channel(scale) + centred * _channel(k1) + _channel(k2)
    return {
        "dx": dx.reshape(np.shape(x)),
        "dgamma": dgamma,
        "dbeta": dbeta,
        "k1": k1,
        "k2": k2,
    }


ACT_NONE, ACT_RELU, ACT_LEAKY_RELU = 0, 1, 2


def activation(pre, act, slope=0.0):
    """ReLU max(pre, 0), LeakyReLU (pre if pre > 0 else slope * pre), or pre."""
    pre = np.asarray(pre, dtype=np.float64)
    if act == ACT_RELU:
        return np.where(pre > 0, pre, 0.0)
    if act == ACT_LEAKY_RELU:
        return np.where(pre > 0, pre, float(slope) * pre)
    return pre


def activation_gate(pre, act, slope=0.0):
    """d act / d pre: 1 where pre > 0, else 0 (ReLU) or slope (LeakyReLU)."""
    pre = np.asarray(pre, dtype=np.float64)
    if act == ACT_RELU:
        return np.where(pre > 0, 1.0, 0.0)
    if act == ACT_LEAKY_RELU:
        return np.where(pre > 0, 1.0, float(slope))
    return np.ones_like(pre)


def batch_norm_act_forward_train(x, gamma, beta, running_mean, running_var, momentum, eps, act,
                                 slope=0.0):
    """Training forward of act(BatchNorm(x)).  The dict of
    batch_norm_forward_train with y = act(pre) and pre = the BatchNorm output."""
    out = batch_norm_forward_train(x, gamma, beta, running_mean, running_var, momentum, eps)
    out["pre"] = out["y"]
    out["y"] = activation(out["pre"], act, slope)
    return out


def batch_norm_act_backward(x, dy, gamma, beta, eps, act, slope=0.0):
    """Backward of act(BatchNorm(x)) given the forward's input: pre is
    recomputed from x, dy is gated by d act / d pre, then the BatchNorm
    backward.  Returns the dict of batch_norm_backward plus pre."""
    C = np.asarray(gamma).shape[0]
    pre = batch_norm_forward_train(x, gamma, beta, np.zeros(C), np.ones(C), 0.0, eps)["y"]
    gated = np.asarray(dy, dtype=np.float64) * activation_gate(pre, act, slope)
    out = batch_norm_backward(x, gated, gamma, eps)
    out["pre"] = pre
    return out


# Channels-last (NHWC) BatchNorm: the same definition with the channel as the
# last axis.  x is [..., C]; the channel axis is moved to position 1 and back.

def _to_channel_first(a):
    return np.moveaxis(np.asarray(a, dtype=np.float64), -1, 1)


def _to_channel_last(a):
    return np.moveaxis(a, 1, -1)


def batch_norm_nhwc_forward_train(x, gamma, beta, running_mean, running_var, momentum, eps,
                                  act=ACT_NONE, slope=0.0):
    """Training forward of act(BatchNorm(x)) for a channels-last x [..., C].
    Returns the dict of batch_norm_forward_train (y channels-last)."""
    out = batch_norm_act_forward_train(_to_channel_first(x), gamma, beta, running_mean,
                                       running_var, momentum, eps, act, slope)
    out["y"] = _to_channel_last(out["y"])
    out["pre"] = _to_channel_last(out["pre"])
    return out


def batch_norm_nhwc_backward(x, dy, gamma, beta, eps, act=ACT_NONE, slope=0.0):
    """Backward of act(BatchNorm(x)) for channels-last x, dy [..., C]."""
    out = batch_norm_act_backward(_to_channel_first(x), _to_channel_first(dy), gamma, beta, eps,
                                  act, slope)
    out["dx"] = _to_channel_last(out["dx"])
    out["pre"] = _to_channel_last(out["pre"])
    return out
