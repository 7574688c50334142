"""Plant plausible mistakes in copies of the oracle; the pins must catch each.

Each mutant is the oracle module's source with one textual change (a dropped
term, a flipped sign, a wrong axis, an operand swapped), compiled into a
fresh module.  The real oracle passes every pin (test_oracle_pins.py); a
mutant that passes them all would mean the pins cannot tell that mistake
apart from the truth.  Nothing here touches the GPU or the library.
"""

import inspect
import types

import pytest

from oracle import bn as obn, rmsnorm as orms, layernorm as oln

from . import pins

MUTATIONS = [
    # BatchNorm
    (obn, pins.BN_PINS, "k2 = -scale * dbeta / M", "k2 = scale * dbeta / M"),
    (obn, pins.BN_PINS, "k1 = -scale * inv_std * inv_std * sum_dy_xc / M",
     "k1 = -scale * inv_std * sum_dy_xc / M"),
    (obn, pins.BN_PINS, "dgamma = sum_dy_xc * inv_std", "dgamma = sum_dy_xc"),
    (obn, pins.BN_PINS, "dbeta = dy3.sum(axis=(0, 2))",
     "dbeta = dy3.sum(axis=(0, 2)) / M"),
    (obn, pins.BN_PINS, "+ m * var * (M / (M - 1.0))", "+ m * var"),
    (obn, pins.BN_PINS, "y = centred * _channel(scale) + _channel(beta)",
     "y = x3 * _channel(scale) + _channel(beta)"),
    (obn, pins.BN_PINS, "var = (centred * centred).sum(axis=(0, 2)) / M",
     "var = (centred * centred).sum(axis=(0, 2)) / (M - 1)"),
    (obn, pins.BN_PINS, "dx = dy3 * _channel(scale) + centred * _channel(k1)",
     "dx = dy3 * _channel(gamma) + centred * _channel(k1)"),
    (obn, pins.BN_PINS, "new_rm = (1.0 - m) * np.asarray(running_mean, np.float64) + m * mean",
     "new_rm = m * np.asarray(running_mean, np.float64) + (1.0 - m) * mean"),
    (obn, pins.BN_PINS, "return np.where(pre > 0, 1.0, float(slope))",
     "return np.where(pre > 0, 1.0, 0.0)"),
    (obn, pins.BN_PINS, "gated = np.asarray(dy, dtype=np.float64) * activation_gate(pre, act, slope)",
     "gated = np.asarray(dy, dtype=np.float64)"),
    (obn, pins.BN_PINS, "return np.where(pre > 0, pre, float(slope) * pre)",
     "return np.where(pre > 0, pre, 0.0)"),
    (obn, pins.BN_PINS, "return np.moveaxis(np.asarray(a, dtype=np.float64), -1, 1)",
     "return np.asarray(a, dtype=np.float64).reshape(np.shape(a)[0], np.shape(a)[-1], -1)"),
    (obn, pins.BN_PINS, 'out["dx"] = _to_channel_last(out["dx"])',
     'out["dx"] = out["dx"].reshape(np.shape(x))'),
    # RMSNorm
    (orms, pins.RMS_PINS, "x * (rstd3 * row_sum / H)", "x * (rstd3 * row_sum)"),
    (orms, pins.RMS_PINS, "rstd3 = rstd * rstd * rstd", "rstd3 = rstd * rstd"),
    (orms, pins.RMS_PINS, "dw = (dy * x * rstd[:, None]).sum(axis=0)",
     "dw = (dy * x).sum(axis=0)"),
    (orms, pins.RMS_PINS, "row_sum = (w[None, :] * dy * x).sum(axis=1)",
     "row_sum = (dy * x).sum(axis=1)"),
    (orms, pins.RMS_PINS, "rstd[:, None] * w[None, :] * dy - x",
     "rstd[:, None] * w[None, :] * dy + x"),
    # LayerNorm
    (oln, pins.LN_PINS, "+ dmean / H", "- dmean / H"),
    (oln, pins.LN_PINS, "dvar = -0.5 *", "dvar = 0.5 *"),
    (oln, pins.LN_PINS, "dx = dresidual * float(scale) * keep",
     "dx = dresidual * keep"),
    (oln, pins.LN_PINS, "dgamma = (dy * xhat).sum(axis=0)",
     "dgamma = (dy * centred).sum(axis=0)"),
    (oln, pins.LN_PINS, "dz = dz + _f64(dz_extra)", "dz = dz"),
    (oln, pins.LN_PINS, "t = t * np.asarray(mask, dtype=np.float64)", "t = t"),
    (oln, pins.LN_PINS, "g = dy * gamma", "g = dy"),
    (oln, pins.LN_PINS, "dbias = None if bias is None else dx.sum(axis=0)",
     "dbias = None if bias is None else dresidual.sum(axis=0)"),
    # forwards
    (orms, pins.RMS_PINS, "y = x * rstd[:, None] * wv[None, :]", "y = x * rstd[:, None]"),
    (orms, pins.RMS_PINS, "return 1.0 / np.sqrt((x * x).mean(axis=1) + eps)",
     "return 1.0 / np.sqrt((x * x).mean(axis=1))"),
    (oln, pins.LN_PINS, "y = centred * rstd[:, None] * g[None, :] + b[None, :]",
     "y = centred * rstd[:, None] * g[None, :]"),
    (oln, pins.LN_PINS, "return mu, 1.0 / np.sqrt(var + eps)", "return mu, 1.0 / np.sqrt(var)"),
    (oln, pins.LN_PINS, "var = (c * c).mean(axis=1)", "var = (c * c).sum(axis=1) / (z.shape[1] - 1)"),
    (oln, pins.LN_PINS, "    dx = dz * float(scale) * keep\n", "    dx = dz * keep\n"),
    (oln, pins.LN_PINS, '"dbias": dx.sum(axis=0) if with_dbias else None',
     '"dbias": dz.sum(axis=0) if with_dbias else None'),
]


def _mutant(module, old, new):
    src = inspect.getsource(module)
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType(module.__name__ + "_mutant")
    exec(compile(src.replace(old, new, 1), f"<mutant {old}>", "exec"),
         mod.__dict__)
    return mod


@pytest.mark.parametrize("module,pin_list,old,new", MUTATIONS,
                         ids=[m[2][:40] for m in MUTATIONS])
def test_mutant_is_caught(module, pin_list, old, new):
    pytest.importorskip("sympy")
    mod = _mutant(module, old, new)
    caught = []
    for pin in pin_list:
        try:
            pin(mod)
        except AssertionError as e:
            caught.append(f"{pin.__name__}: {e}")
    assert caught, f"mutant {old!r} -> {new!r} passed every pin"
