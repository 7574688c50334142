"""Checks that pin the float64 oracle to things other than itself.

Each ``pin_*`` function takes the oracle module under test (the real one or a
deliberately mutated copy) and raises ``AssertionError`` when it disagrees
with an independent source:

* PyTorch float64 autograd of ``F.batch_norm`` / ``F.layer_norm`` /
  ``F.rms_norm`` (a separate implementation of the same operations);
* central finite differences of the oracle's own forward (the backward must
  be its gradient);
* closed-form invariants of the gradients;
* exact rational arithmetic with sympy (symbolic differentiation).

``tests/test_oracle_pins.py`` runs them on the real oracle, and
``tests/test_oracle_mutants.py`` checks that every planted mistake is caught.
"""

import numpy as np
import torch
import torch.nn.functional as F

RTOL = 1e-10


def _close(a, b, rtol=RTOL, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= atol + rtol * scale, f"{what}: max abs err {err:.3e}"


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- BatchNorm

def _bn_data(seed, shape=(4, 3, 5, 6), offset=0.0):
    r = _rng(seed)
    C = shape[1]
    mu = r.uniform(-offset, offset, C) if offset else np.zeros(C)
    sig = r.uniform(0.3, 2.0, C)
    x = mu[None, :, None, None] + sig[None, :, None, None] * r.standard_normal(shape)
    gamma = r.uniform(0.5, 1.5, C)
    beta = r.normal(0.0, 0.1, C)
    dy = r.standard_normal(shape)
    rm = r.normal(0, 1, C)
    rv = r.uniform(0.5, 2.0, C)
    return x, gamma, beta, dy, rm, rv


def pin_bn_forward_vs_torch(bn):
    for seed, offset in ((1, 0.0), (2, 500.0)):
        x, gamma, beta, _, rm, rv = _bn_data(seed, offset=offset)
        eps, mom = 1e-5, 0.1
        out = bn.batch_norm_forward_train(x, gamma, beta, rm, rv, mom, eps)
        trm, trv = torch.tensor(rm), torch.tensor(rv)
        ty, tmean, tinvstd = torch.native_batch_norm(
            torch.tensor(x), torch.tensor(gamma), torch.tensor(beta),
            trm, trv, True, mom, eps)
        _close(out["y"], ty.numpy(), what="bn y")
        _close(out["mean"], tmean.numpy(), what="bn mean")
        _close(out["inv_std"], tinvstd.numpy(), what="bn inv_std")
        _close(out["scale"], gamma * tinvstd.numpy(), what="bn scale")
        _close(out["running_mean"], trm.numpy(), what="bn running_mean")
        _close(out["running_var"], trv.numpy(), what="bn running_var")
        torch_var = torch.tensor(x).transpose(0, 1).reshape(
            x.shape[1], -1).var(dim=1, unbiased=False)
        _close(out["var"], torch_var.numpy(), what="bn var")
        y2 = bn.batch_norm_apply(x, out["mean"], out["scale"], beta)
        _close(y2, ty.numpy(), what="bn apply")


def pin_bn_backward_vs_torch(bn):
    for seed, offset in ((3, 0.0), (4, 300.0)):
        x, gamma, beta, dy, _, _ = _bn_data(seed, offset=offset)
        eps = 1e-5
        tx = torch.tensor(x, requires_grad=True)
        tg = torch.tensor(gamma, requires_grad=True)
        tb = torch.tensor(beta, requires_grad=True)
        y = F.batch_norm(tx, None, None, tg, tb, training=True, eps=eps)
        y.backward(torch.tensor(dy))
        out = bn.batch_norm_backward(x, dy, gamma, eps)
        _close(out["dx"], tx.grad.numpy(), what="bn dx")
        _close(out["dgamma"], tg.grad.numpy(), what="bn dgamma")
        _close(out["dbeta"], tb.grad.numpy(), what="bn dbeta")


def pin_bn_finite_differences(bn):
    x, gamma, beta, dy, rm, rv = _bn_data(5, shape=(2, 3, 2, 2))
    eps, h = 1e-3, 1e-6

    def loss(xv, gv, bv):
        y = bn.batch_norm_forward_train(xv, gv, bv, rm, rv, 0.1, eps)["y"]
        return float((y * dy).sum())

    out = bn.batch_norm_backward(x, dy, gamma, eps)
    fd_x = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd_x[idx] = (loss(xp, gamma, beta) - loss(xm, gamma, beta)) / (2 * h)
    fd_g = np.zeros_like(gamma)
    fd_b = np.zeros_like(beta)
    for c in range(gamma.size):
        gp, gm = gamma.copy(), gamma.copy()
        gp[c] += h
        gm[c] -= h
        fd_g[c] = (loss(x, gp, beta) - loss(x, gm, beta)) / (2 * h)
        bp, bm = beta.copy(), beta.copy()
        bp[c] += h
        bm[c] -= h
        fd_b[c] = (loss(x, gamma, bp) - loss(x, gamma, bm)) / (2 * h)
    _close(out["dx"], fd_x, rtol=1e-6, what="bn FD dx")
    _close(out["dgamma"], fd_g, rtol=1e-6, what="bn FD dgamma")
    _close(out["dbeta"], fd_b, rtol=1e-6, what="bn FD dbeta")


def pin_bn_invariants(bn):
    x, gamma, beta, dy, rm, rv = _bn_data(6, shape=(5, 4, 3, 7), offset=50.0)
    eps = 0.3  # large eps so the eps-dependent identities are not trivial
    f = bn.batch_norm_forward_train(x, gamma, beta, rm, rv, 0.1, eps)
    b = bn.batch_norm_backward(x, dy, gamma, eps)
    xc = x - x.mean(axis=(0, 2, 3), keepdims=True)
    var = (xc * xc).mean(axis=(0, 2, 3))
    scale = gamma / np.sqrt(var + eps)
    S = (dy * xc).sum(axis=(0, 2, 3))
    # sum_{b,h,w} dx = 0 per channel
    _close(b["dx"].sum(axis=(0, 2, 3)), np.zeros_like(gamma), atol=1e-9,
           what="sum dx")
    # sum dx * (x - mean) = scale * S * eps / (var + eps)
    _close((b["dx"] * xc).sum(axis=(0, 2, 3)), scale * S * eps / (var + eps),
           what="sum dx*xc")
    _close(b["dbeta"], dy.sum(axis=(0, 2, 3)), what="dbeta = sum dy")
    # dy = 1 everywhere shifts y by a constant per channel, which the
    # normalisation removes: dx must vanish.
    ones = np.ones_like(dy)
    b1 = bn.batch_norm_backward(x, ones, gamma, eps)
    _close(b1["dx"], np.zeros_like(dy), atol=1e-9, what="dx for dy=1")
    # mean(y) = beta, var(y) = gamma^2 var / (var + eps)
    y = f["y"]
    _close(y.mean(axis=(0, 2, 3)), beta, atol=1e-12, what="mean y")
    _close(y.var(axis=(0, 2, 3)), gamma ** 2 * var / (var + eps),
           what="var y")


def pin_bn_running_ema(bn):
    x, gamma, beta, _, rm0, rv0 = _bn_data(7, shape=(3, 2, 4, 5), offset=10.0)
    m, eps, k = 0.1, 1e-5, 7
    M = x.shape[0] * x.shape[2] * x.shape[3]
    mean = x.mean(axis=(0, 2, 3))
    var_unb = x.var(axis=(0, 2, 3), ddof=1)
    rm, rv = rm0.copy(), rv0.copy()
    for _ in range(k):
        out = bn.batch_norm_forward_train(x, gamma, beta, rm, rv, m, eps)
        rm, rv = out["running_mean"], out["running_var"]
    decay = (1 - m) ** k
    _close(rm, decay * rm0 + (1 - decay) * mean, what="running_mean EMA")
    _close(rv, decay * rv0 + (1 - decay) * var_unb, what="running_var EMA")
    assert M > 1


def pin_bn_exact_rational(bn):
    sympy = __import__("sympy")
    R = sympy.Rational
    xs = [[R(3), R(-1)], [R(2), R(5)]]        # [B=2, C=1, HW=2] flattened
    dys = [[R(1), R(-2)], [R(1, 2), R(3)]]
    g, bt, eps = R(3, 2), R(-1, 10), R(1, 4)
    syms = sympy.symbols("x0:4")
    flat = list(syms)
    M = 4
    mu = sum(flat) / M
    var = sum((v - mu) ** 2 for v in flat) / M
    ys = [(v - mu) / sympy.sqrt(var + eps) * g + bt for v in flat]
    dflat = [dys[0][0], dys[0][1], dys[1][0], dys[1][1]]
    L = sum(yv * d for yv, d in zip(ys, dflat))
    subs = dict(zip(syms, [xs[0][0], xs[0][1], xs[1][0], xs[1][1]]))
    grad = [float(sympy.N(sympy.diff(L, s).subs(subs), 30)) for s in syms]
    yvals = [float(sympy.N(yv.subs(subs), 30)) for yv in ys]
    gsym, bsym = sympy.symbols("g b")
    Lg = sum(((v - mu) / sympy.sqrt(var + eps) * gsym + bsym) * d
             for v, d in zip(flat, dflat))
    dgamma = float(sympy.N(sympy.diff(Lg, gsym).subs(subs), 30))
    x = np.array([[[3.0, -1.0]], [[2.0, 5.0]]])
    dy = np.array([[[1.0, -2.0]], [[0.5, 3.0]]])
    f = bn.batch_norm_forward_train(x, [1.5], [-0.1], [0.0], [1.0], 0.1, 0.25)
    b = bn.batch_norm_backward(x, dy, [1.5], 0.25)
    _close(f["y"].reshape(-1), yvals, rtol=1e-13, what="exact y")
    _close(b["dx"].reshape(-1), grad, rtol=1e-13, what="exact dx")
    _close(b["dgamma"], [dgamma], rtol=1e-13, what="exact dgamma")


def pin_bn_act_vs_torch(bn):
    """act(BatchNorm) forward and backward against torch float64 autograd of
    F.relu / F.leaky_relu(F.batch_norm(...))."""
    x, gamma, beta, dy, rm, rv = _bn_data(31, offset=20.0)
    beta = beta + np.linspace(-0.8, 0.8, beta.size)  # both signs of pre in every channel
    eps = 1e-5
    for act, slope, fn in ((bn.ACT_RELU, 0.0, lambda t: F.relu(t)),
                           (bn.ACT_LEAKY_RELU, 0.1, lambda t: F.leaky_relu(t, 0.1))):
        tx = torch.tensor(x, requires_grad=True)
        tg = torch.tensor(gamma, requires_grad=True)
        tb = torch.tensor(beta, requires_grad=True)
        y = fn(F.batch_norm(tx, None, None, tg, tb, training=True, eps=eps))
        y.backward(torch.tensor(dy))
        f = bn.batch_norm_act_forward_train(x, gamma, beta, rm, rv, 0.1, eps, act, slope)
        _close(f["y"], y.detach().numpy(), what=f"act {act} y")
        b = bn.batch_norm_act_backward(x, dy, gamma, beta, eps, act, slope)
        _close(b["dx"], tx.grad.numpy(), what=f"act {act} dx")
        _close(b["dgamma"], tg.grad.numpy(), what=f"act {act} dgamma")
        _close(b["dbeta"], tb.grad.numpy(), what=f"act {act} dbeta")


def pin_bn_nhwc_vs_torch(bn):
    """Channels-last BatchNorm (x [N, H, W, C]) against torch float64 autograd
    of F.batch_norm on the same data permuted by torch to [N, C, H, W]; all
    four sizes differ, so a wrong axis fails on shape or values."""
    r = _rng(41)
    N, H, W, C = 3, 4, 5, 6
    x = r.standard_normal((N, H, W, C)) * r.uniform(0.5, 2.0, C) + r.uniform(-5, 5, C)
    dy = r.standard_normal((N, H, W, C))
    gamma, beta = r.uniform(0.5, 1.5, C), r.uniform(-0.5, 0.5, C)
    eps = 1e-5
    for act, slope, fn in ((bn.ACT_NONE, 0.0, lambda t: t),
                           (bn.ACT_RELU, 0.0, lambda t: F.relu(t))):
        tx = torch.tensor(x, requires_grad=True)
        tg = torch.tensor(gamma, requires_grad=True)
        tb = torch.tensor(beta, requires_grad=True)
        y = fn(F.batch_norm(tx.permute(0, 3, 1, 2), None, None, tg, tb, training=True, eps=eps))
        y.permute(0, 2, 3, 1).backward(torch.tensor(dy))
        f = bn.batch_norm_nhwc_forward_train(x, gamma, beta, np.zeros(C), np.ones(C), 0.1, eps,
                                             act, slope)
        _close(f["y"], y.permute(0, 2, 3, 1).detach().numpy(), what=f"nhwc {act} y")
        b = bn.batch_norm_nhwc_backward(x, dy, gamma, beta, eps, act, slope)
        _close(b["dx"], tx.grad.numpy(), what=f"nhwc {act} dx")
        _close(b["dgamma"], tg.grad.numpy(), what=f"nhwc {act} dgamma")
        _close(b["dbeta"], tb.grad.numpy(), what=f"nhwc {act} dbeta")


BN_PINS = [pin_bn_forward_vs_torch, pin_bn_backward_vs_torch,
           pin_bn_finite_differences, pin_bn_invariants, pin_bn_running_ema,
           pin_bn_exact_rational, pin_bn_act_vs_torch, pin_bn_nhwc_vs_torch]


# ------------------------------------------------------------------ RMSNorm

def _rms_data(seed, R=6, H=11):
    r = _rng(seed)
    x = r.standard_normal((R, H)) * r.uniform(0.2, 3.0, (R, 1))
    dy = r.standard_normal((R, H))
    w = r.uniform(0.5, 1.5, H)
    return x, dy, w


def pin_rms_vs_torch(rms):
    x, dy, w = _rms_data(11)
    eps = 1e-5
    tx = torch.tensor(x, requires_grad=True)
    tw = torch.tensor(w, requires_grad=True)
    y = F.rms_norm(tx, (x.shape[1],), tw, eps=eps)
    y.backward(torch.tensor(dy))
    rstd = rms.rms_norm_rstd(x, eps)
    _close(x * rstd[:, None] * w[None, :], y.detach().numpy(), what="rms fwd")
    out = rms.rms_norm_backward(x, dy, w, rstd)
    _close(out["dx"], tx.grad.numpy(), what="rms dx")
    _close(out["dw"], tw.grad.numpy(), what="rms dw")


def pin_rms_finite_differences(rms):
    x, dy, w = _rms_data(12, R=3, H=7)
    eps, h = 1e-2, 1e-6

    def loss(xv, wv):
        rstd = rms.rms_norm_rstd(xv, eps)
        return float((xv * rstd[:, None] * wv[None, :] * dy).sum())

    out = rms.rms_norm_backward(x, dy, w, rms.rms_norm_rstd(x, eps))
    fd_x = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd_x[idx] = (loss(xp, w) - loss(xm, w)) / (2 * h)
    fd_w = np.zeros_like(w)
    for j in range(w.size):
        wp, wm = w.copy(), w.copy()
        wp[j] += h
        wm[j] -= h
        fd_w[j] = (loss(x, wp) - loss(x, wm)) / (2 * h)
    _close(out["dx"], fd_x, rtol=1e-6, what="rms FD dx")
    _close(out["dw"], fd_w, rtol=1e-6, what="rms FD dw")


def pin_rms_invariants(rms):
    x, dy, w = _rms_data(13, R=5, H=9)
    eps = 0.2
    rstd = rms.rms_norm_rstd(x, eps)
    out = rms.rms_norm_backward(x, dy, w, rstd)
    ms = (x * x).mean(axis=1)
    S = (w[None, :] * dy * x).sum(axis=1)
    # sum_j x_j dx_j = rstd * S * eps / (ms + eps)
    _close((x * out["dx"]).sum(axis=1), rstd * S * eps / (ms + eps),
           what="sum x*dx")
    # w = 1, dy = x: dx = rstd * x * (1 - rstd^2 * ms) = rstd * x * eps/(ms+eps)
    ones = np.ones_like(w)
    o2 = rms.rms_norm_backward(x, x, ones, rstd)
    _close(o2["dx"], x * (rstd * eps / (ms + eps))[:, None], what="dx, dy=x")


def pin_rms_exact_rational(rms):
    sympy = __import__("sympy")
    R = sympy.Rational
    xs = [R(1), R(-2), R(3, 2)]
    dys = [R(2), R(1, 2), R(-1)]
    ws = [R(1, 2), R(2), R(1)]
    eps = R(1, 10)
    syms = sympy.symbols("x0:3")
    ms = sum(s * s for s in syms) / 3
    L = sum(s / sympy.sqrt(ms + eps) * wv * d
            for s, wv, d in zip(syms, ws, dys))
    subs = dict(zip(syms, xs))
    grad = [float(sympy.N(sympy.diff(L, s).subs(subs), 30)) for s in syms]
    x = np.array([[1.0, -2.0, 1.5]])
    out = rms.rms_norm_backward(x, np.array([[2.0, 0.5, -1.0]]),
                                np.array([0.5, 2.0, 1.0]),
                                rms.rms_norm_rstd(x, 0.1))
    _close(out["dx"][0], grad, rtol=1e-13, what="exact rms dx")


def pin_rms_forward(rms):
    """The training forward against torch's float64 F.rms_norm, and the
    closed form mean(y^2) = ms / (ms + eps) for unit weights."""
    x, _, w = _rms_data(14, R=5, H=10)
    eps = 0.05
    out = rms.rms_norm_forward(x, w, eps)
    ty = F.rms_norm(torch.tensor(x), (x.shape[1],), torch.tensor(w), eps=eps)
    _close(out["y"], ty.numpy(), what="rms forward y vs torch")
    o1 = rms.rms_norm_forward(x, None, eps)
    ms = (x * x).mean(axis=1)
    _close((o1["y"] ** 2).mean(axis=1), ms / (ms + eps), what="mean y^2")
    _close(o1["y"], x * o1["rstd"][:, None], what="unit weights: y = x*rstd")


RMS_PINS = [pin_rms_vs_torch, pin_rms_finite_differences, pin_rms_invariants,
            pin_rms_exact_rational, pin_rms_forward]


# ---------------------------------------------------------------- LayerNorm

def _ln_data(seed, R=5, H=13):
    r = _rng(seed)
    inp = r.standard_normal((R, H))
    res = r.standard_normal((R, H)) * 2.0 + 0.3
    bias = r.standard_normal(H)
    mask = (r.uniform(size=(R, H)) < 0.8).astype(np.float64)
    gamma = r.uniform(0.5, 1.5, H)
    beta = r.normal(0, 0.1, H)
    dy = r.standard_normal((R, H))
    dzx = r.standard_normal((R, H))
    return inp, res, bias, mask, gamma, beta, dy, dzx


def pin_ln_plain_vs_torch(ln):
    inp, _, _, _, gamma, beta, dy, dzx = _ln_data(21)
    eps = 1e-5
    H = inp.shape[1]
    tx = torch.tensor(inp, requires_grad=True)
    tg = torch.tensor(gamma, requires_grad=True)
    tb = torch.tensor(beta, requires_grad=True)
    y = F.layer_norm(tx, (H,), tg, tb, eps)
    y.backward(torch.tensor(dy))
    mu, rstd = ln.layer_norm_saved_stats(inp, eps)
    out = ln.layer_norm_backward(dy, inp, mu, rstd, gamma)
    _close(out["dx"], tx.grad.numpy(), what="ln dx")
    _close(out["dgamma"], tg.grad.numpy(), what="ln dgamma")
    _close(out["dbeta"], tb.grad.numpy(), what="ln dbeta")
    out2 = ln.layer_norm_backward(dy, inp, mu, rstd, gamma, dz_extra=dzx)
    _close(out2["dx"], tx.grad.numpy() + dzx, what="ln dx + extra")


def pin_ln_fused_vs_torch(ln):
    inp, res, bias, mask, gamma, beta, dy, dzx = _ln_data(22)
    eps, s = 1e-5, 1.0 / 0.8
    H = inp.shape[1]
    ti = torch.tensor(inp, requires_grad=True)
    tr = torch.tensor(res, requires_grad=True)
    tbias = torch.tensor(bias, requires_grad=True)
    tg = torch.tensor(gamma, requires_grad=True)
    tb = torch.tensor(beta, requires_grad=True)
    z = tr + torch.tensor(mask) * s * (ti + tbias)
    y = F.layer_norm(z, (H,), tg, tb, eps)
    loss = (y * torch.tensor(dy)).sum() + (z * torch.tensor(dzx)).sum()
    loss.backward()
    zz = ln.dropout_add(inp, res, bias, mask, s)
    _close(zz, z.detach().numpy(), what="dropout_add")
    mu, rstd = ln.layer_norm_saved_stats(zz, eps)
    out = ln.fused_bias_dropout_add_layer_norm_backward(
        dy, inp, res, bias, mask, s, mu, rstd, gamma, dz_extra=dzx)
    _close(out["dx"], ti.grad.numpy(), what="fused dx")
    _close(out["dresidual"], tr.grad.numpy(), what="fused dresidual")
    _close(out["dbias"], tbias.grad.numpy(), what="fused dbias")
    _close(out["dgamma"], tg.grad.numpy(), what="fused dgamma")
    _close(out["dbeta"], tb.grad.numpy(), what="fused dbeta")


def pin_ln_finite_differences(ln):
    inp, res, bias, mask, gamma, beta, dy, _ = _ln_data(23, R=3, H=5)
    eps, s, h = 1e-2, 1.25, 1e-6

    def loss(iv, rv, bv, gv):
        z = ln.dropout_add(iv, rv, bv, mask, s)
        mu, rstd = ln.layer_norm_saved_stats(z, eps)
        y = (z - mu[:, None]) * rstd[:, None] * gv[None, :] + beta[None, :]
        return float((y * dy).sum())

    z = ln.dropout_add(inp, res, bias, mask, s)
    mu, rstd = ln.layer_norm_saved_stats(z, eps)
    out = ln.fused_bias_dropout_add_layer_norm_backward(
        dy, inp, res, bias, mask, s, mu, rstd, gamma)

    def fd(arr, fn):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            g[idx] = (fn(p) - fn(m)) / (2 * h)
        return g

    _close(out["dx"], fd(inp, lambda a: loss(a, res, bias, gamma)),
           rtol=1e-6, what="ln FD dx")
    _close(out["dresidual"], fd(res, lambda a: loss(inp, a, bias, gamma)),
           rtol=1e-6, what="ln FD dresidual")
    _close(out["dbias"], fd(bias, lambda a: loss(inp, res, a, gamma)),
           rtol=1e-6, what="ln FD dbias")
    _close(out["dgamma"], fd(gamma, lambda a: loss(inp, res, bias, a)),
           rtol=1e-6, what="ln FD dgamma")


def pin_ln_invariants(ln):
    inp, res, bias, mask, gamma, beta, dy, _ = _ln_data(24, R=4, H=9)
    eps, s = 0.25, 1.5
    z = ln.dropout_add(inp, res, bias, mask, s)
    mu, rstd = ln.layer_norm_saved_stats(z, eps)
    out = ln.fused_bias_dropout_add_layer_norm_backward(
        dy, inp, res, bias, mask, s, mu, rstd, gamma)
    dz = out["dresidual"]
    xhat = (z - mu[:, None]) * rstd[:, None]
    g = dy * gamma[None, :]
    var = ((z - mu[:, None]) ** 2).mean(axis=1)
    _close(dz.sum(axis=1), np.zeros(z.shape[0]), atol=1e-9, what="sum dz")
    _close((dz * xhat).sum(axis=1),
           rstd * (g * xhat).sum(axis=1) * eps / (var + eps),
           what="sum dz*xhat")
    assert np.all(out["dx"][mask == 0] == 0.0), "dx must vanish where dropped"
    _close(out["dx"][mask == 1], dz[mask == 1] * s, what="dx = dres*s")
    _close(out["dbias"], out["dx"].sum(axis=0), what="dbias = sum dx")
    _close(out["dbeta"], dy.sum(axis=0), what="dbeta = sum dy")


def pin_ln_forward(ln):
    """The training forwards against torch's float64 native_layer_norm
    (which returns y, mean and rstd), the fused z against the same
    bias-dropout-add written in torch, and the closed forms of a unit-affine
    LayerNorm: zero row mean, mean(y^2) = var / (var + eps)."""
    inp, res, bias, mask, gamma, beta, _, _ = _ln_data(25, R=4, H=11)
    eps, s = 0.1, 1.25
    tz = (torch.tensor(res) + torch.tensor(mask) * s
          * (torch.tensor(inp) + torch.tensor(bias)[None, :]))
    ty, tmu, trstd = torch.native_layer_norm(tz, (inp.shape[1],), torch.tensor(gamma),
                                             torch.tensor(beta), eps)
    out = ln.fused_bias_dropout_add_layer_norm_forward(inp, res, bias, mask, s, gamma, beta, eps)
    _close(out["z"], tz.numpy(), what="fused forward z vs torch")
    _close(out["y"], ty.numpy(), what="fused forward y vs torch")
    _close(out["mean"], tmu.numpy().reshape(-1), what="forward mean vs torch")
    _close(out["rstd"], trstd.numpy().reshape(-1), what="forward rstd vs torch")
    p = ln.layer_norm_forward(res, None, None, eps)
    var = res.var(axis=1)
    _close(p["y"].mean(axis=1), np.zeros(res.shape[0]), atol=1e-12, what="row mean of y")
    _close((p["y"] ** 2).mean(axis=1), var / (var + eps), what="mean y^2")


def pin_ln_saved_z_vs_torch(ln):
    """The saved-z backward against torch float64 autograd of
    LayerNorm(residual + mask * s * (inp + bias)): the gradients of inp,
    residual and bias, with z given as the value torch computed."""
    inp, res, bias, mask, gamma, beta, dy, dzx = _ln_data(26)
    eps, s = 1e-5, 1.0 / 0.8
    H = inp.shape[1]
    ti = torch.tensor(inp, requires_grad=True)
    tr = torch.tensor(res, requires_grad=True)
    tbias = torch.tensor(bias, requires_grad=True)
    tg = torch.tensor(gamma, requires_grad=True)
    z = tr + torch.tensor(mask) * s * (ti + tbias)
    y, mu, rstd = torch.native_layer_norm(z, (H,), tg, torch.tensor(beta), eps)
    loss = (y * torch.tensor(dy)).sum() + (z * torch.tensor(dzx)).sum()
    loss.backward()
    out = ln.layer_norm_backward_saved_z(dy, z.detach().numpy(), mask, s,
                                         mu.detach().numpy().reshape(-1),
                                         rstd.detach().numpy().reshape(-1), gamma, dz_extra=dzx)
    _close(out["dx"], ti.grad.numpy(), what="saved-z dx")
    _close(out["dresidual"], tr.grad.numpy(), what="saved-z dresidual")
    _close(out["dbias"], tbias.grad.numpy(), what="saved-z dbias")
    _close(out["dgamma"], tg.grad.numpy(), what="saved-z dgamma")


LN_PINS = [pin_ln_plain_vs_torch, pin_ln_fused_vs_torch,
           pin_ln_finite_differences, pin_ln_invariants, pin_ln_forward,
           pin_ln_saved_z_vs_torch]
