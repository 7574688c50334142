"""The C ABI library on the host: it builds, loads, exports every symbol the
header declares, and rejects bad arguments before touching CUDA.  No GPU is
needed: argument validation runs before any CUDA call, and fake (never
dereferenced) device addresses are enough to exercise it."""

import ctypes
import os
import re

import pytest

from bwd_bn_pass_gb300 import gbnorm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, EINVAL, EDTYPE, EALIGN, EWORKSPACE, ECUDA = 0, -1, -2, -3, -4, -5
P = ctypes.c_void_p
A16 = P(0x10000)   # 16-byte aligned fake address
A4 = P(0x10004)    # 4-byte aligned only
NULL = None


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^GBN_API\s+[\w\s\*]+?\b(gbn_\w+)\s*\(", text, re.M)
    return names


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ("gbn_bn_forward_train", "gbn_bn_apply", "gbn_bn_backward",
              "gbn_rmsnorm_backward", "gbn_layernorm_backward"):
        assert n in names


def test_library_exports_every_declared_symbol(gbn):
    L = gbn.lib()
    for name in declared_symbols():
        assert hasattr(L, name), f"{name} not exported"
        assert name in gbn.exported_symbols(), f"{name} missing from the binding"


def test_abi_version_and_status_strings(gbn):
    L = gbn.lib()
    assert L.gbn_abi_version() == 1
    for code in (OK, EINVAL, EDTYPE, EALIGN, EWORKSPACE, ECUDA, -6, 12345):
        assert isinstance(L.gbn_status_string(code), bytes)
    assert L.gbn_status_string(EWORKSPACE) == b"workspace too small"


def _fwd(L, x=A16, dtype=0, B=4, C=3, HW=5, gamma=NULL, beta=NULL, rm=NULL, rv=NULL,
         mom=0.1, eps=1e-5, y=A16, stats=A16, ws=A16, nbytes=1 << 20):
    return L.gbn_bn_forward_train(x, dtype, B, C, HW, gamma, beta, rm, rv, mom, eps, y, stats,
                                  ws, nbytes, NULL)


def test_bn_forward_argument_errors(gbn):
    L = gbn.lib()
    assert _fwd(L, dtype=7) == EDTYPE
    assert _fwd(L, B=-1) == EINVAL
    assert _fwd(L, HW=-3) == EINVAL
    assert _fwd(L, B=1, HW=1) == EINVAL          # M = 1: no unbiased running var
    assert _fwd(L, B=0) == EINVAL                # M = 0 in training
    assert _fwd(L, x=NULL) == EINVAL
    assert _fwd(L, y=NULL) == EINVAL
    assert _fwd(L, stats=NULL) == EINVAL
    assert _fwd(L, ws=NULL) == EINVAL
    assert _fwd(L, stats=A4) == EALIGN
    assert _fwd(L, ws=A4) == EALIGN
    assert _fwd(L, eps=float("nan")) == EINVAL
    assert _fwd(L, eps=-1.0) == EINVAL
    assert _fwd(L, mom=float("nan")) == EINVAL
    assert _fwd(L, B=1 << 40, C=1 << 40) == EINVAL   # element count overflow
    assert _fwd(L, B=1 << 20, HW=1 << 12) == EINVAL  # per-channel count >= 2^31
    assert _fwd(L, C=0) == OK                    # nothing to do, nothing launched


def test_bn_noalloc_argument_errors(gbn):
    """The allocation-free forward rejects bad arguments before any CUDA call
    (it resolves its fixed scratch array only afterwards), with the codes of
    gbn_bn_forward_train."""
    L = gbn.lib()

    def na(x=A16, dtype=0, B=4, C=3, HW=5, y=A16, stats=A16, mom=0.1, eps=1e-5):
        return L.gbn_bn_forward_train_noalloc(x, dtype, B, C, HW, NULL, NULL, NULL, NULL, mom,
                                              eps, y, stats, NULL)

    assert na(dtype=7) == EDTYPE
    assert na(B=-1) == EINVAL
    assert na(B=1, HW=1) == EINVAL
    assert na(x=NULL) == EINVAL
    assert na(y=NULL) == EINVAL
    assert na(stats=NULL) == EINVAL
    assert na(stats=A4) == EALIGN
    assert na(eps=float("nan")) == EINVAL
    assert na(mom=float("nan")) == EINVAL
    assert na(C=0) == OK


def test_bn_other_entry_points_argument_errors(gbn):
    L = gbn.lib()
    assert L.gbn_bn_stats(A16, 3, 2, 2, 2, A16, 4096, NULL) == EDTYPE
    assert L.gbn_bn_stats(NULL, 0, 2, 2, 2, A16, 4096, NULL) == EINVAL
    assert L.gbn_bn_apply(A16, 0, 2, 2, 2, NULL, NULL, NULL, NULL, A16, NULL) == EINVAL
    assert L.gbn_bn_apply(A16, 0, 2, 2, 2, A4, NULL, NULL, NULL, A16, NULL) == EALIGN
    assert L.gbn_bn_apply(A16, 0, 0, 2, 2, NULL, NULL, NULL, NULL, A16, NULL) == OK
    assert L.gbn_bn_backward(A16, NULL, 0, 2, 2, 2, A16, A16, A16, A16, 4096, NULL) == EINVAL
    assert L.gbn_bn_backward(A16, A16, 0, 2, 2, 2, A16, NULL, A16, A16, 4096, NULL) == EINVAL
    assert L.gbn_bn_backward(A16, A16, 0, 2, 2, 2, A4, A16, A16, A16, 4096, NULL) == EALIGN
    assert L.gbn_bn_backward(A16, A16, 1, 1, 2, 1, A16, A16, A16, A16, 4096, NULL) == EINVAL
    assert L.gbn_bn_grad_sums(A16, A16, 0, 2, 2, 2, NULL, A16, 4096, NULL) == EINVAL
    assert L.gbn_bn_finalize_dx(A16, A16, 0, 2, 2, 2, A16, A16, NULL, A16, 4096, NULL) == EINVAL
    assert L.gbn_bn_workspace_bytes(-1, 2, 2, -1) == 0


def test_bn_act_argument_errors(gbn):
    """Unknown activations and non-finite LeakyReLU slopes are rejected
    before anything touches a device."""
    L = gbn.lib()

    def fwd(act, slope, C=3):
        return L.gbn_bn_forward_train_act(A16, 0, 4, C, 5, NULL, NULL, NULL, NULL, 0.1, 1e-5,
                                          act, slope, A16, A16, A16, 1 << 20, NULL)

    def bwd(act, slope, C=3):
        return L.gbn_bn_backward_act(A16, A16, 0, 4, C, 5, A16, NULL, act, slope, A16, A16, A16,
                                     1 << 20, NULL)

    def app(act, slope, C=3):
        return L.gbn_bn_apply_act(A16, 0, 4, C, 5, A16, NULL, NULL, NULL, act, slope, A16, NULL)

    for f in (fwd, bwd, app):
        assert f(3, 0.0) == EINVAL
        assert f(-1, 0.0) == EINVAL
        assert f(2, float("nan")) == EINVAL
        assert f(2, float("inf")) == EINVAL
        assert f(1, float("nan"), C=0) == OK     # ReLU ignores the slope
        assert f(2, -0.5, C=0) == OK             # any finite slope
    assert L.gbn_bn_forward_train_act(A16, 7, 4, 3, 5, NULL, NULL, NULL, NULL, 0.1, 1e-5, 1,
                                      0.0, A16, A16, A16, 1 << 20, NULL) == EDTYPE


def test_bn_nhwc_argument_errors(gbn):
    L = gbn.lib()

    def fwd(x=A16, dtype=0, M=8, C=4, act=0, slope=0.0, y=A16, stats=A16, ws=A16, n=1 << 20,
            eps=1e-5):
        return L.gbn_bn_nhwc_forward_train(x, dtype, M, C, NULL, NULL, NULL, NULL, 0.1, eps, act,
                                           slope, y, stats, ws, n, NULL)

    def bwd(x=A16, dy=A16, dtype=0, M=8, C=4, stats=A16, dx=A16, grads=A16, ws=A16):
        return L.gbn_bn_nhwc_backward(x, dy, dtype, M, C, stats, NULL, 0, 0.0, dx, grads, ws,
                                      1 << 20, NULL)

    assert fwd(dtype=5) == EDTYPE
    assert fwd(M=-1) == EINVAL
    assert fwd(M=1) == EINVAL                      # one row: no unbiased running var
    assert fwd(M=1 << 31) == EINVAL                # per-channel count >= 2^31
    assert fwd(act=9) == EINVAL
    assert fwd(x=NULL) == EINVAL
    assert fwd(stats=NULL) == EINVAL
    assert fwd(ws=A4) == EALIGN
    assert fwd(eps=float("nan")) == EINVAL
    assert fwd(C=0) == OK                          # nothing to do
    assert bwd(dy=NULL) == EINVAL
    assert bwd(grads=NULL) == EINVAL
    assert bwd(dtype=3) == EDTYPE
    assert bwd(C=0) == OK
    assert L.gbn_bn_nhwc_workspace_bytes(-1, 4, -1) == 0
    assert L.gbn_bn_nhwc_apply(A16, 0, 8, 4, NULL, NULL, NULL, NULL, 0, 0.0, A16, NULL) == EINVAL
    assert L.gbn_bn_nhwc_apply(A16, 0, 8, 4, A16, NULL, NULL, NULL, 5, 0.0, A16, NULL) == EINVAL
    assert L.gbn_bn_nhwc_apply(A16, 0, 0, 4, NULL, NULL, NULL, NULL, 0, 0.0, A16, NULL) == OK


def test_bn_small_channel_switch(gbn):
    L = gbn.lib()
    prev = L.gbn_bn_set_small_max_elems(100)
    assert L.gbn_bn_small_max_elems() == 100
    assert L.gbn_bn_set_small_max_elems(-5) == 100
    assert L.gbn_bn_set_small_max_elems(1 << 40) == 0      # negative stored as 0
    assert L.gbn_bn_set_small_max_elems(prev) == 2048      # capped at the kernels' limit


def test_bn_persistent_tmem_switch(gbn):
    L = gbn.lib()
    prev = L.gbn_bn_set_persistent_tmem(0)
    assert prev in (0, 1)
    assert L.gbn_bn_set_persistent_tmem(7) == 0
    assert L.gbn_bn_set_persistent_tmem(prev) == 1          # nonzero stored as 1


def test_bn_persistent_steal_switch(gbn):
    L = gbn.lib()
    prev = L.gbn_bn_set_persistent_steal(0)
    assert prev in (0, 1)
    assert L.gbn_bn_set_persistent_steal(3) == 0
    assert L.gbn_bn_set_persistent_steal(prev) == 1         # nonzero stored as 1


def test_bn_persistent_threshold(gbn):
    L = gbn.lib()
    prev = L.gbn_bn_set_persistent_min_bytes(12345)
    assert prev >= 0
    assert L.gbn_bn_set_persistent_min_bytes(-7) == 12345
    assert L.gbn_bn_set_persistent_min_bytes(prev) == 0     # negative stored as 0


def _rms(L, dtype=1, R=4, H=64, dy=A16, x=A16, w=A16, rstd=A16, dx=A16, dw=A16, ws=A16):
    return L.gbn_rmsnorm_backward(dy, x, w, dtype, rstd, R, H, dx, dw, ws, 1 << 20, NULL)


def test_rmsnorm_argument_errors(gbn):
    L = gbn.lib()
    assert _rms(L, dtype=5) == EDTYPE
    assert _rms(L, R=-1) == EINVAL
    assert _rms(L, w=NULL) == EINVAL
    assert _rms(L, dw=NULL) == EINVAL
    assert _rms(L, rstd=NULL) == EINVAL
    assert _rms(L, ws=A4) == EALIGN
    assert _rms(L, H=0) == OK
    assert L.gbn_rowwise_workspace_bytes(4, 64, 9, 0, -1) == 0


def _ln(L, dtype=1, R=4, H=64, residual=NULL, bias=NULL, mask=NULL, scale=1.0,
        dres=NULL, dbias=NULL, gamma=A16, ws=A16, mean=A16):
    return L.gbn_layernorm_backward(A16, A16, dtype, mean, A16, gamma, R, H, residual, bias,
                                    mask, scale, NULL, A16, dres, A16, A16, dbias, ws, 1 << 20,
                                    NULL)


def test_layernorm_argument_errors(gbn):
    L = gbn.lib()
    assert _ln(L, dtype=2) == EDTYPE
    assert _ln(L, H=-1) == EINVAL
    assert _ln(L, bias=A16) == EINVAL            # bias without residual
    assert _ln(L, mask=A16) == EINVAL            # mask without residual
    assert _ln(L, dres=A16) == EINVAL            # dresidual without residual
    assert _ln(L, dbias=A16) == EINVAL
    assert _ln(L, gamma=NULL) == EINVAL
    assert _ln(L, mean=NULL) == EINVAL
    assert _ln(L, residual=A16, scale=float("nan")) == EINVAL
    assert _ln(L, ws=A4) == EALIGN


def _rmsf(L, dtype=1, R=4, H=64, x=A16, w=A16, eps=1e-5, y=A16, rstd=A16):
    return L.gbn_rmsnorm_forward(x, w, dtype, R, H, eps, y, rstd, NULL)


def _lnf(L, dtype=1, R=4, H=64, x=A16, residual=NULL, bias=NULL, mask=NULL, scale=1.0,
         eps=1e-5, y=A16, z=NULL, mean=A16, rstd=A16):
    return L.gbn_layernorm_forward(x, dtype, R, H, residual, bias, mask, scale, A16, A16, eps,
                                   y, z, mean, rstd, NULL)


def test_layernorm_backward_flag_errors(gbn):
    L = gbn.lib()

    def ex(flags, residual=NULL, bias=NULL):
        return L.gbn_layernorm_backward_ex(A16, A16, 1, A16, A16, A16, 4, 64, residual, bias,
                                           NULL, 1.0, NULL, A16, A16, A16, A16, NULL, A16,
                                           1 << 20, flags, NULL)
    assert ex(4) == EINVAL                      # unknown flag bit
    assert ex(1, residual=A16) == EINVAL        # saved z with a residual
    assert ex(1, bias=A16) == EINVAL            # saved z with a bias
    assert ex(2) == EINVAL                      # fp32 dresidual without a fused form


def test_forward_argument_errors(gbn):
    L = gbn.lib()
    assert _rmsf(L, dtype=3) == EDTYPE
    assert _rmsf(L, R=-1) == EINVAL
    assert _rmsf(L, H=0) == EINVAL               # empty rows have no mean
    assert _rmsf(L, x=NULL) == EINVAL
    assert _rmsf(L, rstd=NULL) == EINVAL
    assert _rmsf(L, eps=-1.0) == EINVAL
    assert _rmsf(L, R=0) == OK                   # nothing to do
    assert _lnf(L, dtype=3) == EDTYPE
    assert _lnf(L, bias=A16) == EINVAL           # bias without residual
    assert _lnf(L, mask=A16) == EINVAL           # mask without residual
    assert _lnf(L, z=A16) == EINVAL              # z output without residual
    assert _lnf(L, mean=NULL) == EINVAL
    assert _lnf(L, y=NULL) == EINVAL
    assert _lnf(L, residual=A16, scale=float("nan")) == EINVAL
    assert _lnf(L, eps=float("nan")) == EINVAL


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host without GPU only")
def test_valid_call_without_gpu_reports_cuda_error(gbn):
    L = gbn.lib()
    assert _fwd(L) == ECUDA
    assert _rms(L) == ECUDA
    assert _rmsf(L) == ECUDA
    assert _lnf(L, residual=A16, bias=A16, mask=A16, z=A16) == ECUDA
    assert L.gbn_init(-1) == ECUDA
