"""ctypes binding of libgbnorm.so (see include/gbnorm.h for the C ABI).

Argument marshalling only: every step of every call runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors; this module checks their
device, dtype and contiguity, allocates missing outputs / workspaces with
torch, and passes ``data_ptr()`` plus the current CUDA stream to the C
function.  There is no CPU fallback: if the shared library is missing or a
call fails, an exception is raised.
"""

import ctypes
import math
import os

import torch

from . import build as _build

GBN_OK = 0
GBN_F32 = 0
GBN_BF16 = 1
GBN_ROW_RMS = 0
GBN_ROW_LN = 1
GBN_ROW_LN_FUSED = 2
GBN_DEV_WAIT_TIMEOUT = 1
GBN_ACT_NONE = 0
GBN_ACT_RELU = 1
GBN_ACT_LEAKY_RELU = 2
_ACTS = {None: GBN_ACT_NONE, "none": GBN_ACT_NONE, "relu": GBN_ACT_RELU,
         "leaky_relu": GBN_ACT_LEAKY_RELU}

_DTYPE_CODE = {torch.float32: GBN_F32, torch.bfloat16: GBN_BF16}

_lib = None


class GbnError(RuntimeError):
    """A nonzero status returned by the C library."""

    def __init__(self, fn, status):
        text = _lib.gbn_status_string(status).decode() if _lib else "?"
        super().__init__(f"{fn} failed with status {status}: {text}")
        self.status = status


def library_path():
    return _build.library_path()


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "gbn_abi_version": (_INT, []),
    "gbn_status_string": (ctypes.c_char_p, [_INT]),
    "gbn_init": (_INT, [_INT]),
    "gbn_get_device_status": (_INT, [_INT, ctypes.POINTER(_INT), _INT]),
    "gbn_selftest_bounded_wait": (_INT, [_I64, _P]),
    "gbn_bn_workspace_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "gbn_bn_set_persistent_min_bytes": (_I64, [_I64]),
    "gbn_bn_set_small_max_elems": (_I64, [_I64]),
    "gbn_bn_small_max_elems": (_I64, []),
    "gbn_bn_small_blocks_per_channel": (_INT, [_I64, _I64, _I64]),
    "gbn_bn_persistent_min_bytes": (_I64, []),
    "gbn_bn_set_wide_offsets": (_INT, [_INT]),
    "gbn_bn_set_persistent_tmem": (_INT, [_INT]),
    "gbn_bn_set_persistent_steal": (_INT, [_INT]),
    "gbn_bn_forward_train": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _F, _F,
                                    _P, _P, _P, _SZ, _P]),
    "gbn_bn_forward_train_noalloc": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _F,
                                            _F, _P, _P, _P]),
    "gbn_bn_forward_train_act": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _F, _F,
                                        _INT, _F, _P, _P, _P, _SZ, _P]),
    "gbn_bn_stats": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _SZ, _P]),
    "gbn_bn_finalize_apply": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _F, _F,
                                     _P, _P, _P, _SZ, _P]),
    "gbn_bn_apply": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P]),
    "gbn_bn_apply_act": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _INT, _F, _P, _P]),
    "gbn_bn_backward": (_INT, [_P, _P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "gbn_bn_backward_act": (_INT, [_P, _P, _INT, _I64, _I64, _I64, _P, _P, _INT, _F, _P, _P,
                                   _P, _SZ, _P]),
    "gbn_bn_grad_sums": (_INT, [_P, _P, _INT, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "gbn_bn_finalize_dx": (_INT, [_P, _P, _INT, _I64, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "gbn_bn_nhwc_workspace_bytes": (_SZ, [_I64, _I64, _INT]),
    "gbn_bn_nhwc_forward_train": (_INT, [_P, _INT, _I64, _I64, _P, _P, _P, _P, _F, _F, _INT, _F,
                                         _P, _P, _P, _SZ, _P]),
    "gbn_bn_nhwc_apply": (_INT, [_P, _INT, _I64, _I64, _P, _P, _P, _P, _INT, _F, _P, _P]),
    "gbn_bn_nhwc_backward": (_INT, [_P, _P, _INT, _I64, _I64, _P, _P, _INT, _F, _P, _P, _P, _SZ,
                                    _P]),
    "gbn_rowwise_workspace_bytes": (_SZ, [_I64, _I64, _INT, _INT, _INT]),
    "gbn_rmsnorm_backward": (_INT, [_P, _P, _P, _INT, _P, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "gbn_layernorm_backward": (_INT, [_P, _P, _INT, _P, _P, _P, _I64, _I64, _P, _P, _P, _F,
                                      _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "gbn_layernorm_backward_ex": (_INT, [_P, _P, _INT, _P, _P, _P, _I64, _I64, _P, _P, _P, _F,
                                         _P, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "gbn_rmsnorm_forward": (_INT, [_P, _P, _INT, _I64, _I64, _F, _P, _P, _P]),
    "gbn_layernorm_forward": (_INT, [_P, _INT, _I64, _I64, _P, _P, _P, _F, _P, _P, _F, _P, _P,
                                     _P, _P, _P]),
}


def lib():
    """Load the shared library (once).  Raises ImportError if it is not built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGNATURES)


# ------------------------------------------------------------- helpers --

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(fn, status):
    if status != GBN_OK:
        raise GbnError(fn, status)


def _cuda(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _same_device(ref, *named):
    for name, t in named:
        if t is not None and t.device != ref.device:
            raise ValueError(f"{name} is on {t.device}, expected {ref.device}")


def _fp32_vec(t, name, C):
    if t is None:
        return None
    _cuda(t, name)
    if t.dtype != torch.float32:
        # An fp64 (or any non-fp32) statistics tensor is rejected, never
        # reinterpreted: an in-place fp32 update would misread its bytes.
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.numel() != C:
        raise ValueError(f"{name} must have {C} elements")
    return t


def _code(dtype):
    if dtype not in _DTYPE_CODE:
        raise TypeError(f"unsupported dtype {dtype}; use float32 or bfloat16")
    return _DTYPE_CODE[dtype]


def _bn_dims(x):
    if x.dim() < 2:
        raise ValueError("batch norm input must be (N, C, ...)")
    B, C = x.shape[0], x.shape[1]
    HW = math.prod(x.shape[2:]) if x.dim() > 2 else 1
    return B, C, HW


def init(device=None):
    dev = torch.cuda.current_device() if device is None else int(device)
    _check("gbn_init", lib().gbn_init(dev))


def abi_version():
    return lib().gbn_abi_version()


def get_device_status(device=None, clear=False):
    dev = -1 if device is None else int(device)
    v = ctypes.c_int(0)
    _check("gbn_get_device_status", lib().gbn_get_device_status(dev, ctypes.byref(v), int(clear)))
    return v.value


def selftest_bounded_wait(limit_ns=50_000_000, device=None):
    """Launch the bounded-wait self-test (a wait nothing satisfies, given up
    after `limit_ns`) on the current stream of `device`."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    with torch.cuda.device(dev):
        _check("gbn_selftest_bounded_wait",
               lib().gbn_selftest_bounded_wait(int(limit_ns), _stream(dev)))


# ----------------------------------------------------------- BatchNorm --

def bn_set_persistent_min_bytes(nbytes):
    """Input bytes from which the composite BatchNorm calls take the
    single-launch persistent kernel (process-wide); returns the previous
    value."""
    return lib().gbn_bn_set_persistent_min_bytes(int(nbytes))


def bn_set_small_max_elems(m):
    """Per-block element limit of the composite BatchNorm calls'
    single-launch small-channel kernels (default and maximum 2048; 0
    disables them): a channel of at most m elements takes one block, one of
    at most 8*m a thread-block cluster of 2, 4 or 8 blocks.  Returns the
    previous value."""
    return lib().gbn_bn_set_small_max_elems(int(m))


def bn_persistent_min_bytes():
    return lib().gbn_bn_persistent_min_bytes()


def bn_small_max_elems():
    return lib().gbn_bn_small_max_elems()


def bn_small_blocks_per_channel(shape):
    """Blocks per channel (1, 2, 4 or 8) with which the composite BatchNorm
    calls run an NCHW shape in the single-launch small-channel kernels on
    the current device (below the persistent kernel's threshold), or 0 for
    the two-launch kernels."""
    B, C = shape[0], shape[1]
    HW = 1
    for d in shape[2:]:
        HW *= d
    return lib().gbn_bn_small_blocks_per_channel(int(B), int(C), int(HW))


def bn_set_persistent_tmem(enable):
    """Whether the persistent BatchNorm kernel keeps stages in tensor memory
    between its passes (default on; results are bit-identical either way).
    Returns the previous setting."""
    return lib().gbn_bn_set_persistent_tmem(1 if enable else 0)


def bn_set_persistent_steal(enable):
    """Whether CTAs of the persistent BatchNorm kernel take other CTAs' last
    stages at the end of its output pass (default on; results are
    bit-identical either way).  Returns the previous setting."""
    return lib().gbn_bn_set_persistent_steal(1 if enable else 0)


def bn_set_wide_offsets(force):
    """Make the two-launch BatchNorm kernels use 64-bit vector offsets even
    for tensors that do not need them (a test hook; results are identical).
    Process-wide; returns the previous setting."""
    return bool(lib().gbn_bn_set_wide_offsets(1 if force else 0))


def bn_workspace_bytes(B, C, HW, device=None):
    dev = -1 if device is None else int(device)
    return int(lib().gbn_bn_workspace_bytes(B, C, HW, dev))


def bn_stats_tensor(C, device):
    """Empty stats buffer (8*C fp32: rows 0..3 public, 4..7 private)."""
    return torch.empty(8 * C, dtype=torch.float32, device=device)


def bn_workspace(x):
    B, C, HW = _bn_dims(x)
    with torch.cuda.device(x.device):
        n = bn_workspace_bytes(B, C, HW)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=x.device)


def _act_code(act):
    if act not in _ACTS:
        raise ValueError(f"act must be one of {sorted(k for k in _ACTS if k)} or None")
    return _ACTS[act]


def bn_forward_train(x, gamma=None, beta=None, running_mean=None, running_var=None,
                     momentum=0.1, eps=1e-5, *, y=None, stats=None, ws=None, act=None,
                     slope=0.01):
    """Training forward.  Returns (y, stats); running stats updated in place.

    ``stats[:4*C].view(4, C)`` = (mean, var, inv_std, gamma*inv_std).  With
    ``act`` ("relu" / "leaky_relu", negative slope ``slope``) y is the
    activation of the BatchNorm output (gbn_bn_forward_train_act)."""
    code = _act_code(act)
    _cuda(x, "x")
    B, C, HW = _bn_dims(x)
    for name, t in (("gamma", gamma), ("beta", beta), ("running_mean", running_mean),
                    ("running_var", running_var)):
        _fp32_vec(t, name, C)
    y = torch.empty_like(x) if y is None else _cuda(y, "y")
    stats = bn_stats_tensor(C, x.device) if stats is None else _cuda(stats, "stats")
    ws = bn_workspace(x) if ws is None else _cuda(ws, "ws")
    _same_device(x, ("y", y), ("stats", stats), ("ws", ws), ("gamma", gamma), ("beta", beta),
                 ("running_mean", running_mean), ("running_var", running_var))
    args = (_ptr(x), _code(x.dtype), B, C, HW, _ptr(gamma), _ptr(beta), _ptr(running_mean),
            _ptr(running_var), float(momentum), float(eps))
    tail = (_ptr(y), _ptr(stats), _ptr(ws), ws.numel() * ws.element_size(), _stream(x.device))
    with torch.cuda.device(x.device):
        if code == GBN_ACT_NONE:
            name, st = "gbn_bn_forward_train", lib().gbn_bn_forward_train(*args, *tail)
        else:
            name = "gbn_bn_forward_train_act"
            st = lib().gbn_bn_forward_train_act(*args, code, float(slope), *tail)
    _check(name, st)
    return y, stats


def bn_forward_train_noalloc(x, gamma=None, beta=None, running_mean=None, running_var=None,
                             momentum=0.1, eps=1e-5, *, y=None, stats=None):
    """Training forward whose scratch is the library's fixed device array
    (for callers that cannot allocate); see gbn_bn_forward_train_noalloc."""
    _cuda(x, "x")
    B, C, HW = _bn_dims(x)
    for name, t in (("gamma", gamma), ("beta", beta), ("running_mean", running_mean),
                    ("running_var", running_var)):
        _fp32_vec(t, name, C)
    y = torch.empty_like(x) if y is None else _cuda(y, "y")
    stats = bn_stats_tensor(C, x.device) if stats is None else _cuda(stats, "stats")
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_forward_train_noalloc(
            _ptr(x), _code(x.dtype), B, C, HW, _ptr(gamma), _ptr(beta), _ptr(running_mean),
            _ptr(running_var), float(momentum), float(eps), _ptr(y), _ptr(stats),
            _stream(x.device))
    _check("gbn_bn_forward_train_noalloc", st)
    return y, stats


def bn_stats(x, ws):
    _cuda(x, "x")
    B, C, HW = _bn_dims(x)
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_stats(_ptr(x), _code(x.dtype), B, C, HW, _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(x.device))
    _check("gbn_bn_stats", st)


def bn_finalize_apply(x, gamma, beta, running_mean, running_var, momentum, eps, y, stats, ws):
    _cuda(x, "x")
    B, C, HW = _bn_dims(x)
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_finalize_apply(
            _ptr(x), _code(x.dtype), B, C, HW, _ptr(gamma), _ptr(beta), _ptr(running_mean),
            _ptr(running_var), float(momentum), float(eps), _ptr(y), _ptr(stats), _ptr(ws),
            ws.numel() * ws.element_size(), _stream(x.device))
    _check("gbn_bn_finalize_apply", st)


def bn_apply(x, beta=None, *, stats=None, mean=None, scale=None, y=None, act=None,
             slope=0.01):
    """Centred apply (x - mean)*scale + beta from a training stats buffer or
    from per-channel mean/scale (inference), optionally through ``act``."""
    code = _act_code(act)
    _cuda(x, "x")
    B, C, HW = _bn_dims(x)
    for name, t in (("beta", beta), ("mean", mean), ("scale", scale)):
        _fp32_vec(t, name, C)
    y = torch.empty_like(x) if y is None else _cuda(y, "y")
    args = (_ptr(x), _code(x.dtype), B, C, HW, _ptr(stats), _ptr(mean), _ptr(scale), _ptr(beta))
    with torch.cuda.device(x.device):
        if code == GBN_ACT_NONE:
            name, st = "gbn_bn_apply", lib().gbn_bn_apply(*args, _ptr(y), _stream(x.device))
        else:
            name = "gbn_bn_apply_act"
            st = lib().gbn_bn_apply_act(*args, code, float(slope), _ptr(y), _stream(x.device))
    _check(name, st)
    return y


def bn_backward(x, dy, stats, *, dx=None, grads=None, ws=None, beta=None, act=None,
                slope=0.01):
    """Training backward.  Returns (dx, grads) with grads.view(4, C) =
    (dgamma, dbeta, k1, k2).  With ``act`` it is the backward of
    ``bn_forward_train(..., act=act, slope=slope)`` given that forward's
    ``beta`` (gbn_bn_backward_act)."""
    code = _act_code(act)
    _cuda(x, "x")
    _cuda(dy, "dy")
    if dy.shape != x.shape or dy.dtype != x.dtype:
        raise ValueError("dy must match x in shape and dtype")
    B, C, HW = _bn_dims(x)
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx")
    grads = (torch.empty(4 * C, dtype=torch.float32, device=x.device) if grads is None
             else _cuda(grads, "grads"))
    ws = bn_workspace(x) if ws is None else _cuda(ws, "ws")
    _fp32_vec(beta, "beta", C)
    _same_device(x, ("dy", dy), ("stats", stats), ("dx", dx), ("grads", grads), ("ws", ws),
                 ("beta", beta))
    tail = (_ptr(dx), _ptr(grads), _ptr(ws), ws.numel() * ws.element_size(), _stream(x.device))
    with torch.cuda.device(x.device):
        if code == GBN_ACT_NONE:
            name = "gbn_bn_backward"
            st = lib().gbn_bn_backward(_ptr(x), _ptr(dy), _code(x.dtype), B, C, HW,
                                       _ptr(stats), *tail)
        else:
            name = "gbn_bn_backward_act"
            st = lib().gbn_bn_backward_act(_ptr(x), _ptr(dy), _code(x.dtype), B, C, HW,
                                           _ptr(stats), _ptr(beta), code, float(slope), *tail)
    _check(name, st)
    return dx, grads


def bn_grad_sums(x, dy, stats, ws):
    B, C, HW = _bn_dims(x)
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_grad_sums(_ptr(x), _ptr(dy), _code(x.dtype), B, C, HW, _ptr(stats),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(x.device))
    _check("gbn_bn_grad_sums", st)


def bn_finalize_dx(x, dy, stats, dx, grads, ws):
    B, C, HW = _bn_dims(x)
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_finalize_dx(_ptr(x), _ptr(dy), _code(x.dtype), B, C, HW, _ptr(stats),
                                      _ptr(dx), _ptr(grads), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(x.device))
    _check("gbn_bn_finalize_dx", st)


# ------------------------------------------------------------ row-wise --

def _nhwc_dims(x):
    if x.dim() < 2 or not x.is_contiguous():
        raise ValueError("channels-last BatchNorm wants a contiguous [..., C] tensor")
    C = x.shape[-1]
    return x.numel() // C if C else 0, C


def bn_nhwc_workspace(x):
    M, C = _nhwc_dims(x)
    with torch.cuda.device(x.device):
        n = lib().gbn_bn_nhwc_workspace_bytes(M, C, -1)
    if n == 0:
        raise ValueError(f"bad channels-last BatchNorm shape {tuple(x.shape)}")
    return torch.empty(n, dtype=torch.uint8, device=x.device)


def bn_nhwc_forward_train(x, gamma=None, beta=None, running_mean=None, running_var=None,
                          momentum=0.1, eps=1e-5, *, y=None, stats=None, ws=None, act=None,
                          slope=0.01):
    """Channels-last training forward: x is a contiguous [..., C] tensor (e.g.
    [N, H, W, C]); the channel is the last dimension.  Returns (y, stats)."""
    code = _act_code(act)
    _cuda(x, "x")
    M, C = _nhwc_dims(x)
    for name, t in (("gamma", gamma), ("beta", beta), ("running_mean", running_mean),
                    ("running_var", running_var)):
        _fp32_vec(t, name, C)
    y = torch.empty_like(x) if y is None else _cuda(y, "y")
    stats = bn_stats_tensor(C, x.device) if stats is None else _cuda(stats, "stats")
    ws = bn_nhwc_workspace(x) if ws is None else _cuda(ws, "ws")
    _same_device(x, ("y", y), ("stats", stats), ("ws", ws), ("gamma", gamma), ("beta", beta),
                 ("running_mean", running_mean), ("running_var", running_var))
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_nhwc_forward_train(
            _ptr(x), _code(x.dtype), M, C, _ptr(gamma), _ptr(beta), _ptr(running_mean),
            _ptr(running_var), float(momentum), float(eps), code, float(slope), _ptr(y),
            _ptr(stats), _ptr(ws), ws.numel() * ws.element_size(), _stream(x.device))
    _check("gbn_bn_nhwc_forward_train", st)
    return y, stats


def bn_nhwc_apply(x, beta=None, *, stats=None, mean=None, scale=None, y=None, act=None,
                  slope=0.01):
    """Channels-last centred apply from a training stats buffer or from
    per-channel mean / scale (inference), optionally through ``act``."""
    code = _act_code(act)
    _cuda(x, "x")
    M, C = _nhwc_dims(x)
    for name, t in (("beta", beta), ("mean", mean), ("scale", scale)):
        _fp32_vec(t, name, C)
    y = torch.empty_like(x) if y is None else _cuda(y, "y")
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_nhwc_apply(_ptr(x), _code(x.dtype), M, C, _ptr(stats), _ptr(mean),
                                     _ptr(scale), _ptr(beta), code, float(slope), _ptr(y),
                                     _stream(x.device))
    _check("gbn_bn_nhwc_apply", st)
    return y


def bn_nhwc_backward(x, dy, stats, *, dx=None, grads=None, ws=None, beta=None, act=None,
                     slope=0.01):
    """Channels-last training backward.  Returns (dx, grads) with
    grads.view(4, C) = (dgamma, dbeta, k1, k2)."""
    code = _act_code(act)
    _cuda(x, "x")
    _cuda(dy, "dy")
    if dy.shape != x.shape or dy.dtype != x.dtype:
        raise ValueError("dy must match x in shape and dtype")
    M, C = _nhwc_dims(x)
    _fp32_vec(beta, "beta", C)
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx")
    grads = (torch.empty(4 * C, dtype=torch.float32, device=x.device) if grads is None
             else _cuda(grads, "grads"))
    ws = bn_nhwc_workspace(x) if ws is None else _cuda(ws, "ws")
    _same_device(x, ("dy", dy), ("stats", stats), ("dx", dx), ("grads", grads), ("ws", ws),
                 ("beta", beta))
    with torch.cuda.device(x.device):
        st = lib().gbn_bn_nhwc_backward(
            _ptr(x), _ptr(dy), _code(x.dtype), M, C, _ptr(stats), _ptr(beta), code,
            float(slope), _ptr(dx), _ptr(grads), _ptr(ws), ws.numel() * ws.element_size(),
            _stream(x.device))
    _check("gbn_bn_nhwc_backward", st)
    return dx, grads


def rowwise_workspace_bytes(R, H, kind, dtype, device=None):
    dev = -1 if device is None else int(device)
    return int(lib().gbn_rowwise_workspace_bytes(R, H, kind, _code(dtype), dev))


def rowwise_workspace(R, H, kind, dtype, device):
    with torch.cuda.device(device):
        n = rowwise_workspace_bytes(R, H, kind, dtype)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def _rows(t, name):
    _cuda(t, name)
    if t.dim() < 1:
        raise ValueError(f"{name} must have a last (normalised) dimension")
    H = t.shape[-1]
    return (t.numel() // H if H else 0), H


def rmsnorm_backward(dy, x, w, rstd, *, dx=None, dw=None, ws=None):
    """RMSNorm backward from the saved rstd (fp32, one per row).
    Returns (dx, dweight)."""
    R, H = _rows(x, "x")
    _cuda(dy, "dy")
    _cuda(w, "w")
    _cuda(rstd, "rstd")
    if dy.shape != x.shape or dy.dtype != x.dtype or w.dtype != x.dtype or w.numel() != H:
        raise ValueError("dy/x/w shapes or dtypes disagree")
    if rstd.dtype != torch.float32 or rstd.numel() != R:
        raise TypeError("rstd must be float32 with one value per row")
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx")
    dw = torch.empty_like(w) if dw is None else _cuda(dw, "dw")
    ws = rowwise_workspace(R, H, GBN_ROW_RMS, x.dtype, x.device) if ws is None else ws
    _same_device(x, ("dy", dy), ("w", w), ("rstd", rstd), ("dx", dx), ("dw", dw), ("ws", ws))
    with torch.cuda.device(x.device):
        st = lib().gbn_rmsnorm_backward(_ptr(dy), _ptr(x), _ptr(w), _code(x.dtype), _ptr(rstd),
                                        R, H, _ptr(dx), _ptr(dw), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(x.device))
    _check("gbn_rmsnorm_backward", st)
    return dx, dw


GBN_LN_SAVED_Z = 1
GBN_LN_DRES_F32 = 2


def layernorm_backward(dy, x, mean, rstd, gamma, *, residual=None, bias=None, mask=None,
                       dropout_scale=1.0, dz_extra=None, dx=None, dresidual=None, dgamma=None,
                       dbeta=None, dbias=None, ws=None, want_dresidual=True, want_dbias=True,
                       saved_z=False, dres_f32=False):
    """LayerNorm backward; fused with bias+dropout+add when ``residual`` is
    given (then ``x`` is the dropout input), or from the saved LayerNorm
    input when ``saved_z`` (then ``x`` is z, there is no residual or bias, and
    the mask / dropout_scale still give dx, dresidual and dbias).
    ``dres_f32`` writes dresidual in fp32.  Returns a dict with dx,
    dresidual, dgamma, dbeta, dbias (None where not computed)."""
    R, H = _rows(x, "x")
    fused = residual is not None or saved_z
    for name, t in (("dy", dy), ("mean", mean), ("rstd", rstd), ("gamma", gamma)):
        _cuda(t, name)
    if dy.shape != x.shape or dy.dtype != x.dtype or gamma.dtype != x.dtype:
        raise ValueError("dy/x/gamma dtypes or shapes disagree")
    if mean.dtype != torch.float32 or rstd.dtype != torch.float32:
        raise TypeError("mean and rstd must be float32")
    if mask is not None:
        _cuda(mask, "mask")
        if mask.dtype == torch.bool:
            mask = mask.view(torch.uint8)
        if mask.dtype != torch.uint8:
            raise TypeError("mask must be bool or uint8")
    if dz_extra is not None and (_cuda(dz_extra, "dz_extra").dtype != torch.float32):
        raise TypeError("dz_extra must be float32")
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx")
    if fused:
        if residual is not None:
            _cuda(residual, "residual")
        if dresidual is None and want_dresidual:
            dresidual = torch.empty_like(x, dtype=torch.float32 if dres_f32 else x.dtype)
        if dbias is None and want_dbias and (bias is not None or saved_z):
            dbias = torch.empty_like(gamma)
    dgamma = torch.empty_like(gamma) if dgamma is None else dgamma
    dbeta = torch.empty_like(gamma) if dbeta is None else dbeta
    kind = GBN_ROW_LN_FUSED if fused else GBN_ROW_LN
    ws = rowwise_workspace(R, H, kind, x.dtype, x.device) if ws is None else ws
    _same_device(x, ("dy", dy), ("mean", mean), ("rstd", rstd), ("gamma", gamma),
                 ("residual", residual), ("bias", bias), ("mask", mask), ("dz_extra", dz_extra),
                 ("dx", dx), ("dresidual", dresidual), ("dgamma", dgamma), ("dbeta", dbeta),
                 ("dbias", dbias), ("ws", ws))
    with torch.cuda.device(x.device):
        flags = (GBN_LN_SAVED_Z if saved_z else 0) | (GBN_LN_DRES_F32 if dres_f32 else 0)
        st = lib().gbn_layernorm_backward_ex(
            _ptr(dy), _ptr(x), _code(x.dtype), _ptr(mean), _ptr(rstd), _ptr(gamma), R, H,
            _ptr(residual), _ptr(bias), _ptr(mask), float(dropout_scale), _ptr(dz_extra),
            _ptr(dx), _ptr(dresidual), _ptr(dgamma), _ptr(dbeta), _ptr(dbias), _ptr(ws),
            ws.numel() * ws.element_size(), flags, _stream(x.device))
    _check("gbn_layernorm_backward_ex", st)
    return {"dx": dx, "dresidual": dresidual, "dgamma": dgamma, "dbeta": dbeta,
            "dbias": dbias}


def rmsnorm_forward(x, w=None, eps=1e-5, *, y=None, rstd=None):
    """RMSNorm training forward.  Returns (y, rstd) with rstd fp32 [rows]."""
    R, H = _rows(x, "x")
    if w is not None and (_cuda(w, "w").dtype != x.dtype or w.numel() != H):
        raise ValueError("w must match x's dtype and last dimension")
    y = torch.empty_like(x) if y is None else _cuda(y, "y")
    rstd = torch.empty(R, dtype=torch.float32, device=x.device) if rstd is None else rstd
    if _cuda(rstd, "rstd").dtype != torch.float32 or rstd.numel() != R:
        raise TypeError("rstd must be float32 with one value per row")
    _same_device(x, ("w", w), ("y", y), ("rstd", rstd))
    with torch.cuda.device(x.device):
        st = lib().gbn_rmsnorm_forward(_ptr(x), _ptr(w), _code(x.dtype), R, H, float(eps),
                                       _ptr(y), _ptr(rstd), _stream(x.device))
    _check("gbn_rmsnorm_forward", st)
    return y, rstd


def layernorm_forward(x, gamma=None, beta=None, eps=1e-5, *, residual=None, bias=None,
                      mask=None, dropout_scale=1.0, y=None, z=None, mean=None, rstd=None,
                      want_z=True):
    """LayerNorm training forward; fused with bias+dropout+add when
    ``residual`` is given (then ``x`` is the dropout input and z = residual +
    mask*dropout_scale*(x + bias) is returned as the residual-stream output).
    Returns a dict with y, z (None when not fused or not wanted), mean, rstd."""
    R, H = _rows(x, "x")
    fused = residual is not None
    for name, t in (("gamma", gamma), ("beta", beta), ("bias", bias)):
        if t is not None and (_cuda(t, name).dtype != x.dtype or t.numel() != H):
            raise ValueError(f"{name} must match x's dtype and last dimension")
    if fused and (_cuda(residual, "residual").shape != x.shape or residual.dtype != x.dtype):
        raise ValueError("residual must match x")
    if mask is not None:
        _cuda(mask, "mask")
        if mask.dtype == torch.bool:
            mask = mask.view(torch.uint8)
        if mask.dtype != torch.uint8:
            raise TypeError("mask must be bool or uint8")
    y = torch.empty_like(x) if y is None else _cuda(y, "y")
    if fused and z is None and want_z:
        z = torch.empty_like(x)
    mean = torch.empty(R, dtype=torch.float32, device=x.device) if mean is None else mean
    rstd = torch.empty(R, dtype=torch.float32, device=x.device) if rstd is None else rstd
    for name, t in (("mean", mean), ("rstd", rstd)):
        if _cuda(t, name).dtype != torch.float32 or t.numel() != R:
            raise TypeError(f"{name} must be float32 with one value per row")
    _same_device(x, ("gamma", gamma), ("beta", beta), ("residual", residual), ("bias", bias),
                 ("mask", mask), ("y", y), ("z", z), ("mean", mean), ("rstd", rstd))
    with torch.cuda.device(x.device):
        st = lib().gbn_layernorm_forward(
            _ptr(x), _code(x.dtype), R, H, _ptr(residual), _ptr(bias), _ptr(mask),
            float(dropout_scale), _ptr(gamma), _ptr(beta), float(eps), _ptr(y), _ptr(z),
            _ptr(mean), _ptr(rstd), _stream(x.device))
    _check("gbn_layernorm_forward", st)
    return {"y": y, "z": z, "mean": mean, "rstd": rstd}
