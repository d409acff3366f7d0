"""ctypes binding of libgbnorm.so: the C ABI of include/gbnorm.h, one Python
function per entry point, under the same names.

Argument marshalling only: tensors become device pointers, shapes become
(M, N) with every leading dimension folded into M, dtypes become the
library's codes, and the current torch stream is passed as the CUDA stream.
An input whose rows are not contiguous (a head-major view, a row-strided
slice) is passed in place with a gbn_rows layout when its last stride is 1
and its leading dimensions fold into at most three levels; only other
layouts are copied.  Outputs are always contiguous.
Every step of the computation runs in the CUDA kernels; there is no
fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

GBN_F32, GBN_BF16, GBN_F16 = 0, 1, 2
GBN_OP_DYT, GBN_OP_LAYERNORM, GBN_OP_RMSNORM = 0, 1, 2
GBN_OK = 0
# RMSNorm expressions: Llama (weight after the cast), weight before the cast, Gemma (1 + w)
GBN_RMS_CAST_FIRST, GBN_RMS_WEIGHT_FIRST, GBN_RMS_GEMMA = 0, 1, 2
GBN_ESCRATCH = 6
GBN_STATIC_WS_BYTES = 8 << 20  # size of the library's static scratch array
SIZE_MAX = ctypes.c_size_t(-1).value

_DTYPES = {torch.float32: GBN_F32, torch.bfloat16: GBN_BF16, torch.float16: GBN_F16}

# The entry points the header declares, with their ctypes signatures.
_P, _I64, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class gbn_rows(ctypes.Structure):
    """Row r of an input starts at element (r % n1)*s1 + ((r / n1) % n2)*s2
    + (r / (n1*n2))*s3 of it."""
    _fields_ = [("n1", ctypes.c_int64), ("s1", ctypes.c_int64), ("n2", ctypes.c_int64),
                ("s2", ctypes.c_int64), ("s3", ctypes.c_int64)]


_R = ctypes.POINTER(gbn_rows)
SIGNATURES = {
    "gbn_status_string": ([_I], ctypes.c_char_p),
    "gbn_bwd_workspace_bytes": ([_I, _I64, _I64, _I, _I, _I], _SZ),
    "gbn_read_faults": ([ctypes.POINTER(ctypes.c_uint), _I], _I),
    "gbn_selftest_wait_timeout": ([ctypes.c_longlong, _P, _P], _I),
    "dyt_fwd": ([_P, _P, _P, _P, _P, _I64, _I64, _I, _I, _P], _I),
    "dyt_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _I, _P, _SZ, _P], _I),
    "layernorm_fwd": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P], _I),
    "layernorm_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _I, _P, _SZ, _P], _I),
    "rmsnorm_fwd": ([_P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P], _I),
    "rmsnorm_bwd": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P, _SZ, _P], _I),
    "rmsnorm_fwd_ex": ([_P, _P, _P, _P, _I64, _I64, _F, _I, _I, _I, _P], _I),
    "rmsnorm_bwd_ex": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _I, _P, _SZ, _P], _I),
    "rmsnorm_bwd_static_ws": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P], _I),
    "dyt_fwd_rows": ([_P, _R, _P, _P, _P, _P, _I64, _I64, _I, _I, _P], _I),
    "dyt_bwd_rows": ([_P, _R, _P, _R, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _I, _P, _SZ, _P],
                     _I),
    "layernorm_fwd_rows": ([_P, _R, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P], _I),
    "layernorm_bwd_rows": ([_P, _R, _P, _R, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _I, _P, _SZ,
                            _P], _I),
    "rmsnorm_fwd_rows": ([_P, _R, _P, _P, _P, _I64, _I64, _F, _I, _I, _I, _P], _I),
    "rmsnorm_bwd_rows": ([_P, _R, _P, _R, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _I, _P, _SZ,
                          _P], _I),
}

_lock = threading.Lock()
_handle = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libgbnorm.so (built in-tree by normalization_layers_fwd_gb300.build)."""
    global _handle
    with _lock:
        if _handle is not None and path is None:
            return _handle
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with `python -m normalization_layers_fwd_gb300.build`"
                " (nvcc, sm_103a); there is no fallback implementation")
        lib = ctypes.CDLL(p)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        if path is None:
            _handle = lib
        return lib


class GbnError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().gbn_status_string(status).decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


def _check(status: int, where: str):
    if status != GBN_OK:
        raise GbnError(status, where)


# -------------------------------------------------------------- marshalling

def _code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16") from None


def _rows(x: torch.Tensor):
    """(contiguous x, M, N): leading dimensions fold into rows."""
    if not x.is_cuda:
        raise ValueError("activations must be CUDA tensors")
    if x.dim() < 1:
        raise ValueError("activations need at least one dimension")
    x = x.contiguous()
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    return x, M, N


def row_layout(x: torch.Tensor):
    """(x or a contiguous copy, gbn_rows or None): None when x's rows are
    contiguous; a layout when its last stride is 1 and its leading dimensions
    (size-1 ones dropped, adjacent ones merged where they nest) fold into at
    most three levels; otherwise a contiguous copy and None."""
    if not x.is_cuda:
        raise ValueError("activations must be CUDA tensors")
    if x.dim() < 1:
        raise ValueError("activations need at least one dimension")
    if x.is_contiguous() or x.numel() == 0:
        return x.contiguous(), None
    lay = fold_rows(tuple(x.shape), tuple(x.stride()))
    return (x, lay) if lay is not None else (x.contiguous(), None)


def fold_rows(shape, strides):
    """The gbn_rows of a non-empty tensor of this shape and these element
    strides, or None when it has none (last stride not 1, or more than three
    leading levels after dropping size-1 dimensions and merging nested ones)."""
    if shape[-1] > 1 and strides[-1] != 1:
        return None
    levels = []  # (size, stride), innermost first
    for n, st in zip(reversed(shape[:-1]), reversed(strides[:-1])):
        if n == 1:
            continue
        if levels and st == levels[-1][0] * levels[-1][1]:
            levels[-1] = (levels[-1][0] * n, levels[-1][1])
        else:
            levels.append((n, st))
    if len(levels) > 3:
        return None
    levels += [(1, 0)] * (3 - len(levels))
    (n1, s1), (n2, s2), (_, s3) = levels
    return gbn_rows(n1, s1, n2, s2, s3)


def _lay(layout):
    return None if layout is None else ctypes.byref(layout)


def _out(x):
    """A contiguous output of x's shape and dtype."""
    return torch.empty(x.shape, dtype=x.dtype, device=x.device)


def _input_rows(x, dy=None):
    """(x, x layout, dy, dy layout, M, N) for the *_rows entry points."""
    x, xl = row_layout(x)
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    dyl = None
    if dy is not None:
        if dy.shape != x.shape or dy.dtype != x.dtype:
            raise ValueError("dy must match x in shape and dtype")
        dy, dyl = row_layout(dy)
    return x, xl, dy, dyl, M, N


def _param(p, like: torch.Tensor, n: int, name: str, required: bool = True):
    if p is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if not p.is_cuda or p.device != like.device:
        raise ValueError(f"{name} must be on {like.device}")
    if p.numel() != n:
        raise ValueError(f"{name} has {p.numel()} elements, expected {n}")
    return p.contiguous()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


_ws_cache: dict = {}


def workspace(op: int, M: int, N: int, xt: int, pt: int, device: torch.device):
    """A cached device scratch buffer large enough for one backward call."""
    n = load().gbn_bwd_workspace_bytes(op, M, N, xt, pt, device.index)
    if n == SIZE_MAX:
        raise GbnError(1, "gbn_bwd_workspace_bytes")
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < n:
        buf = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf, n


def read_faults(clear: bool = True) -> int:
    """The current device's fault word (synchronizes); 0 when healthy."""
    v = ctypes.c_uint(0)
    _check(load().gbn_read_faults(ctypes.byref(v), int(clear)), "gbn_read_faults")
    return v.value


# ---------------------------------------------------------------------- DyT

def dyt_fwd(x, alpha, gamma, beta, y=None):
    """y = gamma * tanh(alpha * x) + beta (alpha: 1 element)."""
    x, xl, _, _, M, N = _input_rows(x)
    alpha = _param(alpha, x, 1, "alpha")
    gamma = _param(gamma, x, N, "gamma")
    beta = _param(beta, x, N, "beta")
    if beta.dtype != gamma.dtype or alpha.dtype != gamma.dtype:
        raise TypeError("alpha, gamma and beta must share one dtype")
    y = _out(x) if y is None else y
    if xl is None:
        st = load().dyt_fwd(_ptr(x), _ptr(alpha), _ptr(gamma), _ptr(beta), _ptr(y), M, N,
                            _code(x), _code(gamma), _stream(x.device))
    else:
        st = load().dyt_fwd_rows(_ptr(x), _lay(xl), _ptr(alpha), _ptr(gamma), _ptr(beta), _ptr(y),
                                 M, N, _code(x), _code(gamma), _stream(x.device))
    _check(st, "dyt_fwd")
    return y


def dyt_bwd(x, dy, alpha, gamma, need_dalpha=True, need_dgamma=True, need_dbeta=True):
    """(dx, dalpha, dgamma, dbeta); parameter gradients in gamma's dtype."""
    x, xl, dy, dyl, M, N = _input_rows(x, dy)
    alpha = _param(alpha, x, 1, "alpha")
    gamma = _param(gamma, x, N, "gamma")
    dx = _out(x)
    da = torch.empty(1, dtype=gamma.dtype, device=x.device) if need_dalpha else None
    dg = torch.empty(N, dtype=gamma.dtype, device=x.device) if need_dgamma else None
    db = torch.empty(N, dtype=gamma.dtype, device=x.device) if need_dbeta else None
    ws, nbytes = workspace(GBN_OP_DYT, M, N, _code(x), _code(gamma), x.device)
    _check(load().dyt_bwd_rows(_ptr(x), _lay(xl), _ptr(dy), _lay(dyl), _ptr(alpha), _ptr(gamma),
                               _ptr(dx), _ptr(da), _ptr(dg), _ptr(db), M, N, _code(x),
                               _code(gamma), _ptr(ws), nbytes, _stream(x.device)), "dyt_bwd")
    return dx, da, dg, db


# ---------------------------------------------------------------- LayerNorm

def layernorm_fwd(x, gamma=None, beta=None, eps=1e-5, save_stats=True):
    """(y, mean, rstd); mean/rstd are float32 [M] (None when not saved)."""
    x, xl, _, _, M, N = _input_rows(x)
    gamma = _param(gamma, x, N, "gamma", required=False)
    beta = _param(beta, x, N, "beta", required=False)
    if gamma is not None and beta is not None and gamma.dtype != beta.dtype:
        raise TypeError("gamma and beta must share one dtype")
    p = gamma if gamma is not None else beta
    pt = _code(p) if p is not None else GBN_F32
    y = _out(x)
    mean = torch.empty(M, dtype=torch.float32, device=x.device) if save_stats else None
    rstd = torch.empty(M, dtype=torch.float32, device=x.device) if save_stats else None
    _check(load().layernorm_fwd_rows(_ptr(x), _lay(xl), _ptr(gamma), _ptr(beta), _ptr(y),
                                     _ptr(mean), _ptr(rstd), M, N, float(eps), _code(x), pt,
                                     _stream(x.device)), "layernorm_fwd")
    return y, mean, rstd


def layernorm_bwd(x, dy, mean, rstd, gamma=None, need_dgamma=True, need_dbeta=True,
                  param_dtype=None):
    """(dx, dgamma, dbeta) from the forward's saved mean and rstd."""
    x, xl, dy, dyl, M, N = _input_rows(x, dy)
    gamma = _param(gamma, x, N, "gamma", required=False)
    mean = _param(mean, x, M, "mean").float()
    rstd = _param(rstd, x, M, "rstd").float()
    pdt = gamma.dtype if gamma is not None else (param_dtype or torch.float32)
    dx = _out(x)
    dg = torch.empty(N, dtype=pdt, device=x.device) if need_dgamma else None
    db = torch.empty(N, dtype=pdt, device=x.device) if need_dbeta else None
    pt = _DTYPES[pdt]
    ws, nbytes = workspace(GBN_OP_LAYERNORM, M, N, _code(x), pt, x.device)
    _check(load().layernorm_bwd_rows(_ptr(x), _lay(xl), _ptr(dy), _lay(dyl), _ptr(mean),
                                     _ptr(rstd), _ptr(gamma), _ptr(dx), _ptr(dg), _ptr(db), M, N,
                                     _code(x), pt, _ptr(ws), nbytes, _stream(x.device)),
           "layernorm_bwd")
    return dx, dg, db


# ------------------------------------------------------------------ RMSNorm

def rmsnorm_fwd(x, w, eps=1e-6, save_rstd=True, variant=GBN_RMS_CAST_FIRST):
    """(y, rstd): weight * (x.float() * rsqrt(mean(x^2) + eps)).to(x.dtype), or
    the weight-first / Gemma expression (variant, gbn_rms_variant)."""
    x, xl, _, _, M, N = _input_rows(x)
    w = _param(w, x, N, "w")
    y = _out(x)
    rstd = torch.empty(M, dtype=torch.float32, device=x.device) if save_rstd else None
    _check(load().rmsnorm_fwd_rows(_ptr(x), _lay(xl), _ptr(w), _ptr(y), _ptr(rstd), M, N,
                                   float(eps), _code(x), _code(w), int(variant),
                                   _stream(x.device)), "rmsnorm_fwd")
    return y, rstd


def rmsnorm_bwd(x, dy, w, rstd=None, eps=1e-6, need_dw=True, variant=GBN_RMS_CAST_FIRST):
    """(dx, dw); rstd None recomputes it exactly as the forward does."""
    x, xl, dy, dyl, M, N = _input_rows(x, dy)
    w = _param(w, x, N, "w")
    rstd = _param(rstd, x, M, "rstd", required=False)
    dx = _out(x)
    dw = torch.empty(N, dtype=w.dtype, device=x.device) if need_dw else None
    ws, nbytes = workspace(GBN_OP_RMSNORM, M, N, _code(x), _code(w), x.device)
    _check(load().rmsnorm_bwd_rows(_ptr(x), _lay(xl), _ptr(dy), _lay(dyl), _ptr(w), _ptr(rstd),
                                   _ptr(dx), _ptr(dw), M, N, float(eps), _code(x), _code(w),
                                   int(variant), _ptr(ws), nbytes, _stream(x.device)),
           "rmsnorm_bwd")
    return dx, dw


def rmsnorm_bwd_static_ws(x, dy, w, rstd=None, eps=1e-6, need_dw=True):
    """(dx, dw) like rmsnorm_bwd, with the library's static scratch array in
    place of a workspace allocated here: for callers that cannot allocate
    device memory.  Raises GbnError (GBN_ESCRATCH) when the shape needs more
    scratch than GBN_STATIC_WS_BYTES."""
    x, M, N = _rows(x)
    dy = dy.contiguous()
    if dy.shape != x.shape or dy.dtype != x.dtype:
        raise ValueError("dy must match x in shape and dtype")
    w = _param(w, x, N, "w")
    rstd = _param(rstd, x, M, "rstd", required=False)
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=w.dtype, device=x.device) if need_dw else None
    _check(load().rmsnorm_bwd_static_ws(_ptr(x), _ptr(dy), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw),
                                        M, N, float(eps), _code(x), _code(w), _stream(x.device)),
           "rmsnorm_bwd_static_ws")
    return dx, dw
