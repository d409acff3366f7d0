"""Float64 CPU oracle for DyT, LayerNorm and RMSNorm (forward and backward).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
baseline leg of the benchmark may import this package; the product path
never does.  The arithmetic lives in ``oracle.c`` (plain C, float64, serial
sums in index order); this module only builds that file with gcc, marshals
numpy arrays to it and returns numpy arrays.

Inputs are numpy arrays: ``float32``, ``float64``, ``float16`` or
``uint16`` (raw bfloat16 bit patterns).  They are widened exactly inside the C code.
Parameters (gamma, beta, weight) are passed as float64 arrays holding the
exact values of the stored parameters.

Every function returns float64 values *before* the final rounding to the
output dtype; the tests apply that rounding and the tolerance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, F64, F16 = 0, 1, 2, 3
MATH, PARITY = 0, 1
# RMSNorm expression variants: weight after the cast (Llama), weight before
# the cast, and Gemma's (1 + weight) before the cast.
RMS_CAST_FIRST, RMS_WEIGHT_FIRST, RMS_GEMMA = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_handle = None

# -ffp-contract=off keeps gcc from fusing multiply-adds, so x86 and Arm hosts
# evaluate every expression with the same roundings.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (idempotent); return its path."""
    with _lock:
        fresh = os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)
        if fresh and not force:
            return _SO
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
        return _SO


def _lib():
    global _handle
    if _handle is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        sigs = {
            "orc_round_bf16": ([D], D),
            "orc_bf16_near_tie": ([D], I),
            "orc_round_bf16_array": ([P, P, I64], None),
            "orc_round_f16": ([D], D),
            "orc_round_f16_array": ([P, P, I64], None),
            "orc_dyt_fwd_rows": ([P, I, I64, I64, D, P, P, P, I64, P, P], I),
            "orc_dyt_bwd_rows": ([P, P, I, I64, I64, D, P, P, I64, P], I),
            "orc_dyt_bwd_cols": ([P, P, I, I64, I64, D, P, P, P, P, P, P, P], I),
            "orc_ln_fwd_rows": ([P, I, I64, I64, D, P, P, P, I64, P, P, P, P], I),
            "orc_ln_bwd_rows": ([P, P, I, I64, I64, P, P, P, P, I64, P, P], I),
            "orc_ln_bwd_cols": ([P, P, I, I64, I64, P, P, P, P, P, P], I),
            "orc_rms_fwd_rows": ([P, I, I64, I64, D, P, I, I, P, I64, P, P, P, P], I),
            "orc_rms_bwd_rows": ([P, P, I, I, I64, I64, D, P, I, I, P, I64, P, P, P], I),
            "orc_rms_bwd_cols": ([P, P, I, I, I64, I64, D, I, I, P, P, P], I),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _handle = lib
    return _handle


# ------------------------------------------------------------------ helpers

def _act(a: np.ndarray):
    """Activation array -> (contiguous array, dtype code, M, N)."""
    a = np.ascontiguousarray(a)
    if a.ndim != 2:
        raise ValueError("activations must be 2-D [M, N]")
    code = {np.dtype(np.float32): F32, np.dtype(np.uint16): BF16,
            np.dtype(np.float64): F64, np.dtype(np.float16): F16}.get(a.dtype)
    if code is None:
        raise TypeError(f"unsupported activation dtype {a.dtype}")
    return a, code, a.shape[0], a.shape[1]


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= M):
        raise IndexError("row index out of range")
    return r, r.size


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} returned {rc}")


# -------------------------------------------------------------- rounding

def round_bf16(v: float) -> float:
    """float64 -> nearest bfloat16 value (ties to even), returned as float."""
    return _lib().orc_round_bf16(float(v))


def round_bf16_array(a) -> np.ndarray:
    """Elementwise float64 -> nearest bfloat16 value, as float64."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    out = np.empty_like(a)
    _lib().orc_round_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_near_tie(v: float) -> bool:
    return bool(_lib().orc_bf16_near_tie(float(v)))


def round_f16(v: float) -> float:
    """float64 -> nearest IEEE binary16 value (ties to even), as float."""
    return _lib().orc_round_f16(float(v))


def round_f16_array(a) -> np.ndarray:
    """Elementwise float64 -> nearest binary16 value, as float64."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    out = np.empty_like(a)
    _lib().orc_round_f16_array(_ptr(a), _ptr(out), a.size)
    return out


# ------------------------------------------------------------------- DyT

def dyt_fwd(x, alpha, gamma, beta, rows=None):
    """y (before output rounding) and its scale |gamma t| + |beta|."""
    x, xt, M, N = _act(x)
    g, b = _f64(gamma), _f64(beta)
    r, nr = _rows(rows, M)
    y = np.empty((nr, N)); ys = np.empty((nr, N))
    _check(_lib().orc_dyt_fwd_rows(_ptr(x), xt, M, N, float(alpha), _ptr(g), _ptr(b),
                                   _ptr(r), nr, _ptr(y), _ptr(ys)), "dyt_fwd")
    return y, ys


def dyt_bwd_rows(x, dy, alpha, gamma, rows=None):
    x, xt, M, N = _act(x)
    dy, dt, _, _ = _act(dy)
    assert dt == xt and dy.shape == x.shape
    g = _f64(gamma)
    r, nr = _rows(rows, M)
    dx = np.empty((nr, N))
    _check(_lib().orc_dyt_bwd_rows(_ptr(x), _ptr(dy), xt, M, N, float(alpha), _ptr(g),
                                   _ptr(r), nr, _ptr(dx)), "dyt_bwd_rows")
    return dx


def dyt_bwd_cols(x, dy, alpha, gamma):
    x, xt, M, N = _act(x)
    dy, dt, _, _ = _act(dy)
    assert dt == xt and dy.shape == x.shape
    g = _f64(gamma)
    out = {k: np.empty(N) for k in ("dgamma", "dgamma_ss", "dbeta", "dbeta_ss")}
    da = np.empty(1); da_ss = np.empty(1)
    _check(_lib().orc_dyt_bwd_cols(_ptr(x), _ptr(dy), xt, M, N, float(alpha), _ptr(g),
                                   _ptr(out["dgamma"]), _ptr(out["dgamma_ss"]),
                                   _ptr(out["dbeta"]), _ptr(out["dbeta_ss"]),
                                   _ptr(da), _ptr(da_ss)), "dyt_bwd_cols")
    out["dalpha"] = float(da[0]); out["dalpha_ss"] = float(da_ss[0])
    return out


# ------------------------------------------------------------- LayerNorm

def ln_fwd(x, eps, gamma=None, beta=None, rows=None):
    """(y, y_scale, mean, rstd) in float64."""
    x, xt, M, N = _act(x)
    g, b = _f64(gamma), _f64(beta)
    r, nr = _rows(rows, M)
    y = np.empty((nr, N)); ys = np.empty((nr, N)); mu = np.empty(nr); rs = np.empty(nr)
    _check(_lib().orc_ln_fwd_rows(_ptr(x), xt, M, N, float(eps), _ptr(g), _ptr(b), _ptr(r),
                                  nr, _ptr(y), _ptr(ys), _ptr(mu), _ptr(rs)), "ln_fwd")
    return y, ys, mu, rs


def ln_bwd_rows(x, dy, mean, rstd, gamma=None, rows=None):
    """(dx, dx_scale); mean/rstd are the saved per-row statistics of ALL rows."""
    x, xt, M, N = _act(x)
    dy, dt, _, _ = _act(dy)
    assert dt == xt and dy.shape == x.shape
    mu, rs, g = _f64(mean), _f64(rstd), _f64(gamma)
    assert mu.shape == (M,) and rs.shape == (M,)
    r, nr = _rows(rows, M)
    dx = np.empty((nr, N)); dxs = np.empty((nr, N))
    _check(_lib().orc_ln_bwd_rows(_ptr(x), _ptr(dy), xt, M, N, _ptr(mu), _ptr(rs), _ptr(g),
                                  _ptr(r), nr, _ptr(dx), _ptr(dxs)), "ln_bwd_rows")
    return dx, dxs


def ln_bwd_cols(x, dy, mean, rstd):
    x, xt, M, N = _act(x)
    dy, dt, _, _ = _act(dy)
    assert dt == xt and dy.shape == x.shape
    mu, rs = _f64(mean), _f64(rstd)
    out = {k: np.empty(N) for k in ("dgamma", "dgamma_ss", "dbeta", "dbeta_ss")}
    _check(_lib().orc_ln_bwd_cols(_ptr(x), _ptr(dy), xt, M, N, _ptr(mu), _ptr(rs),
                                  _ptr(out["dgamma"]), _ptr(out["dgamma_ss"]),
                                  _ptr(out["dbeta"]), _ptr(out["dbeta_ss"])), "ln_bwd_cols")
    return out


# --------------------------------------------------------------- RMSNorm

def rms_fwd(x, eps, w, mode=PARITY, rows=None, variant=RMS_CAST_FIRST):
    """(y, y_scale, rstd, y_allow).  y_allow: largest change of y that a
    float32 implementation may legitimately show where the rounding of the
    normalized value is near a bfloat16 tie (zero elsewhere)."""
    x, xt, M, N = _act(x)
    wv = _f64(w)
    r, nr = _rows(rows, M)
    y = np.empty((nr, N)); ys = np.empty((nr, N)); rs = np.empty(nr); al = np.empty((nr, N))
    _check(_lib().orc_rms_fwd_rows(_ptr(x), xt, M, N, float(eps), _ptr(wv), int(mode),
                                   int(variant), _ptr(r), nr, _ptr(y), _ptr(ys), _ptr(rs),
                                   _ptr(al)), "rms_fwd")
    return y, ys, rs, al


def rms_bwd_rows(x, dy, eps, w, w_dtype_code=F32, mode=PARITY, rows=None,
                 variant=RMS_CAST_FIRST):
    """(dx, dx_scale, dx_allow); w_dtype_code is F32 or the activation's 16-bit code."""
    x, xt, M, N = _act(x)
    dy, dt, _, _ = _act(dy)
    assert dt == xt and dy.shape == x.shape
    wv = _f64(w)
    r, nr = _rows(rows, M)
    dx = np.empty((nr, N)); dxs = np.empty((nr, N)); al = np.empty((nr, N))
    _check(_lib().orc_rms_bwd_rows(_ptr(x), _ptr(dy), xt, int(w_dtype_code), M, N, float(eps),
                                   _ptr(wv), int(mode), int(variant), _ptr(r), nr, _ptr(dx),
                                   _ptr(dxs), _ptr(al)),
           "rms_bwd_rows")
    return dx, dxs, al


def rms_bwd_cols(x, dy, eps, w_dtype_code, mode=PARITY, variant=RMS_CAST_FIRST):
    """(dw, dw_ss, dw_allow); w_dtype_code is F32 or the activation's 16-bit code
    (selects the term rounding)."""
    x, xt, M, N = _act(x)
    dy, dt, _, _ = _act(dy)
    assert dt == xt and dy.shape == x.shape
    dw = np.empty(N); ss = np.empty(N); al = np.empty(N)
    _check(_lib().orc_rms_bwd_cols(_ptr(x), _ptr(dy), xt, int(w_dtype_code), M, N, float(eps),
                                   int(mode), int(variant), _ptr(dw), _ptr(ss), _ptr(al)),
           "rms_bwd_cols")
    return dw, ss, al
