"""Comparison rules between the CUDA outputs and the float64 oracle.

Tolerances (each rule names the arithmetic it comes from):

* bfloat16 (and IEEE binary16) outputs must lie within 1 ULP of the
  nearest bf16 (f16) value to o, o being the
  oracle's float64 value before the final rounding.  The ULP distance is
  taken from ordered bit patterns, as the fused-RMSNorm page measures it
  (DeepSpeed PR 8645 quoted in PR 8664, "Correctness evidence (1)").
  Two counted exceptions, never silent:
  - cancellation: |g - o| <= max(2^-19 * scale, 2^-120), where scale is the
    sum of the magnitudes of the final expression's addends.  The kernels
    compute in float32 (unit roundoff 2^-24); 2^-19 leaves 32 roundings of
    headroom.  This is the page's "8 ULP or absolute 1e-7" input-gradient
    rule (PR 8664 review follow-up) made relative to the data's magnitude;
  - near-tie intermediate rounding (RMSNorm only): where a value passed
    through a bfloat16 rounding point within 2^-17 of a midpoint, a float32
    kernel may round it to the other neighbour; the oracle returns the
    largest change that flip causes ("allow"), and then
    |g - o| <= allow + ulp(bf16(o)).
* float32 outputs: |g - o| <= 1e-5 * max(|o|, scale) (+ 2^-120).
* reduced gradients (column sums): |g - o| <= 1e-4 * max(|o|, sqrt(sum of
  squared terms)); in bfloat16 either that or 1 ULP of bf16(o).
* NaN positions must agree exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

CANCEL_REL = 2.0 ** -19
TINY = 2.0 ** -120
F32_RTOL = 1e-5
RED_RTOL = 1e-4
MAX_EXCEPTION_FRAC = 1e-3


# ------------------------------------------------------------ conversions

def to_oracle(t: torch.Tensor) -> np.ndarray:
    """Activation tensor -> the oracle's input array (exact), [rows, N]."""
    t = t.detach().cpu().contiguous()
    if t.dim() > 2:
        t = t.reshape(-1, t.shape[-1])
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).reshape(t.shape)
    if t.dtype in (torch.float32, torch.float16):
        return t.numpy()
    raise TypeError(t.dtype)


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a float32/bfloat16 tensor."""
    return t.detach().cpu().to(torch.float64).numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_of_f64(v: np.ndarray, fmt: str = "bf16") -> np.ndarray:
    """Bit patterns of float64 values exactly representable in fmt (bf16/f16)."""
    v = np.asarray(v, dtype=np.float64)
    if fmt == "f16":
        with np.errstate(over="ignore"):
            return v.astype(np.float16).view(np.uint16)
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_distance_bf16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(ordered(a_bits) - ordered(b_bits))


def bf16_ulp(v: np.ndarray, fmt: str = "bf16") -> np.ndarray:
    """Spacing of fmt at |v| (v representable): bfloat16 keeps 8 significant
    bits down to 2^-126, binary16 11 bits down to 2^-14."""
    bits, emin = (11, -14.0) if fmt == "f16" else (8, -126.0)
    a = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.where(np.isfinite(a), 2.0 ** (e - (bits - 1)), np.inf)


_ROUND = {"bf16": lambda v: oracle.round_bf16_array(v), "f16": lambda v: oracle.round_f16_array(v)}


def fmt_of(t: torch.Tensor):
    return {torch.bfloat16: "bf16", torch.float16: "f16"}.get(t.dtype)


# ------------------------------------------------------------------ checks

class Report(dict):
    def line(self):
        return " ".join(f"{k}={v}" for k, v in self.items())


def _fail(name, mask, g, o, extra=""):
    idx = np.argwhere(mask)[:5]
    items = [(tuple(int(i) for i in ix), float(g[tuple(ix)]), float(o[tuple(ix)])) for ix in idx]
    raise AssertionError(f"{name}: {int(mask.sum())} of {mask.size} elements out of tolerance; "
                         f"first (index, gpu, oracle): {items} {extra}")


def check_nan(name, g, o):
    ng, no = np.isnan(g), np.isnan(o)
    if not np.array_equal(ng, no):
        _fail(name + " NaN positions", ng != no, g, o)
    return ng


def check_bf16(name, g_t: torch.Tensor, o, scale, allow=None, cap=True) -> Report:
    """16-bit (bfloat16 or binary16) output vs oracle value o (float64,
    before rounding).

    The cap on counted exceptions does not apply at width one, where the
    input gradient is (nearly) all cancellation: DeepSpeed PR 8664 notes
    that a width-one norm's computed input gradient is rounding noise.
    cap=False lifts it for other such outputs (LayerNorm's input gradient
    at width two, eps / (var + eps) times the size of its terms); every
    element must still be within 1 ULP or the cancellation bound."""
    fmt = fmt_of(g_t)
    gb = bf16_bits(g_t).reshape(o.shape)
    g = f64(g_t).reshape(o.shape)
    nan = check_nan(name, g, o)
    ref = _ROUND[fmt](np.where(nan, 0.0, o))
    rb = bits_of_f64(ref, fmt)
    d = ulp_distance_bf16(gb, rb)
    d = np.where(nan, 0, d)
    both_inf = np.isinf(g) & np.isinf(ref) & (np.sign(g) == np.sign(ref))
    d = np.where(both_inf, 0, d)
    with np.errstate(invalid="ignore"):
        err = np.abs(g - o)
    ok1 = d <= 1
    okc = err <= np.maximum(CANCEL_REL * scale, TINY)
    oka = (np.zeros_like(ok1) if allow is None
           else ((allow > 0) & (err <= allow + bf16_ulp(ref, fmt))))
    bad = ~(ok1 | okc | oka | nan)
    if bad.any():
        _fail(name, bad, g, o, f"(max ulp {int(d[bad].max())})")
    exc = (~ok1) & ~nan
    n = int(o.size)
    if cap and o.ndim == 2 and o.shape[1] > 1 and exc.sum() > max(8, MAX_EXCEPTION_FRAC * n):
        raise AssertionError(f"{name}: {int(exc.sum())} counted exceptions in {n} elements")
    within1 = float(np.mean(ok1 | nan)) if n else 1.0
    with np.errstate(invalid="ignore"):
        policy = np.abs(g - ref) <= 2.0 ** -6 + 2.0 ** -6 * np.abs(ref)
    return Report(name=name, n=n, max_ulp=int(d.max()) if n else 0, within_1ulp=round(within1, 6),
                  cancel_exc=int((exc & okc).sum()), tie_exc=int((exc & oka & ~okc).sum()),
                  bf16_policy_violations=int((~policy & ~nan).sum()))


def check_f32(name, g_t: torch.Tensor, o, scale, allow=None, rtol=F32_RTOL) -> Report:
    g = f64(g_t).reshape(o.shape)
    nan = check_nan(name, g, o)
    with np.errstate(invalid="ignore"):
        err = np.abs(g - o)
        tol = rtol * np.maximum(np.abs(o), scale) + TINY + (0 if allow is None else allow)
    bad = ~(err <= tol) & ~nan
    if bad.any():
        _fail(name, bad, g, o)
    with np.errstate(invalid="ignore", divide="ignore"):
        rel = np.where(nan, 0.0, err / np.maximum(np.abs(o), scale))
    return Report(name=name, n=int(o.size), max_rel=float(np.nanmax(rel)) if o.size else 0.0)


def check_reduced(name, g_t: torch.Tensor, o, ss, allow=None) -> Report:
    """A parameter gradient (column sum) in its parameter dtype."""
    o = np.asarray(o, dtype=np.float64).reshape(-1)
    ss = np.asarray(ss, dtype=np.float64).reshape(-1)
    g = f64(g_t).reshape(-1)
    nan = check_nan(name, g, o)
    with np.errstate(invalid="ignore"):
        err = np.abs(g - o)
    tol = RED_RTOL * np.maximum(np.abs(o), np.sqrt(ss)) + TINY
    if allow is not None:
        tol = tol + np.asarray(allow, dtype=np.float64).reshape(-1)
    ok = err <= tol
    fmt = fmt_of(g_t)
    if fmt:
        ref = _ROUND[fmt](np.where(nan, 0.0, o))
        d = ulp_distance_bf16(bf16_bits(g_t).reshape(-1), bits_of_f64(ref, fmt))
        ok = ok | (d <= 1)
    bad = ~ok & ~nan
    if bad.any():
        _fail(name, bad, g, o)
    with np.errstate(invalid="ignore", divide="ignore"):
        rel = np.where(nan, 0.0, err / np.maximum(np.abs(o), np.sqrt(ss)))
    return Report(name=name, n=int(o.size), max_rel=float(np.nanmax(rel)) if o.size else 0.0)


def check_out(name, g_t, o, scale, allow=None, cap=True):
    if fmt_of(g_t):
        return check_bf16(name, g_t, o, scale, allow, cap)
    return check_f32(name, g_t, o, scale, allow)
