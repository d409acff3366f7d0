"""Run one layer forward + backward through the C ABI and compare every
output with the float64 oracle.

`rows=None` compares every row; otherwise only the listed rows of the
row-wise outputs (y, dx, saved statistics) are compared, while parameter
gradients are always compared in full against the oracle's column sums over
all rows.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from normalization_layers_fwd_gb300 import _lib
from _parity import check_f32, check_out, check_reduced, f64, to_oracle


def _sel(t, rows):
    if rows is None:
        return t
    return t.index_select(0, torch.as_tensor(rows, dtype=torch.long, device=t.device))


def _pcode(t):
    return {torch.bfloat16: oracle.BF16, torch.float16: oracle.F16}.get(t.dtype, oracle.F32)


def dyt_case(x, dy, alpha, gamma, beta, rows=None, cols=True):
    y = _lib.dyt_fwd(x, alpha, gamma, beta)
    dx, da, dg, db = _lib.dyt_bwd(x, dy, alpha, gamma)
    torch.cuda.synchronize()
    xo, dyo = to_oracle(x), to_oracle(dy)
    a = float(f64(alpha)[0])
    g64, b64 = f64(gamma), f64(beta)
    reps = []
    yo, ys = oracle.dyt_fwd(xo, a, g64, b64, rows)
    reps.append(check_out("dyt y", _sel(y, rows), yo, ys))
    dxo = oracle.dyt_bwd_rows(xo, dyo, a, g64, rows)
    reps.append(check_out("dyt dx", _sel(dx, rows), dxo, np.abs(dxo)))
    if cols:
        c = oracle.dyt_bwd_cols(xo, dyo, a, g64)
        reps.append(check_reduced("dyt dgamma", dg, c["dgamma"], c["dgamma_ss"]))
        reps.append(check_reduced("dyt dbeta", db, c["dbeta"], c["dbeta_ss"]))
        reps.append(check_reduced("dyt dalpha", da, [c["dalpha"]], [c["dalpha_ss"]]))
    return reps, dict(y=y, dx=dx, da=da, dg=dg, db=db)


def layernorm_case(x, dy, gamma, beta, eps, rows=None, cols=True, stats=None):
    reps = []
    xo, dyo = to_oracle(x), to_oracle(dy)
    g64 = None if gamma is None else f64(gamma)
    b64 = None if beta is None else f64(beta)
    out = {}
    if stats is None:
        y, mean, rstd = _lib.layernorm_fwd(x, gamma, beta, eps)
        torch.cuda.synchronize()
        yo, ys, muo, rso = oracle.ln_fwd(xo, eps, g64, b64, rows)
        reps.append(check_out("ln y", _sel(y, rows), yo, ys))
        reps.append(check_f32("ln mean", _sel(mean, rows), muo, np.maximum(np.abs(muo), 1 / rso)))
        reps.append(check_f32("ln rstd", _sel(rstd, rows), rso, np.abs(rso)))
        out["y"] = y
    else:
        mean, rstd = stats
    dx, dg, db = _lib.layernorm_bwd(x, dy, mean, rstd, gamma, param_dtype=torch.float32
                                    if gamma is None else None)
    torch.cuda.synchronize()
    mu64, rs64 = f64(mean), f64(rstd)
    dxo, dxs = oracle.ln_bwd_rows(xo, dyo, mu64, rs64, g64, rows)
    # at width two x-hat is +-sqrt(var / (var + eps)), so dx is eps / (var + eps)
    # times the size of its terms: all cancellation, as at width one
    reps.append(check_out("ln dx", _sel(dx, rows), dxo, dxs, cap=x.shape[-1] > 2))
    if cols:
        c = oracle.ln_bwd_cols(xo, dyo, mu64, rs64)
        reps.append(check_reduced("ln dgamma", dg, c["dgamma"], c["dgamma_ss"]))
        reps.append(check_reduced("ln dbeta", db, c["dbeta"], c["dbeta_ss"]))
    out.update(dx=dx, dg=dg, db=db, mean=mean, rstd=rstd)
    return reps, out


def rmsnorm_case(x, dy, w, eps, rows=None, cols=True, variant=0):
    """variant: the library's RMSNorm expression code (0 Llama, 1 weight
    first, 2 Gemma), compared with the oracle's expression of that name."""
    reps = []
    ov = {0: oracle.RMS_CAST_FIRST, 1: oracle.RMS_WEIGHT_FIRST, 2: oracle.RMS_GEMMA}[variant]
    y, rstd = _lib.rmsnorm_fwd(x, w, eps, variant=variant)
    dx, dw = _lib.rmsnorm_bwd(x, dy, w, rstd, eps, variant=variant)
    dx2, dw2 = _lib.rmsnorm_bwd(x, dy, w, None, eps, variant=variant)
    torch.cuda.synchronize()
    # the saved rstd is a cache: recomputing it must give identical bits
    def bits(t):
        return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)
    assert torch.equal(bits(dx), bits(dx2))
    assert torch.equal(bits(dw), bits(dw2))
    xo, dyo = to_oracle(x), to_oracle(dy)
    w64 = f64(w)
    yo, ys, rso, yal = oracle.rms_fwd(xo, eps, w64, oracle.PARITY, rows, variant=ov)
    reps.append(check_out("rms y", _sel(y, rows), yo, ys, yal))
    reps.append(check_f32("rms rstd", _sel(rstd, rows), rso, np.abs(rso)))
    dxo, dxs, dxal = oracle.rms_bwd_rows(xo, dyo, eps, w64, _pcode(w), oracle.PARITY, rows,
                                         variant=ov)
    reps.append(check_out("rms dx", _sel(dx, rows), dxo, dxs, dxal))
    if cols:
        dwo, ss, al = oracle.rms_bwd_cols(xo, dyo, eps, _pcode(w), oracle.PARITY, variant=ov)
        reps.append(check_reduced("rms dw", dw, dwo, ss, al))
    return reps, dict(y=y, rstd=rstd, dx=dx, dw=dw)


def run_workload(wl, device="cuda", rows=None, cols=True, inputs=None):
    """Generate a workload's inputs on `device` and run its case."""
    inp = inputs if inputs is not None else wl.inputs(device=device)
    if wl.op == "dyt":
        return dyt_case(inp["x"], inp["dy"], inp["alpha"], inp["gamma"], inp["beta"], rows, cols)
    if wl.op == "layernorm":
        return layernorm_case(inp["x"], inp["dy"], inp.get("gamma"), inp.get("beta"), wl.eps, rows,
                              cols)
    return rmsnorm_case(inp["x"], inp["dy"], inp["weight"], wl.eps, rows, cols)
