"""Bit-identical reruns at the benchmark workloads' full sizes.

Every workload (the four fixed shapes, the alpha = +inf edge case, and the
30 points of the width sweep) runs its forward and backward three times on
the same inputs, in the launch layout the benchmark times, and every output
is compared bytewise with the first run's: y, dx, the saved statistics and
every parameter gradient (dgamma, dbeta, dalpha, dweight).  The DeepSpeed
PR 8664 page ("Numerics") asks that identical fused runs give repeatable
input and weight gradients; here the fixed launch table and the
atomic-free two-stage column sums make that hold for every output, and
these tests check it where the persistent grid loops over many row blocks
and the partial-row count sits at its SM cap.
"""
from __future__ import annotations

import pytest
import torch

from normalization_layers_fwd_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

REPEATS = 3


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from normalization_layers_fwd_gb300 import build
    build.build()
    _lib.load()


def run_once(wl, inp):
    """Every output of one forward + backward (the backward alone, on the
    forward's saved statistics, for the backward-only workload)."""
    x, dy = inp["x"], inp["dy"]
    if wl.op == "dyt":
        y = _lib.dyt_fwd(x, inp["alpha"], inp["gamma"], inp["beta"])
        dx, da, dg, db = _lib.dyt_bwd(x, dy, inp["alpha"], inp["gamma"])
        return {"y": y, "dx": dx, "dalpha": da, "dgamma": dg, "dbeta": db}
    if wl.op == "layernorm":
        y, mean, rstd = _lib.layernorm_fwd(x, inp["gamma"], inp["beta"], wl.eps)
        dx, dg, db = _lib.layernorm_bwd(x, dy, mean, rstd, inp["gamma"])
        out = {"mean": mean, "rstd": rstd, "dx": dx, "dgamma": dg, "dbeta": db}
        if not wl.bwd_only:
            out["y"] = y
        return out
    y, rstd = _lib.rmsnorm_fwd(x, inp["weight"], wl.eps)
    dx, dw = _lib.rmsnorm_bwd(x, dy, inp["weight"], rstd, wl.eps)
    return {"y": y, "rstd": rstd, "dx": dx, "dweight": dw}


def _bits(t):
    return t.contiguous().view(torch.uint8)


WORKLOADS = [synth.DYT_F32_SMALL, synth.LN_BWD_TALL, synth.DYT_BF16_TALL,
             synth.DYT_BF16_ALPHA_INF, synth.RMS_BF16] + synth.sweep_all()


@pytest.mark.parametrize("wl", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_reruns_are_bit_identical(wl):
    inp = wl.inputs(device="cuda")
    first = run_once(wl, inp)
    torch.cuda.synchronize()
    assert first, wl.name
    for rep in range(2, REPEATS + 1):
        again = run_once(wl, inp)
        torch.cuda.synchronize()
        assert again.keys() == first.keys()
        for k, t in first.items():
            assert t.dtype == again[k].dtype and t.shape == again[k].shape
            assert torch.equal(_bits(t), _bits(again[k])), f"{wl.name} {k}: run {rep} differs"
        del again
    del first, inp
    torch.cuda.empty_cache()
