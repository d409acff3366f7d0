"""GPU parity at the benchmark workloads' full sizes, in the launch layout the
benchmark times.

Row-wise outputs (y, dx, saved statistics) are compared on sampled rows,
which the oracle computes one by one; parameter gradients are compared in
full against the oracle's float64 column sums over every row.  The oracle
calls run on a thread pool (each call is single-threaded C that releases
the GIL), one call per workload.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import threading

import numpy as np
import pytest
import torch

import oracle
from _parity import check_f32, check_out, check_reduced, f64, to_oracle
from normalization_layers_fwd_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

SAMPLE_ROWS = 1024


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from normalization_layers_fwd_gb300 import build
    build.build()
    _lib.load()


def sample_rows(M, seed):
    rng = np.random.default_rng(seed)
    r = set(rng.integers(0, M, SAMPLE_ROWS).tolist()) | {0, 1, M // 2, M - 2, M - 1}
    return np.array(sorted(x for x in r if 0 <= x < M), dtype=np.int64)


def _sel(t, rows):
    return t.index_select(0, torch.as_tensor(rows, device=t.device)).cpu()


def _pcode(t):
    return oracle.BF16 if t.dtype == torch.bfloat16 else oracle.F32


def gpu_run(wl, stats_from_oracle=False):
    """Run forward + backward on the GPU; return host copies of what the
    oracle comparison needs (and nothing else stays on the device)."""
    inp = wl.inputs(device="cuda")
    x, dy = inp["x"], inp["dy"]
    rows = sample_rows(wl.M, synth.seed_for(wl.index, wl.name + "/rows"))
    host = {"rows": rows, "xo": to_oracle(x), "dyo": to_oracle(dy)}
    if wl.op == "dyt":
        y = _lib.dyt_fwd(x, inp["alpha"], inp["gamma"], inp["beta"])
        dx, da, dg, db = _lib.dyt_bwd(x, dy, inp["alpha"], inp["gamma"])
        host.update(y=_sel(y, rows), dx=_sel(dx, rows), da=da.cpu(), dg=dg.cpu(), db=db.cpu(),
                    alpha=float(f64(inp["alpha"])[0]), gamma=f64(inp["gamma"]),
                    beta=f64(inp["beta"]))
    elif wl.op == "layernorm":
        g, b = inp["gamma"], inp["beta"]
        if stats_from_oracle:
            # the backward-only workload: saved statistics come from the
            # oracle's forward, rounded once to float32, and feed both sides
            _, _, mu, rs = oracle.ln_fwd(host["xo"], wl.eps, None, None)
            mean = torch.from_numpy(mu.astype(np.float32)).cuda()
            rstd = torch.from_numpy(rs.astype(np.float32)).cuda()
        else:
            y, mean, rstd = _lib.layernorm_fwd(x, g, b, wl.eps)
            host.update(y=_sel(y, rows), mean_s=_sel(mean, rows), rstd_s=_sel(rstd, rows))
        dx, dg, db = _lib.layernorm_bwd(x, dy, mean, rstd, g)
        host.update(dx=_sel(dx, rows), dg=dg.cpu(), db=db.cpu(), mean=f64(mean), rstd=f64(rstd),
                    gamma=f64(g), beta=f64(b))
    else:
        w = inp["weight"]
        y, rstd = _lib.rmsnorm_fwd(x, w, wl.eps)
        dx, dw = _lib.rmsnorm_bwd(x, dy, w, rstd, wl.eps)
        host.update(y=_sel(y, rows), rstd_s=_sel(rstd, rows), dx=_sel(dx, rows), dw=dw.cpu(),
                    w=f64(w), wcode=_pcode(w))
    torch.cuda.synchronize()
    del inp
    return host


def oracle_check(wl, h):
    """Compare one workload's GPU results with the oracle; return reports."""
    xo, dyo, rows = h["xo"], h["dyo"], h["rows"]
    reps = []
    if wl.op == "dyt":
        yo, ys = oracle.dyt_fwd(xo, h["alpha"], h["gamma"], h["beta"], rows)
        reps.append(check_out(f"{wl.name} y", h["y"], yo, ys))
        dxo = oracle.dyt_bwd_rows(xo, dyo, h["alpha"], h["gamma"], rows)
        reps.append(check_out(f"{wl.name} dx", h["dx"], dxo, np.abs(dxo)))
        c = oracle.dyt_bwd_cols(xo, dyo, h["alpha"], h["gamma"])
        reps.append(check_reduced(f"{wl.name} dgamma", h["dg"], c["dgamma"], c["dgamma_ss"]))
        reps.append(check_reduced(f"{wl.name} dbeta", h["db"], c["dbeta"], c["dbeta_ss"]))
        reps.append(check_reduced(f"{wl.name} dalpha", h["da"], [c["dalpha"]], [c["dalpha_ss"]]))
    elif wl.op == "layernorm":
        if "y" in h:
            yo, ys, muo, rso = oracle.ln_fwd(xo, wl.eps, h["gamma"], h["beta"], rows)
            reps.append(check_out(f"{wl.name} y", h["y"], yo, ys))
            reps.append(check_f32(f"{wl.name} mean", h["mean_s"], muo,
                                  np.maximum(np.abs(muo), 1 / rso)))
            reps.append(check_f32(f"{wl.name} rstd", h["rstd_s"], rso, rso))
        dxo, dxs = oracle.ln_bwd_rows(xo, dyo, h["mean"], h["rstd"], h["gamma"], rows)
        reps.append(check_out(f"{wl.name} dx", h["dx"], dxo, dxs))
        c = oracle.ln_bwd_cols(xo, dyo, h["mean"], h["rstd"])
        reps.append(check_reduced(f"{wl.name} dgamma", h["dg"], c["dgamma"], c["dgamma_ss"]))
        reps.append(check_reduced(f"{wl.name} dbeta", h["db"], c["dbeta"], c["dbeta_ss"]))
    else:
        yo, ys, rso, yal = oracle.rms_fwd(xo, wl.eps, h["w"], oracle.PARITY, rows)
        reps.append(check_out(f"{wl.name} y", h["y"], yo, ys, yal))
        reps.append(check_f32(f"{wl.name} rstd", h["rstd_s"], rso, rso))
        dxo, dxs, dxal = oracle.rms_bwd_rows(xo, dyo, wl.eps, h["w"], h["wcode"], oracle.PARITY,
                                             rows)
        reps.append(check_out(f"{wl.name} dx", h["dx"], dxo, dxs, dxal))
        dwo, ss, al = oracle.rms_bwd_cols(xo, dyo, wl.eps, h["wcode"], oracle.PARITY)
        reps.append(check_reduced(f"{wl.name} dw", h["dw"], dwo, ss, al))
    return reps


def run_many(workloads, stats_from_oracle=False):
    """GPU work in this thread, oracle checks on a bounded thread pool."""
    workers = max(1, min(16, (os.cpu_count() or 2) - 1))
    gate = threading.Semaphore(workers + 2)  # bound host memory held by queued inputs
    futs = []

    def job(wl, h):
        try:
            return oracle_check(wl, h)
        finally:
            gate.release()

    with cf.ThreadPoolExecutor(workers) as ex:
        for wl in workloads:
            gate.acquire()
            futs.append(ex.submit(job, wl, gpu_run(wl, stats_from_oracle)))
        reps = []
        for f in futs:
            reps.extend(f.result())
    for r in reps:
        print(r.line())
    return reps


def test_workload_dyt_f32_4096x64():
    run_many([synth.DYT_F32_SMALL])


def test_workload_layernorm_bwd_401408x24():
    run_many([synth.LN_BWD_TALL], stats_from_oracle=True)


def test_workload_dyt_bf16_1048576x128_and_alpha_inf():
    run_many([synth.DYT_BF16_TALL, synth.DYT_BF16_ALPHA_INF])


def test_workload_rmsnorm_bf16_16384x2048():
    run_many([synth.RMS_BF16])


@pytest.mark.parametrize("op", ["dyt", "layernorm", "rmsnorm"])
def test_workload_sweep(op):
    run_many([synth.sweep(op, n) for n in synth.SWEEP_WIDTHS])
