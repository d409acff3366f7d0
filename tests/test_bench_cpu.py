"""bench.py's host logic without a GPU: the algorithmic bytes per launch,
the workloads' shapes, and the JSON line of the reference arm (the float64
oracle, which runs on the host)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from normalization_layers_fwd_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("M,N,sx,sp", [(4096, 64, 4, 4), (1 << 21, 128, 2, 4), (7, 24, 2, 2)])
def test_alg_bytes_per_launch(M, N, sx, sp):
    """What each launch must move: activations read and written, the saved
    statistics (fp32 per row), the parameters read and their gradients
    written."""
    E = M * N
    assert bench.alg_bytes("dyt", "fwd", M, N, sx, sp) == 2 * E * sx + (2 * N + 1) * sp
    assert bench.alg_bytes("dyt", "bwd", M, N, sx, sp) == 3 * E * sx + (N + 1) * sp + (2 * N + 1) * sp
    assert bench.alg_bytes("layernorm", "fwd", M, N, sx, sp) == 2 * E * sx + 8 * M + 2 * N * sp
    assert bench.alg_bytes("layernorm", "bwd", M, N, sx, sp) == 3 * E * sx + 8 * M + 3 * N * sp
    assert bench.alg_bytes("rmsnorm", "fwd", M, N, sx, sp) == 2 * E * sx + 4 * M + N * sp
    assert bench.alg_bytes("rmsnorm", "bwd", M, N, sx, sp) == 3 * E * sx + 4 * M + 2 * N * sp


def test_sweep_workload_shapes():
    wls, desc = bench.workloads("sweep")
    assert len(wls) == 30
    assert sorted({w.N for w in wls}) == sorted(synth.SWEEP_WIDTHS)
    for w in wls:
        assert w.M == (1 << 28) // w.N
        assert w.op in ("dyt", "layernorm", "rmsnorm")
    assert "sweep" in desc


def test_headmajor_workload_shapes():
    wls, _ = bench.workloads("headmajor")
    B, H, S, D = bench.HEAD_MAJOR
    assert [w.op for w in wls] == ["dyt", "layernorm", "rmsnorm"]
    for w in wls:
        assert (w.M, w.N, w.lead) == (B * H * S, D, (B, H, S))
    # a small case of the same recipe: the storage is [B, H, S, D], x its
    # transposed view, and the oracle sample takes contiguous rows
    small = synth.head_major("rmsnorm", 1, 3, 5, 16).inputs()
    assert tuple(small["x_storage"].shape) == (1, 3, 5, 16)
    assert tuple(small["x"].shape) == (1, 5, 3, 16)
    assert synth.scaled(wls[0], 10).lead is None


def test_reference_arm_json_line():
    """The oracle arm prints one JSON line with the contract's keys."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-elems", "30000"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_cpu_baseline_times_all_cores_and_one():
    """The CPU baseline runs the oracle on static row blocks over several
    threads and on one thread, over the same sample (the same bytes), and
    records the host's core count and CPU model."""
    wls, _ = bench.workloads("sweep")
    wls = [w for w in wls if w.N in (24, 512)]
    b1, s1, d1 = bench.oracle_sample(wls, 60000, 1)
    b3, s3, d3 = bench.oracle_sample(wls, 60000, 3)
    assert b1 == b3 and s1 > 0 and s3 > 0
    assert "one thread" in d1 and "3 threads" in d3
    cb = bench.cpu_baseline(wls, 60000, 2)
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] > 0
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert cb["nproc"] >= 1 and cb["usable_cores"] >= 1 and cb["cpu_model"]


def test_extra_widths_are_off_the_sweep_paths():
    """The extra breakdown points sit outside the sweep's widths: rows that
    are not 16-byte multiples, and rows wider than 1024 vectors."""
    for N, xd in bench.EXTRA_WIDTHS:
        assert N not in synth.SWEEP_WIDTHS or xd != synth.sweep("dyt", N).xdtype
        row_bytes = N * xd.itemsize
        assert row_bytes % 16 != 0 or row_bytes // 16 > 1024
        w = synth.sweep("layernorm", N, xd)
        assert w.M == (1 << 28) // N and w.xdtype == xd


def test_recorded_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu capture only while the
    kernel sources hash to the value recorded with it; any other hash, or a
    launch the capture does not hold, gives None."""
    key = "layernorm_bwd[16777216x16]"
    rec = {"source_hash": bench.source_hash(),
           "launches": {key: {"dram_read": 1000, "dram_write": 234}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # source_hash reads the kernel sources under ROOT: keep it on the real tree
    real_hash = rec["source_hash"]
    monkeypatch.setattr(bench, "source_hash", lambda: real_hash)
    assert bench.recorded_traffic(key) == 1234
    assert bench.recorded_traffic("dyt_fwd[1x16]") is None
    rec["source_hash"] = "0" * 16
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic(key) is None
