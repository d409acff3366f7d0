"""GPU parity: every output of the CUDA path against the float64 oracle,
element by element, at sizes the oracle finishes in seconds that still span
several row blocks, persistent-loop iterations and a ragged tail.  All calls
go through the C ABI (the ctypes binding)."""
import math

import numpy as np
import pytest
import torch

import oracle
from _cases import dyt_case, layernorm_case, rmsnorm_case
from _golden import kv, shapes
from _parity import check_bf16, f64, to_oracle
from normalization_layers_fwd_gb300 import _lib, synth
from normalization_layers_fwd_gb300.functional import dyt, layer_norm, rms_norm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from normalization_layers_fwd_gb300 import build
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def _inputs(M, N, xdt, pdt, seed, device="cuda", x_std=1.0):
    s = lambda n: synth.seed_for(90, f"{seed}/{n}")  # noqa: E731
    return dict(
        x=synth.normal((M, N), 0.0, x_std, xdt, seed=s("x"), device=device),
        dy=synth.normal((M, N), 0.0, 1.0, xdt, seed=s("dy"), device=device),
        alpha=synth.normal((1,), 0.8, 0.1, pdt, seed=s("a"), device=device),
        gamma=synth.normal((N,), 1.0, 0.1, pdt, seed=s("g"), device=device),
        beta=synth.normal((N,), 0.0, 0.1, pdt, seed=s("b"), device=device),
    )


def _run(op, inp, eps=1e-5, rows=None):
    if op == "dyt":
        return dyt_case(inp["x"], inp["dy"], inp["alpha"], inp["gamma"], inp["beta"], rows)
    if op == "layernorm":
        return layernorm_case(inp["x"], inp["dy"], inp["gamma"], inp["beta"], eps, rows)
    return rmsnorm_case(inp["x"], inp["dy"], inp["gamma"], eps, rows)


# 16-bit widths 8200-16384 (1025-2048 vectors) and float32 widths 4104-8192
# run every kernel on the 4-vector wide schedule (the 16-bit backwards in
# their lean form); 8196 and 16392 are beyond it.  Widths up to 256 whose rows
# are not 16-byte multiples run the row-batched path: element pairs for even
# widths up to 256 (2, 6, 100, 130, 250), single elements for odd ones up to
# 128 (1, 5), rows narrower than 16 bytes included; 129, 255, 258 and 1001
# stay general.
BF16_WIDTHS = [1, 2, 5, 6, 8, 16, 24, 40, 64, 100, 127, 128, 129, 130, 136, 250, 255, 256, 258,
               264, 512, 520, 1000, 1001, 1024, 2048, 3072, 4096, 6000, 8192, 8200, 12288, 16384,
               16392]
F32_WIDTHS = [1, 2, 3, 4, 6, 12, 64, 100, 130, 250, 255, 256, 1024, 2048, 3000, 4096, 4100, 4104,
              6000, 8192, 8196]
F16_WIDTHS = [1, 5, 8, 16, 24, 40, 64, 128, 129, 130, 264, 1000, 2048, 3072, 4096, 6000, 8192,
              8200, 12288]
DTYPES = [(torch.bfloat16, torch.float32), (torch.bfloat16, torch.bfloat16),
          (torch.float32, torch.float32), (torch.float32, torch.bfloat16),
          (torch.float16, torch.float32), (torch.float16, torch.float16)]
WIDTHS = {torch.bfloat16: BF16_WIDTHS, torch.float32: F32_WIDTHS, torch.float16: F16_WIDTHS}
CASES = []
for xdt, pdt in DTYPES:
    for N in WIDTHS[xdt]:
        if pdt != torch.float32 and N not in (24, 128, 130, 2048, 3072, 8192):
            continue
        for op in ("dyt", "layernorm", "rmsnorm"):
            CASES.append((op, xdt, pdt, N))


def _name(c):
    op, xdt, pdt, N = c
    return f"{op}-{str(xdt)[6:]}-{str(pdt)[6:]}-N{N}"


@pytest.mark.parametrize("case", CASES, ids=_name)
def test_parity_small(case):
    op, xdt, pdt, N = case
    M = max(3, min(3001, (1 << 20) // N))
    reps, _ = _run(op, _inputs(M, N, xdt, pdt, _name(case)))
    for r in reps:
        print(r.line())


@pytest.mark.parametrize("variant", [1, 2], ids=["weight_first", "gemma"])
@pytest.mark.parametrize("xdt,pdt", [(torch.bfloat16, torch.float32),
                                     (torch.bfloat16, torch.bfloat16),
                                     (torch.float16, torch.float16),
                                     (torch.bfloat16, torch.float16),
                                     (torch.float32, torch.float32)],
                         ids=["bf16-f32", "bf16-bf16", "f16-f16", "bf16-f16", "f32-f32"])
@pytest.mark.parametrize("N", [8, 24, 128, 1000, 2048, 4096, 8192, 8200])
def test_rms_variants(variant, xdt, pdt, N):
    """The weight-first and Gemma RMSNorm expressions against the oracle
    (vector, multi-vector and general paths; rstd recomputation bit-exact)."""
    M = max(3, min(3001, (1 << 20) // N))
    inp = _inputs(M, N, xdt, pdt, f"rmsv{variant}{N}{xdt}{pdt}")
    reps, _ = rmsnorm_case(inp["x"], inp["dy"], inp["gamma"], 1e-6, variant=variant)
    for r in reps:
        print(r.line())


@pytest.mark.parametrize("op", ["dyt", "layernorm", "rmsnorm"])
@pytest.mark.parametrize("N", [16, 24, 64, 5, 130])
def test_persistent_loop(op, N):
    # enough rows that every resident CTA loops over several row blocks
    M = (1 << 22) // N + 7
    reps, _ = _run(op, _inputs(M, N, torch.bfloat16, torch.float32, f"loop{op}{N}"))
    for r in reps:
        print(r.line())


@pytest.mark.parametrize("op", ["dyt", "layernorm", "rmsnorm"])
@pytest.mark.parametrize("N", [64, 2048])
def test_unaligned_pointers_take_general_path(op, N):
    inp = _inputs(301, N, torch.bfloat16, torch.float32, f"unal{op}{N}")
    for k in ("x", "dy"):
        buf = torch.empty(301 * N + 1, dtype=torch.bfloat16, device="cuda")
        buf[1:].copy_(inp[k].view(-1))
        inp[k] = buf[1:].view(301, N)  # 2-byte misaligned
    _run(op, inp)


@pytest.mark.parametrize("op", ["dyt", "layernorm", "rmsnorm"])
def test_empty_input_writes_zero_grads(op):
    inp = _inputs(0, 128, torch.bfloat16, torch.float32, "empty")
    if op == "dyt":
        dx, da, dg, db = _lib.dyt_bwd(inp["x"], inp["dy"], inp["alpha"], inp["gamma"])
        grads = [da, dg, db]
        assert _lib.dyt_fwd(inp["x"], inp["alpha"], inp["gamma"], inp["beta"]).numel() == 0
    elif op == "layernorm":
        y, mean, rstd = _lib.layernorm_fwd(inp["x"], inp["gamma"], inp["beta"])
        dx, dg, db = _lib.layernorm_bwd(inp["x"], inp["dy"], mean, rstd, inp["gamma"])
        grads = [dg, db]
    else:
        y, rstd = _lib.rmsnorm_fwd(inp["x"], inp["gamma"])
        dx, dw = _lib.rmsnorm_bwd(inp["x"], inp["dy"], inp["gamma"], rstd)
        grads = [dw]
    torch.cuda.synchronize()
    assert dx.numel() == 0
    for g in grads:
        assert torch.count_nonzero(g) == 0 and not torch.isnan(g).any()


def test_dyt_alpha_inf_padded_tile():
    wl = synth.DYT_BF16_ALPHA_INF
    inp = wl.inputs(device="cuda")
    assert torch.count_nonzero(inp["x"]) == inp["x"].numel()  # no exact zeros
    reps, out = dyt_case(inp["x"], inp["dy"], inp["alpha"], inp["gamma"], inp["beta"])
    assert not torch.isnan(out["dg"]).any() and not torch.isnan(out["db"]).any()
    assert not torch.isnan(out["da"]).any() and float(out["da"]) == 0.0
    assert not torch.isnan(out["y"]).any()
    assert torch.isnan(out["dx"]).all()  # dy * gamma * inf * 0, as in the oracle
    for r in reps:
        print(r.line())


@pytest.mark.parametrize("op", ["dyt", "layernorm", "rmsnorm"])
@pytest.mark.parametrize("M,N", shapes())
def test_page_edge_shapes(op, M, N):
    if M * N > (1 << 23):
        pytest.skip("covered by the full-size workload tests")
    _run(op, _inputs(M, N, torch.bfloat16, torch.float32, f"edge{op}{M}x{N}"))


def test_rms_width_one_page_eps():
    eps = kv("rmsnorm_width_one.txt")["eps"]
    inp = _inputs(257, 1, torch.bfloat16, torch.bfloat16, "w1")
    reps, out = rmsnorm_case(inp["x"], inp["dy"], inp["gamma"], eps)
    # nonzero input derivative at width one
    assert torch.count_nonzero(out["dx"]) > 200


@pytest.mark.parametrize("op", ["dyt", "layernorm", "rmsnorm"])
@pytest.mark.parametrize("N,aligned", [(24, True), (128, True), (2048, True), (8192, True),
                                       (130, True), (127, True), (129, True), (130, False)])
def test_bit_identical_reruns(op, N, aligned):
    inp = _inputs(4099, N, torch.bfloat16, torch.float32, f"det{op}{N}")
    if not aligned:
        for k in ("x", "dy"):
            buf = torch.empty(inp[k].numel() + 1, dtype=inp[k].dtype, device="cuda")
            buf[1:].copy_(inp[k].view(-1))
            inp[k] = buf[1:].view(inp[k].shape)

    def once():
        if op == "dyt":
            y = _lib.dyt_fwd(inp["x"], inp["alpha"], inp["gamma"], inp["beta"])
            return [y, *_lib.dyt_bwd(inp["x"], inp["dy"], inp["alpha"], inp["gamma"])]
        if op == "layernorm":
            y, m, r = _lib.layernorm_fwd(inp["x"], inp["gamma"], inp["beta"])
            return [y, m, r, *_lib.layernorm_bwd(inp["x"], inp["dy"], m, r, inp["gamma"])]
        y, r = _lib.rmsnorm_fwd(inp["x"], inp["gamma"])
        return [y, r, *_lib.rmsnorm_bwd(inp["x"], inp["dy"], inp["gamma"], None)]

    a = [t.clone() for t in once()]
    for _ in range(2):
        b = once()
        for u, v in zip(a, b):
            assert u.view(torch.uint8).equal(v.view(torch.uint8)) if u.dtype != torch.float32 else \
                u.view(torch.int32).equal(v.view(torch.int32))


def test_guard_bands_untouched():
    """Outputs and workspace sit inside canary-filled buffers; every call must
    leave the canaries as they were (no out-of-bounds stores)."""
    lib = _lib.load()
    M, N = 1237, 136
    inp = _inputs(M, N, torch.bfloat16, torch.float32, "guard")
    G = 4096  # guard elements on each side
    canary = -12345.0

    def guarded(n, dtype):
        buf = torch.full((n + 2 * G,), canary, dtype=dtype, device="cuda")
        return buf, buf[G:G + n]

    stream = torch.cuda.current_stream().cuda_stream
    outs = {}
    for name, n, dt in [("y", M * N, torch.bfloat16), ("dx", M * N, torch.bfloat16),
                        ("mean", M, torch.float32), ("rstd", M, torch.float32),
                        ("dg", N, torch.float32), ("db", N, torch.float32), ("da", 1, torch.float32)]:
        outs[name] = guarded(n, dt)
    p = lambda k: outs[k][1].data_ptr()  # noqa: E731
    for op in (_lib.GBN_OP_DYT, _lib.GBN_OP_LAYERNORM, _lib.GBN_OP_RMSNORM):
        nbytes = lib.gbn_bwd_workspace_bytes(op, M, N, 1, 0, 0)
        wsb, ws = guarded(nbytes // 4, torch.float32)
        X, DY = inp["x"].data_ptr(), inp["dy"].data_ptr()
        A, Gm, B = inp["alpha"].data_ptr(), inp["gamma"].data_ptr(), inp["beta"].data_ptr()
        if op == _lib.GBN_OP_DYT:
            assert lib.dyt_fwd(X, A, Gm, B, p("y"), M, N, 1, 0, stream) == 0
            assert lib.dyt_bwd(X, DY, A, Gm, p("dx"), p("da"), p("dg"), p("db"), M, N, 1, 0,
                               ws.data_ptr(), nbytes, stream) == 0
        elif op == _lib.GBN_OP_LAYERNORM:
            assert lib.layernorm_fwd(X, Gm, B, p("y"), p("mean"), p("rstd"), M, N, 1e-5, 1, 0,
                                     stream) == 0
            assert lib.layernorm_bwd(X, DY, p("mean"), p("rstd"), Gm, p("dx"), p("dg"), p("db"), M,
                                     N, 1, 0, ws.data_ptr(), nbytes, stream) == 0
        else:
            assert lib.rmsnorm_fwd(X, Gm, p("y"), p("rstd"), M, N, 1e-6, 1, 0, stream) == 0
            assert lib.rmsnorm_bwd(X, DY, Gm, p("rstd"), p("dx"), p("dg"), M, N, 1e-6, 1, 0,
                                   ws.data_ptr(), nbytes, stream) == 0
        torch.cuda.synchronize()
        for name, (buf, _) in list(outs.items()) + [("ws", (wsb, ws))]:
            n = buf.numel() - 2 * G
            assert torch.all(buf[:G] == canary), f"op {op}: store before {name}"
            assert torch.all(buf[G + n:] == canary), f"op {op}: store after {name}"


def test_workspace_too_small_is_rejected():
    lib = _lib.load()
    M, N = 5000, 64
    inp = _inputs(M, N, torch.bfloat16, torch.float32, "wsz")
    need = lib.gbn_bwd_workspace_bytes(_lib.GBN_OP_RMSNORM, M, N, 1, 0, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dx = torch.empty_like(inp["x"])
    dw = torch.empty(N, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = lib.rmsnorm_bwd(inp["x"].data_ptr(), inp["dy"].data_ptr(), inp["gamma"].data_ptr(), None,
                         dx.data_ptr(), dw.data_ptr(), M, N, 1e-6, 1, 0, ws.data_ptr(), 64, s)
    assert rc == 3  # GBN_EWORKSPACE, nothing launched
    rc = lib.rmsnorm_bwd(inp["x"].data_ptr(), inp["dy"].data_ptr(), inp["gamma"].data_ptr(), None,
                         dx.data_ptr(), dw.data_ptr(), M, N, 1e-6, 1, 0, ws.data_ptr(), need, s)
    assert rc == 0
    torch.cuda.synchronize()


def test_layernorm_without_affine():
    inp = _inputs(777, 96, torch.bfloat16, torch.float32, "noaff")
    layernorm_case(inp["x"], inp["dy"], None, None, 1e-5)
    layernorm_case(inp["x"], inp["dy"], inp["gamma"], None, 1e-5)


def test_tanh_against_cuda_tanhf():
    """The kernels' float32 tanh (exp2 identity plus a Maclaurin branch) against
    torch's CUDA tanh over a dense sweep, through dyt_fwd with gamma = 1,
    beta = 0, alpha = 1."""
    z = torch.cat([torch.linspace(-12, 12, 1 << 20), torch.logspace(-8, 1, 4096),
                   -torch.logspace(-8, 1, 4096), torch.tensor([0.0, 0.125, -0.125, 1e-30])])
    z = z.to("cuda", torch.float32).view(-1, 4)[: (z.numel() // 4)]
    one = torch.ones(1, device="cuda")
    t = _lib.dyt_fwd(z, one, torch.ones(4, device="cuda"), torch.zeros(4, device="cuda"))
    ref = torch.tanh(z.double())
    err = ((t.double() - ref).abs() / ref.abs().clamp_min(1e-38)).max().item()
    cuda_err = ((torch.tanh(z).double() - ref).abs() / ref.abs().clamp_min(1e-38)).max().item()
    print(f"max rel err: kernels {err:.3e}, CUDA tanhf {cuda_err:.3e}")
    assert err < 2.0 ** -19  # within 16 float32 ulps everywhere


@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float32])
def test_dyt_large_arguments(xdt):
    """|alpha x| beyond 43.6: tanh is +-1 and sech^2 flushes to 0, so y is
    exactly +-gamma + beta (one rounding) and dx, and every dalpha term, is
    exactly zero (the true sech^2 is below 2^-124)."""
    M, N = 300, 64
    mag = torch.tensor([43.7, 50.0, 88.0, 100.0, 1e4, 3e38])
    x = mag[torch.arange(M * N) % mag.numel()].view(M, N)
    x = torch.where(torch.arange(M * N).view(M, N) % 3 == 0, -x, x).to("cuda", xdt)
    alpha = torch.ones(1, device="cuda")
    gamma = synth.normal((N,), 1.0, 0.1, torch.float32, seed=5, device="cuda")
    beta = synth.normal((N,), 0.0, 0.1, torch.float32, seed=6, device="cuda")
    dy = synth.normal((M, N), 0.0, 1.0, xdt, seed=7, device="cuda")
    y = _lib.dyt_fwd(x, alpha, gamma, beta)
    dx, da, dg, db = _lib.dyt_bwd(x, dy, alpha, gamma)
    sgn = torch.sign(x.float())
    assert torch.equal(y, (sgn * gamma + beta).to(xdt))
    assert torch.equal(dx.float().abs(), torch.zeros_like(dx.float()))
    assert da.item() == 0.0
    torch.testing.assert_close(db, dy.float().sum(0), rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(dg, (dy.float() * sgn).sum(0), rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("op", ["dyt", "layernorm", "rmsnorm"])
@pytest.mark.parametrize("dts", [(torch.bfloat16, torch.float32), (torch.float32, torch.float32),
                                 (torch.float16, torch.float16)], ids=["bf16", "f32", "f16"])
@pytest.mark.parametrize("N", [128, 1000])
def test_degenerate_rows(op, dts, N):
    """Rows the method treats specially, mixed into random ones: constant
    rows (LayerNorm: zero variance, so y = beta), all-zero rows (RMSNorm:
    rstd = 1/sqrt(eps), y = 0; DyT: y = beta), against the oracle; and exact
    results where they are exact (a constant 1.5 sums exactly at N = 128)."""
    xdt, pdt = dts
    M = 301
    inp = _inputs(M, N, xdt, pdt, f"degenerate/{op}/{N}/{xdt}/{pdt}")
    x = inp["x"]
    const = torch.arange(M, device="cuda") % 3 == 0
    fill = 1.5 if op == "layernorm" else 0.0
    x[const] = fill
    inp["x"] = x
    reps, out = _run(op, inp)
    for r in reps:
        print(r.line())
    beta, gamma = inp["beta"], inp["gamma"]
    if op == "layernorm" and N == 128:
        assert torch.equal(out["y"][const], beta.to(xdt).expand(int(const.sum()), N))
    if op == "dyt":
        assert torch.equal(out["y"][const], beta.to(xdt).expand(int(const.sum()), N))
    if op == "rmsnorm":
        assert torch.all(out["y"][const] == 0)


def test_autograd_wrappers_match_direct_calls():
    inp = _inputs(513, 256, torch.bfloat16, torch.float32, "ag")
    for fn, params, direct in [
        (lambda x, a, g, b: dyt(x, a, g, b), ("alpha", "gamma", "beta"), "dyt"),
        (lambda x, g, b: layer_norm(x, g, b, 1e-5), ("gamma", "beta"), "ln"),
        (lambda x, g: rms_norm(x, g, 1e-6), ("gamma",), "rms"),
    ]:
        x = inp["x"].clone().view(9, 57, 256).requires_grad_(True)
        ps = [inp[k].clone().requires_grad_(True) for k in params]
        y = fn(x, *ps)
        y.backward(inp["dy"].view(9, 57, 256))
        if direct == "dyt":
            dx, da, dg, db = _lib.dyt_bwd(inp["x"], inp["dy"], inp["alpha"], inp["gamma"])
            want = [dx, da, dg, db]
        elif direct == "ln":
            _, m, r = _lib.layernorm_fwd(inp["x"], inp["gamma"], inp["beta"], 1e-5)
            want = list(_lib.layernorm_bwd(inp["x"], inp["dy"], m, r, inp["gamma"]))
        else:
            _, r = _lib.rmsnorm_fwd(inp["x"], inp["gamma"], 1e-6)
            want = list(_lib.rmsnorm_bwd(inp["x"], inp["dy"], inp["gamma"], r, 1e-6))
        got = [x.grad.view(513, 256)] + [p.grad for p in ps]
        for g, w in zip(got, want):
            assert torch.equal(g, w)


def test_bounded_wait_self_test_sets_fault_and_returns():
    """A barrier that never completes: the kernel's bounded wait must run
    out (a few milliseconds here), set the fault bit and return, leaving the
    context usable."""
    lib = _lib.load()
    _lib.read_faults(clear=True)
    res = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.gbn_selftest_wait_timeout(1 << 24, res.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(res.item()) == 0
    assert _lib.read_faults(clear=True) & 1
    assert _lib.read_faults(clear=False) == 0
    # the context still works
    inp = _inputs(333, 128, torch.bfloat16, torch.float32, "after_selftest")
    _run("rmsnorm", inp)


def test_fault_word_clean_after_kernels():
    _lib.read_faults(clear=True)
    inp = _inputs(20011, 64, torch.bfloat16, torch.float32, "faultclean")
    for op in ("dyt", "layernorm", "rmsnorm"):
        _run(op, inp)
    assert _lib.read_faults(clear=False) == 0
