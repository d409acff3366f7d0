"""rmsnorm_bwd_static_ws, the RMSNorm backward whose scratch is the library's
static device array, against rmsnorm_bwd with a caller workspace.  Both go
through the C ABI.  Each case makes two calls in a row of the static-scratch
entry point (the second finds the first one's partial sums still in the
array) and checks both against rmsnorm_bwd within the parity tolerance, and
bit for bit, since both run the same kernels with the same launch layout.

The file name sorts last so that pytest collects it after every other test;
it also passes alone in a fresh process (its fixture builds and loads the
library itself)."""
import numpy as np
import pytest
import torch

from _parity import check_out, f64
from normalization_layers_fwd_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from normalization_layers_fwd_gb300 import build
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def _inputs(M, N, xdt, wdt, tag):
    s = lambda n: synth.seed_for(95, f"{tag}/{n}")  # noqa: E731
    return (synth.normal((M, N), 0.0, 1.0, xdt, seed=s("x"), device="cuda"),
            synth.normal((M, N), 0.0, 1.0, xdt, seed=s("dy"), device="cuda"),
            synth.normal((N,), 1.0, 0.1, wdt, seed=s("w"), device="cuda"))


def _same(name, got, ref):
    """got within the parity tolerance of ref (1 bf16 ULP, or 1e-5 relative in
    fp32, NaN positions equal), and bit-identical to it."""
    check_out(name, got, f64(ref), np.abs(f64(ref)))
    assert torch.equal(got.view(torch.int16 if got.dtype == torch.bfloat16 else torch.int32),
                       ref.view(torch.int16 if ref.dtype == torch.bfloat16 else torch.int32)), name


CASES = [
    # (M, N, x dtype, w dtype, give rstd): vector paths and the general path
    (3000, 4096, torch.bfloat16, torch.bfloat16, True),
    (1027, 24, torch.bfloat16, torch.float32, False),
    (5000, 8192, torch.bfloat16, torch.bfloat16, True),
    (4099, 1000, torch.float32, torch.float32, True),
    (700, 1001, torch.float32, torch.float32, False),
    (0, 512, torch.bfloat16, torch.bfloat16, True),
]


@pytest.mark.parametrize("M,N,xdt,wdt,with_rstd", CASES)
def test_static_scratch_matches_caller_workspace(M, N, xdt, wdt, with_rstd):
    x, dy, w = _inputs(M, N, xdt, wdt, f"{M}x{N}/{xdt}/{wdt}")
    eps = 1e-6
    rstd = None
    if with_rstd:
        _, rstd = _lib.rmsnorm_fwd(x, w, eps)
    dx_ref, dw_ref = _lib.rmsnorm_bwd(x, dy, w, rstd, eps)
    for call in (1, 2):
        dx, dw = _lib.rmsnorm_bwd_static_ws(x, dy, w, rstd, eps)
        torch.cuda.synchronize()
        _same(f"dx call {call}", dx, dx_ref)
        _same(f"dw call {call}", dw, dw_ref)
    if M == 0:
        assert torch.all(dw_ref == 0)


def test_static_scratch_interleaved_shapes():
    """Two calls in a row on different shapes: the wider one leaves partial
    sums in the array that the narrower one must not read."""
    a = _inputs(2000, 2048, torch.bfloat16, torch.bfloat16, "wide")
    b = _inputs(333, 128, torch.bfloat16, torch.bfloat16, "narrow")
    ref = [_lib.rmsnorm_bwd(x, dy, w, None, 1e-5) for x, dy, w in (a, b)]
    for _ in range(2):
        for (x, dy, w), (dx_ref, dw_ref) in zip((a, b), ref):
            dx, dw = _lib.rmsnorm_bwd_static_ws(x, dy, w, None, 1e-5)
            torch.cuda.synchronize()
            _same("dx", dx, dx_ref)
            _same("dw", dw, dw_ref)


def test_oversize_call_is_rejected_before_launch():
    """A general-path shape (odd N) whose partial sums exceed the array:
    GBN_ESCRATCH, and dx is left as it was (nothing was launched)."""
    M, N = 4096, 8191
    x, dy, w = _inputs(M, N, torch.bfloat16, torch.bfloat16, "oversize")
    need = _lib.load().gbn_bwd_workspace_bytes(_lib.GBN_OP_RMSNORM, M, N, _lib.GBN_BF16,
                                               _lib.GBN_BF16, 0)
    assert need > _lib.GBN_STATIC_WS_BYTES
    dx = torch.full_like(x, 7.0)
    dw = torch.full((N,), 7.0, dtype=torch.bfloat16, device="cuda")
    P = lambda t: t.data_ptr()  # noqa: E731
    rc = _lib.load().rmsnorm_bwd_static_ws(P(x), P(dy), P(w), None, P(dx), P(dw), M, N, 1e-6,
                                           _lib.GBN_BF16, _lib.GBN_BF16,
                                           torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.GBN_ESCRATCH
    assert b"GBN_ESCRATCH" in _lib.load().gbn_status_string(rc)
    torch.cuda.synchronize()
    assert torch.all(dx == 7.0) and torch.all(dw == 7.0)
    with pytest.raises(_lib.GbnError):
        _lib.rmsnorm_bwd_static_ws(x, dy, w)
    # without dw the array is not needed, so the same shape is accepted
    dx2, none = _lib.rmsnorm_bwd_static_ws(x, dy, w, need_dw=False)
    dx_ref, _ = _lib.rmsnorm_bwd(x, dy, w, need_dw=False)
    assert none is None
    _same("dx without dw", dx2, dx_ref)


def test_documented_limits_hold_on_this_device():
    """The header's limits, as functions of this device's SM count S: the
    vector path needs at most 32 KiB x S of partial sums (so a workspace of
    exactly that size is accepted), and the general path at most 8 MiB up to
    N = 2^19 / S' (S' = S rounded up to even), 16 x S' x N bytes beyond; the
    static array serves the first two and rejects the third."""
    lib = _lib.load()
    S = torch.cuda.get_device_properties(0).multi_processor_count
    Sp = S + (S & 1)
    stream = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731
    # vector path: the widths of each schedule family, M large enough that
    # every launch uses its full persistent grid
    for xdt, code, widths in ((torch.bfloat16, _lib.GBN_BF16, (2048, 4096, 8192)),
                              (torch.float32, _lib.GBN_F32, (1024, 2048, 4096, 8192))):
        for N in widths:
            M = 8 * S
            x, dy, w = _inputs(M, N, xdt, xdt, f"limit/{N}/{xdt}")
            dx = torch.empty_like(x)
            dw = torch.empty_like(w)
            ws = torch.empty(32768 * S, dtype=torch.uint8, device="cuda")
            rc = lib.rmsnorm_bwd(P(x), P(dy), P(w), None, P(dx), P(dw), M, N, 1e-6, code, code,
                                 P(ws), 32768 * S, stream)
            assert rc == _lib.GBN_OK, (N, xdt, rc)
            dx2, dw2 = _lib.rmsnorm_bwd_static_ws(x, dy, w)
            torch.cuda.synchronize()
            _same(f"dx N={N}", dx2, dx)
            _same(f"dw N={N}", dw2, dw)
    # the widest 16-bit vector rows: one partial row of N floats per SM
    for N in (12288, 16384):
        M = 2 * S
        x, dy, w = _inputs(M, N, torch.bfloat16, torch.bfloat16, f"limit/wide/{N}")
        dx = torch.empty_like(x)
        dw = torch.empty_like(w)
        ws = torch.empty(4 * N * S, dtype=torch.uint8, device="cuda")
        rc = lib.rmsnorm_bwd(P(x), P(dy), P(w), None, P(dx), P(dw), M, N, 1e-6, _lib.GBN_BF16,
                             _lib.GBN_BF16, P(ws), 4 * N * S, stream)
        assert rc == _lib.GBN_OK, (N, rc)
        if 4 * N * S <= _lib.GBN_STATIC_WS_BYTES:
            dx_ref, dw_ref = _lib.rmsnorm_bwd(x, dy, w)
            dx2, dw2 = _lib.rmsnorm_bwd_static_ws(x, dy, w)
            torch.cuda.synchronize()
            _same(f"dx N={N}", dx2, dx_ref)
            _same(f"dw N={N}", dw2, dw_ref)
        else:
            with pytest.raises(_lib.GbnError):
                _lib.rmsnorm_bwd_static_ws(x, dy, w)
    # general path (N not a multiple of 8: 16-bit rows are not 16-byte multiples)
    n_fit = (1 << 19) // Sp
    n_fit -= 1 if n_fit % 8 == 0 else 0
    n_over = n_fit + 1 if (n_fit + 1) % 8 else n_fit + 2
    M = 64 * S
    fit = lib.gbn_bwd_workspace_bytes(_lib.GBN_OP_RMSNORM, M, n_fit, _lib.GBN_BF16,
                                      _lib.GBN_BF16, 0)
    over = lib.gbn_bwd_workspace_bytes(_lib.GBN_OP_RMSNORM, M, n_over, _lib.GBN_BF16,
                                       _lib.GBN_BF16, 0)
    assert fit <= _lib.GBN_STATIC_WS_BYTES
    assert over == (16 * Sp * n_over + 255) // 256 * 256 > _lib.GBN_STATIC_WS_BYTES
    x, dy, w = _inputs(M, n_fit, torch.bfloat16, torch.bfloat16, "limit/general")
    dx_ref, dw_ref = _lib.rmsnorm_bwd(x, dy, w)
    dx, dw = _lib.rmsnorm_bwd_static_ws(x, dy, w)
    torch.cuda.synchronize()
    _same("dx general", dx, dx_ref)
    _same("dw general", dw, dw_ref)
    x, dy, w = _inputs(M, n_over, torch.bfloat16, torch.bfloat16, "limit/over")
    with pytest.raises(_lib.GbnError):
        _lib.rmsnorm_bwd_static_ws(x, dy, w)
