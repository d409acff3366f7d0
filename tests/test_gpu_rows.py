"""GPU: inputs read in place through row layouts (gbn_rows).

DeepSpeed PR 8645 ("Where the kernels run", row "Layout") copies a
non-contiguous input before its kernels run; its tests feed a head-major
input and the head-major upstream gradient that attention produces
("Correctness evidence", 1).  Here such inputs are read where they lie:

* layouts whose rows start on 16-byte boundaries take the same vector
  kernels and launch layout as a contiguous copy of the same rows, so every
  output must be bit-identical to the call on the contiguous copy;
* parameter gradients too, except for layouts that permute the storage's
  contiguous rows (head-major, sequence-major): those are read in storage
  order, so their parameter gradients must be bit-identical to the call on
  the storage read as contiguous rows;
* other layouts (odd strides, odd base offsets) take the general kernels and
  are compared with the float64 oracle element by element.
All calls go through the C ABI (the ctypes binding)."""
import pytest
import torch

from _cases import dyt_case, layernorm_case, rmsnorm_case
from normalization_layers_fwd_gb300 import _lib, synth
from normalization_layers_fwd_gb300.functional import rms_norm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from normalization_layers_fwd_gb300 import build
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def _normal(shape, dt, seed, mean=0.0, std=1.0):
    return synth.normal(shape, mean, std, dt, seed=synth.seed_for(91, seed), device="cuda")


def _params(N, pdt, seed):
    return dict(alpha=_normal((1,), pdt, seed + "/a", 0.8, 0.1),
                gamma=_normal((N,), pdt, seed + "/g", 1.0, 0.1),
                beta=_normal((N,), pdt, seed + "/b", 0.0, 0.1))


# ------------------------------------------------------------------ layouts
# Each maker returns a view of logical shape [..., N] over fresh storage.

def head_major(lead, N, dt, seed):
    """[B, H, S, D] storage seen as [B, S, H, D] (lead = (B, S, H))."""
    B, S, H = lead
    return _normal((B, H, S, N), dt, seed).transpose(1, 2)


def seq_major(lead, N, dt, seed):
    """[S, B, H, D] storage seen as [B, S, H, D]."""
    B, S, H = lead
    return _normal((S, B, H, N), dt, seed).transpose(0, 1)


def row_padded(lead, N, dt, seed, pad_bytes=16, offset=0):
    """Rows of N inside rows of N + pad elements, starting at column offset."""
    (M,) = lead
    e = torch.empty((), dtype=dt).element_size()
    pad = pad_bytes // e
    return _normal((M, N + pad), dt, seed)[:, offset:offset + N]


def broadcast(lead, N, dt, seed):
    """One row repeated M times (row stride 0)."""
    (M,) = lead
    return _normal((1, N), dt, seed).expand(M, N)


def _layout_is_vector(v):
    """Whether the library will take the vector path for view v (16-byte
    aligned base and row strides), given N * elem a multiple of 16."""
    e = v.element_size()
    lay = _lib.fold_rows(tuple(v.shape), tuple(v.stride()))
    return (v.data_ptr() % 16 == 0 and lay is not None and
            all((s * e) % 16 == 0 for s in (lay.s1, lay.s2, lay.s3)))


def storage_rows(v):
    """The contiguous rows v's storage holds, when v is a permutation of
    them (a transposed view of a fresh contiguous tensor), else None."""
    base = v._base if v._base is not None else None
    if base is None or not base.is_contiguous() or base.numel() != v.numel():
        return None
    if v.storage_offset() != base.storage_offset():
        return None
    return base.reshape(-1, v.shape[-1])


# ---------------------------------------------------------------- the ops

def _bits(t):
    t = t.contiguous()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def run(op, x, dy, P, eps=1e-5):
    if op == "dyt":
        y = _lib.dyt_fwd(x, P["alpha"], P["gamma"], P["beta"])
        dx, da, dg, db = _lib.dyt_bwd(x, dy, P["alpha"], P["gamma"])
        return dict(y=y, dx=dx, da=da, dg=dg, db=db)
    if op == "layernorm":
        y, mean, rstd = _lib.layernorm_fwd(x, P["gamma"], P["beta"], eps)
        dx, dg, db = _lib.layernorm_bwd(x, dy, mean, rstd, P["gamma"])
        return dict(y=y, mean=mean, rstd=rstd, dx=dx, dg=dg, db=db)
    y, rstd = _lib.rmsnorm_fwd(x, P["gamma"], eps)
    dx, dw = _lib.rmsnorm_bwd(x, dy, P["gamma"], rstd, eps)
    dx2, dw2 = _lib.rmsnorm_bwd(x, dy, P["gamma"], None, eps)
    return dict(y=y, rstd=rstd, dx=dx, dw=dw, dx2=dx2, dw2=dw2)


PARAM_GRADS = {"da", "dg", "db", "dw", "dw2"}


def assert_same_bits(a, b, keys=None):
    assert a.keys() == b.keys()
    for k in a:
        if keys is not None and k not in keys:
            continue
        assert a[k].shape == b[k].shape, k
        assert a[k].is_contiguous(), k
        assert torch.equal(_bits(a[k]), _bits(b[k])), k


def check_layout(op, x, dy, P):
    """Per-row outputs against a contiguous copy; parameter gradients against
    the contiguous copy, or for storage permutations against the storage."""
    got = run(op, x, dy, P)
    want = run(op, x.contiguous(), dy.contiguous(), P)
    xs, dys = storage_rows(x), storage_rows(dy)
    perm = xs is not None and dys is not None and x.stride() == dy.stride()
    assert_same_bits(got, want, None if not perm else set(got) - PARAM_GRADS)
    if perm:
        assert_same_bits(got, run(op, xs, dys, P), set(got) & PARAM_GRADS)
    return perm


OPS = ["dyt", "layernorm", "rmsnorm"]
DT = [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
      (torch.float16, torch.float32)]
DT_ID = ["bf16", "f32", "f16"]


# ------------------------------------------------ vector layouts: bit-exact

VECTOR_CASES = [
    ("head_major", head_major, (2, 67, 8), 64),
    ("head_major", head_major, (2, 33, 32), 128),
    ("head_major", head_major, (1, 19, 4), 256),
    ("seq_major", seq_major, (3, 21, 8), 128),
    ("row_padded", row_padded, (1001,), 1024),
    ("row_padded", row_padded, (601,), 4096),
    ("row_padded", row_padded, (257,), 8192),
    ("broadcast", broadcast, (517,), 128),
]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dts", DT, ids=DT_ID)
@pytest.mark.parametrize("case", VECTOR_CASES, ids=lambda c: f"{c[0]}-N{c[3]}")
def test_vector_layouts_match_contiguous_bits(op, dts, case):
    name, make, lead, N = case
    xdt, pdt = dts
    seed = f"{op}/{name}/{N}/{xdt}"
    x = make(lead, N, xdt, seed + "/x")
    dy = make(lead, N, xdt, seed + "/dy")
    assert not x.is_contiguous() and _layout_is_vector(x)
    perm = check_layout(op, x, dy, _params(N, pdt, seed))
    assert perm == (name in ("head_major", "seq_major"))
    assert _lib.read_faults() == 0


@pytest.mark.parametrize("op", OPS)
def test_mixed_layouts_x_and_dy(op):
    """x head-major and dy contiguous, and the other way round."""
    lead, N = (2, 45, 16), 128
    for xs, dys in ((True, False), (False, True)):
        x = head_major(lead, N, torch.bfloat16, f"mix/{op}/x")
        dy = head_major(lead, N, torch.bfloat16, f"mix/{op}/dy")
        x = x if xs else x.contiguous()
        dy = dy if dys else dy.contiguous()
        P = _params(N, torch.float32, f"mix/{op}")
        assert not check_layout(op, x, dy, P)  # one map for x and dy: not both permuted


def test_persistent_loop_head_major():
    """Enough rows that every CTA walks many row blocks through the ring."""
    lead, N = (4, 520, 32), 128
    for op in OPS:
        x = head_major(lead, N, torch.bfloat16, f"pl/{op}/x")
        dy = head_major(lead, N, torch.bfloat16, f"pl/{op}/dy")
        P = _params(N, torch.bfloat16, f"pl/{op}")
        assert check_layout(op, x, dy, P)


def test_autograd_head_major_rms_norm():
    lead, N = (2, 40, 16), 128
    xv = head_major(lead, N, torch.bfloat16, "ag/x").requires_grad_(True)
    w = _normal((N,), torch.bfloat16, "ag/w", 1.0, 0.1).requires_grad_(True)
    dy = head_major(lead, N, torch.bfloat16, "ag/dy")
    y = rms_norm(xv, w, 1e-6)
    y.backward(dy)
    xc = xv.detach().contiguous().requires_grad_(True)
    wc = w.detach().clone().requires_grad_(True)
    yc = rms_norm(xc, wc, 1e-6)
    yc.backward(dy.contiguous())
    assert torch.equal(_bits(y), _bits(yc))
    assert torch.equal(_bits(xv.grad), _bits(xc.grad))
    # the weight gradient sums the rows in storage order
    ws = w.detach().clone().requires_grad_(True)
    rms_norm(storage_rows(xv).detach(), ws, 1e-6).backward(storage_rows(dy))
    assert torch.equal(_bits(w.grad), _bits(ws.grad))


# ------------------------------------------- general layouts: oracle parity

GENERAL_CASES = [
    ("odd_row_stride", lambda lead, N, dt, s: row_padded(lead, N, dt, s, pad_bytes=4), (999,),
     128),
    ("odd_base", lambda lead, N, dt, s: row_padded(lead, N, dt, s, offset=1), (777,), 256),
    ("odd_stride_wide", lambda lead, N, dt, s: row_padded(lead, N, dt, s, pad_bytes=4), (301,),
     4096),
    ("head_major_odd_width", head_major, (2, 29, 8), 100),
]


def _case(op, x, dy, P, eps=1e-5):
    if op == "dyt":
        return dyt_case(x, dy, P["alpha"], P["gamma"], P["beta"])
    if op == "layernorm":
        return layernorm_case(x, dy, P["gamma"], P["beta"], eps)
    return rmsnorm_case(x, dy, P["gamma"], eps)


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dts", DT, ids=DT_ID)
@pytest.mark.parametrize("case", GENERAL_CASES, ids=lambda c: c[0])
def test_general_layouts_against_oracle(op, dts, case):
    name, make, lead, N = case
    xdt, pdt = dts
    seed = f"gen/{op}/{name}/{xdt}"
    x = make(lead, N, xdt, seed + "/x")
    dy = make(lead, N, xdt, seed + "/dy")
    assert not x.is_contiguous()
    if name != "head_major_odd_width":  # (in f32 its rows are 400 bytes: vector path)
        assert not _layout_is_vector(x)
    reps, _ = _case(op, x, dy, _params(N, pdt, seed))
    for r in reps:
        print(r.line())
    assert _lib.read_faults() == 0


@pytest.mark.parametrize("op", OPS)
def test_head_major_against_oracle(op):
    """The vector-path head-major case, checked against the oracle too."""
    x = head_major((2, 37, 8), 128, torch.bfloat16, f"hmo/{op}/x")
    dy = head_major((2, 37, 8), 128, torch.bfloat16, f"hmo/{op}/dy")
    reps, _ = _case(op, x, dy, _params(128, torch.float32, f"hmo/{op}"))
    for r in reps:
        print(r.line())


def test_more_than_three_levels_is_copied():
    """A layout the C ABI cannot express is copied by the binding: same bits."""
    base = _normal((2, 3, 2, 5, 64), torch.bfloat16, "l4/x")
    x = base.permute(0, 2, 1, 3, 4)
    assert _lib.fold_rows(tuple(x.shape), tuple(x.stride())) is None
    P = _params(64, torch.float32, "l4")
    dy = _normal(tuple(x.shape), torch.bfloat16, "l4/dy")
    assert_same_bits(run("rmsnorm", x, dy, P), run("rmsnorm", x.contiguous(), dy, P))


@pytest.mark.parametrize("op", OPS)
def test_storage_order_ragged_blocks(op):
    """Storage permutations whose row count leaves a ragged last row block,
    with every level size odd (the output map's divisions by 3, 5, 7)."""
    x = head_major((3, 7, 5), 128, torch.bfloat16, f"rag/{op}/x")
    dy = head_major((3, 7, 5), 128, torch.bfloat16, f"rag/{op}/dy")
    assert check_layout(op, x, dy, _params(128, torch.float32, f"rag/{op}"))
    x = seq_major((5, 331, 3), 64, torch.float16, f"rag2/{op}/x")
    dy = seq_major((5, 331, 3), 64, torch.float16, f"rag2/{op}/dy")
    assert check_layout(op, x, dy, _params(64, torch.float32, f"rag2/{op}"))


@pytest.mark.parametrize("variant", [1, 2], ids=["weight_first", "gemma"])
@pytest.mark.parametrize("xdt,wdt", [(torch.bfloat16, torch.bfloat16), (torch.float16, torch.float32),
                                     (torch.float32, torch.float32)], ids=["bf16", "f16", "f32"])
def test_rms_variants_head_major(variant, xdt, wdt):
    """The RMSNorm expression variants on head-major input: per-row outputs
    equal the contiguous call's; the weight gradient equals the call on the
    storage."""
    lead, N = (2, 37, 8), 128
    x = head_major(lead, N, xdt, f"var{variant}/{xdt}/x")
    dy = head_major(lead, N, xdt, f"var{variant}/{xdt}/dy")
    w = _normal((N,), wdt, f"var{variant}/{xdt}/w", 1.0, 0.1)

    def call(a, b):
        y, rstd = _lib.rmsnorm_fwd(a, w, 1e-6, variant=variant)
        dx, dw = _lib.rmsnorm_bwd(a, b, w, rstd, 1e-6, variant=variant)
        return dict(y=y, rstd=rstd, dx=dx, dw=dw)
    got = call(x, dy)
    assert_same_bits(got, call(x.contiguous(), dy.contiguous()), {"y", "rstd", "dx"})
    assert_same_bits(got, call(storage_rows(x), storage_rows(dy)), {"dw"})


@pytest.mark.parametrize("make", [head_major, row_padded], ids=["head_major", "row_padded"])
def test_layernorm_without_affine_strided(make):
    """LayerNorm with neither gamma nor beta on strided input."""
    lead = (2, 41, 8) if make is head_major else (513,)
    N = 256
    x = make(lead, N, torch.bfloat16, f"noaff/{make.__name__}/x")
    dy = make(lead, N, torch.bfloat16, f"noaff/{make.__name__}/dy")

    def call(a, b):
        y, mean, rstd = _lib.layernorm_fwd(a, None, None, 1e-5)
        dx, dg, db = _lib.layernorm_bwd(a, b, mean, rstd, None)
        return dict(y=y, mean=mean, rstd=rstd, dx=dx, dg=dg, db=db)
    got = call(x, dy)
    perm = storage_rows(x) is not None
    assert_same_bits(got, call(x.contiguous(), dy.contiguous()),
                     {"y", "mean", "rstd", "dx"} | (set() if perm else {"dg", "db"}))
    if perm:
        assert_same_bits(got, call(storage_rows(x), storage_rows(dy)), {"dg", "db"})


def test_dyt_bf16_params_head_major():
    """DyT with bf16 parameters on head-major bf16 input, alpha large enough
    that tanh saturates in part of the tensor."""
    lead, N = (2, 53, 4), 64
    x = head_major(lead, N, torch.bfloat16, "dytp/x")
    dy = head_major(lead, N, torch.bfloat16, "dytp/dy")
    P = {k: v.to(torch.bfloat16) for k, v in _params(N, torch.float32, "dytp").items()}
    P["alpha"] = torch.full((1,), 7.0, dtype=torch.bfloat16, device="cuda")
    got = run("dyt", x, dy, P)
    assert_same_bits(got, run("dyt", x.contiguous(), dy.contiguous(), P), {"y", "dx"})
    assert_same_bits(got, run("dyt", storage_rows(x), storage_rows(dy), P), {"da", "dg", "db"})

