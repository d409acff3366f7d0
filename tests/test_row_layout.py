"""Row layouts (gbn_rows) without a GPU: the binding's folding of a strided
tensor into at most three row levels puts every row where torch's strides
put it, and the library validates layouts before touching a device.

A head-major [B, H, S, D] activation seen as [B, S, H, D] (the layout that
attention hands to a per-head norm, DeepSpeed PR 8645, "Correctness
evidence", 1) is the main case."""
import ctypes

import pytest
import torch

from normalization_layers_fwd_gb300 import _lib

GBN_OK, GBN_EINVAL, GBN_EDTYPE, GBN_EWORKSPACE, GBN_ELAUNCH, GBN_EDEVICE = range(6)


def row_starts(v):
    """Element offset of each row of view v in its storage, by torch's own
    indexing: v is a view of arange(storage), so v[..., 0] holds them."""
    return v[..., 0].reshape(-1).tolist()


def layout_starts(lay, M):
    n1, s1, n2, s2, s3 = lay.n1, lay.s1, lay.n2, lay.s2, lay.s3
    return [(r % n1) * s1 + ((r // n1) % n2) * s2 + (r // (n1 * n2)) * s3 for r in range(M)]


def views():
    base = torch.arange(1 << 16, dtype=torch.int64)
    B, H, S, D = 2, 3, 5, 8
    hm = base[: B * H * S * D].view(B, H, S, D)
    yield "head-major as [B,S,H,D]", hm.transpose(1, 2)
    yield "head-major as [S,B,H,D]", hm.permute(2, 0, 1, 3)
    yield "row-strided slice", base[: 40 * 24].view(40, 24)[:, :8]
    yield "column window", base[: 40 * 24].view(40, 24)[:, 8:16]
    yield "every other row", base[: 40 * 24].view(40, 24)[::2]
    yield "3-D slice", base[: 4 * 6 * 32].view(4, 6, 32)[:, 1:5, :16]
    yield "broadcast rows", base[:16].view(1, 16).expand(7, 16)
    yield "broadcast middle", base[: 3 * 16].view(3, 1, 16).expand(3, 4, 16)
    yield "size-1 levels", base[: 5 * 32].view(1, 5, 1, 32)[:, :, :, :16]
    yield "nested levels merge", base[: 2 * 3 * 4 * 16].view(2, 3, 4, 16)[:, :, :, :8]
    yield "four levels", base[: 2 * 3 * 2 * 5 * 8].view(2, 3, 2, 5, 8).permute(0, 2, 1, 3, 4)


@pytest.mark.parametrize("name,v", list(views()), ids=[n for n, _ in views()])
def test_fold_rows_matches_torch_strides(name, v):
    lay = _lib.fold_rows(tuple(v.shape), tuple(v.stride()))
    M = v.numel() // v.shape[-1]
    if lay is None:
        assert name == "four levels"  # more than three levels: the binding copies
        return
    assert lay.n1 >= 1 and lay.n2 >= 1
    off = v.storage_offset()
    assert [s + off for s in layout_starts(lay, M)] == row_starts(v)
    # and each row's elements are contiguous
    assert v.stride(-1) == 1 or v.shape[-1] == 1


def test_fold_rows_rejects_a_strided_last_dimension():
    v = torch.arange(64).view(8, 8).t()
    assert _lib.fold_rows(tuple(v.shape), tuple(v.stride())) is None


def test_head_major_layout_values():
    B, H, S, D = 2, 32, 7, 128
    v = torch.empty(B, H, S, D).transpose(1, 2)  # [B, S, H, D]
    lay = _lib.fold_rows(tuple(v.shape), tuple(v.stride()))
    assert (lay.n1, lay.s1, lay.n2, lay.s2, lay.s3) == (H, S * D, S, D, H * S * D)


@pytest.fixture(scope="module")
def lib():
    from normalization_layers_fwd_gb300 import build
    build.build()
    return _lib.load()


def test_rows_entry_points_validate_layouts(lib):
    p = ctypes.c_void_p(16)
    R = _lib.gbn_rows
    bad = [R(0, 8, 1, 0, 0), R(2, 8, 0, 0, 0), R(2, -8, 1, 0, 0), R(2, 8, 2, -1, 0),
           R(2, 8, 2, 16, -32),
           # row starts beyond 2^62 bytes (or overflowing int64) are rejected
           R(2, 1 << 61, 1, 0, 0), R(2, 8, 2, 16, (1 << 63) - 1), R(8, 1 << 60, 1, 0, 0)]
    for lay in bad:
        ref = ctypes.byref(lay)
        assert lib.dyt_fwd_rows(p, ref, p, p, p, p, 8, 8, 1, 0, None) == GBN_EINVAL
        assert lib.layernorm_fwd_rows(p, ref, None, None, p, None, None, 8, 8, 1e-5, 1, 0,
                                      None) == GBN_EINVAL
        assert lib.rmsnorm_fwd_rows(p, ref, p, p, None, 8, 8, 1e-6, 1, 1, 0, None) == GBN_EINVAL
        assert lib.dyt_bwd_rows(p, None, p, ref, p, p, p, None, None, None, 8, 8, 1, 0, None, 0,
                                None) == GBN_EINVAL
        assert lib.layernorm_bwd_rows(p, ref, p, None, p, p, None, p, None, None, 8, 8, 1, 0,
                                      None, 0, None) == GBN_EINVAL
        assert lib.rmsnorm_bwd_rows(p, None, p, ref, p, None, p, None, 8, 8, 1e-6, 1, 1, 0,
                                    None, 0, None) == GBN_EINVAL
    # the other argument checks still come first
    good = ctypes.byref(R(4, 16, 2, 64, 128))
    assert lib.rmsnorm_fwd_rows(p, good, p, p, None, 8, 8, 1e-6, 1, 1, 3, None) == GBN_EINVAL
    assert lib.dyt_fwd_rows(p, good, p, p, p, p, 8, 8, 7, 0, None) == GBN_EDTYPE


def test_valid_layouts_get_to_the_device_query(lib):
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    p = ctypes.c_void_p(16)
    R = _lib.gbn_rows
    for lay in (R(4, 16, 2, 64, 128), R(8, 8, 1, 0, 0), R(3, 0, 1, 0, 0), R(1 << 40, 8, 1 << 40,
                                                                             0, 0)):
        ref = ctypes.byref(lay)
        assert lib.dyt_fwd_rows(p, ref, p, p, p, p, 8, 8, 1, 0, None) == GBN_EDEVICE
        assert lib.rmsnorm_bwd_rows(p, ref, p, ref, p, None, p, None, 8, 8, 1e-6, 1, 1, 0, None,
                                    0, None) == GBN_EDEVICE
    # an empty input needs no device in the forward
    ref = ctypes.byref(R(4, 16, 2, 64, 128))
    assert lib.dyt_fwd_rows(None, ref, p, p, p, None, 0, 8, 1, 0, None) == GBN_OK


def test_unused_levels_take_any_stride(lib):
    """A level that no row reaches (n1 == 1; n2 == 1; n1 * n2 >= M) may carry
    any stride, however large: it multiplies only zero and must not be scaled
    to bytes (INT64_MAX / 2 times the element size would overflow int64).
    The same stride on a level that rows do reach is rejected."""
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    p = ctypes.c_void_p(16)
    R = _lib.gbn_rows
    huge = (1 << 63) // 2
    unused = [R(1, huge, 8, 16, 0),        # n1 == 1: s1 unused
              R(8, 16, 1, huge, 128),      # n2 == 1: s2 unused
              R(4, 16, 2, 64, huge),       # n1 * n2 == M: s3 unused
              R(1, huge, 1, huge, 16),     # rows only through s3
              R(8, 16, 1 << 62, huge, huge)]
    for lay in unused:
        ref = ctypes.byref(lay)
        assert lib.dyt_fwd_rows(p, ref, p, p, p, p, 8, 8, 1, 0, None) == GBN_EDEVICE, \
            (lay.n1, lay.s1, lay.n2, lay.s2, lay.s3)
        assert lib.layernorm_bwd_rows(p, ref, p, ref, p, p, None, p, None, None, 8, 8, 1, 0,
                                      None, 0, None) == GBN_EDEVICE
    for lay in (R(2, huge, 4, 16, 0), R(2, 16, 2, 0, huge), R(4, 16, 2, huge, 0)):
        ref = ctypes.byref(lay)
        assert lib.dyt_fwd_rows(p, ref, p, p, p, p, 8, 8, 1, 0, None) == GBN_EINVAL
