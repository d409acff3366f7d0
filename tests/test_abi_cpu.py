"""The C ABI without a GPU: libgbnorm.so builds for sm_103a, loads, exports
every function include/gbnorm.h declares, and rejects invalid arguments
with the documented status before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbnorm.h")

GBN_OK, GBN_EINVAL, GBN_EDTYPE, GBN_EWORKSPACE, GBN_ELAUNCH, GBN_EDEVICE = range(6)


@pytest.fixture(scope="module")
def lib():
    from normalization_layers_fwd_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|void)\s*\**\s*(\w+)\s*\(", text,
                      flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"dyt_fwd", "dyt_bwd", "layernorm_fwd", "layernorm_bwd", "rmsnorm_fwd", "rmsnorm_bwd",
            "gbn_bwd_workspace_bytes", "gbn_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    from normalization_layers_fwd_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_binding_signatures_cover_the_header():
    from normalization_layers_fwd_gb300 import _lib
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_status_strings(lib):
    for s in range(7):
        assert lib.gbn_status_string(s).startswith(b"GBN_")
    assert lib.gbn_status_string(99) == b"GBN_UNKNOWN"


def test_invalid_arguments_are_rejected_before_any_device_use(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # bad dtype codes
    assert lib.dyt_fwd(p, p, p, p, p, 4, 8, 7, 0, None) == GBN_EDTYPE
    assert lib.rmsnorm_fwd(p, p, p, None, 4, 8, 1e-6, 1, 9, None) == GBN_EDTYPE
    # RMSNorm with a 16-bit weight of the other 16-bit type has no rounding point
    assert lib.rmsnorm_fwd(p, p, p, None, 4, 8, 1e-6, 1, 2, None) == GBN_EDTYPE
    assert lib.rmsnorm_bwd(p, p, p, None, p, p, 4, 8, 1e-6, 2, 1, None, 0, None) == GBN_EDTYPE
    # ... in the Llama expression only; unknown expression codes are rejected
    assert lib.rmsnorm_fwd_ex(p, p, p, None, 4, 8, 1e-6, 1, 2, 0, None) == GBN_EDTYPE
    assert lib.rmsnorm_fwd_ex(p, p, p, None, 4, 8, 1e-6, 1, 1, 3, None) == GBN_EINVAL
    assert lib.rmsnorm_bwd_ex(p, p, p, None, p, p, 4, 8, 1e-6, 1, 1, -1, None, 0, None) == \
        GBN_EINVAL
    # bad shapes
    assert lib.dyt_fwd(p, p, p, p, p, -1, 8, 1, 0, None) == GBN_EINVAL
    assert lib.dyt_fwd(p, p, p, p, p, 4, 0, 1, 0, None) == GBN_EINVAL
    assert lib.dyt_fwd(p, p, p, p, p, 4, 1 << 31, 1, 0, None) == GBN_EINVAL
    assert lib.layernorm_fwd(p, None, None, p, None, None, 1 << 62, 1 << 20, 1e-5, 1, 0,
                             None) == GBN_EINVAL
    # required pointers
    assert lib.dyt_fwd(p, None, p, p, p, 4, 8, 1, 0, None) == GBN_EINVAL
    assert lib.dyt_fwd(None, p, p, p, p, 4, 8, 1, 0, None) == GBN_EINVAL
    assert lib.rmsnorm_fwd(p, None, p, None, 4, 8, 1e-6, 1, 1, None) == GBN_EINVAL
    assert lib.layernorm_bwd(p, p, None, p, None, p, None, None, 4, 8, 1, 0, None, 0,
                             None) == GBN_EINVAL
    # eps must be finite and >= 0
    assert lib.layernorm_fwd(p, None, None, p, None, None, 4, 8, float("nan"), 1, 0,
                             None) == GBN_EINVAL
    assert lib.rmsnorm_fwd(p, p, p, None, 4, 8, -1.0, 1, 1, None) == GBN_EINVAL
    # pointers must be aligned to their element size
    odd = ctypes.c_void_p(17)
    assert lib.dyt_fwd(odd, p, p, p, p, 4, 8, 1, 0, None) == GBN_EINVAL
    assert lib.dyt_fwd(p, ctypes.c_void_p(18), p, p, p, 4, 8, 1, 0, None) == GBN_EINVAL
    assert lib.rmsnorm_fwd(p, p, p, ctypes.c_void_p(18), 4, 8, 1e-6, 1, 1, None) == GBN_EINVAL
    # misaligned workspace
    assert lib.dyt_bwd(p, p, p, p, p, p, p, p, 4, 8, 1, 0, ctypes.c_void_p(18), 1 << 20,
                       None) == GBN_EINVAL


def test_empty_forward_is_a_noop_without_device(lib):
    p = ctypes.c_void_p(16)
    assert lib.dyt_fwd(None, p, p, p, None, 0, 8, 1, 0, None) == GBN_OK
    assert lib.layernorm_fwd(None, None, None, None, None, None, 0, 8, 1e-5, 1, 0, None) == GBN_OK
    assert lib.rmsnorm_fwd(None, p, None, None, 0, 8, 1e-6, 1, 1, None) == GBN_OK


def test_f16_codes_are_accepted(lib):
    """binary16 (code 2) passes the dtype checks: without a device the call
    gets as far as the device query."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    size_max = ctypes.c_size_t(-1).value
    p = ctypes.c_void_p(16)
    for xt, pt in ((2, 2), (2, 0), (0, 2)):
        assert lib.dyt_fwd(p, p, p, p, p, 4, 8, xt, pt, None) == GBN_EDEVICE
        assert lib.rmsnorm_fwd(p, p, p, None, 4, 8, 1e-6, xt, pt, None) == GBN_EDEVICE
    assert lib.gbn_bwd_workspace_bytes(2, 10, 10, 2, 2, 0) == size_max  # no device here


def test_valid_call_without_a_device_reports_edevice(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    p = ctypes.c_void_p(16)
    assert lib.dyt_fwd(p, p, p, p, p, 4, 8, 1, 0, None) == GBN_EDEVICE


def test_fault_api_validates_without_device(lib):
    import torch
    assert lib.gbn_read_faults(None, 0) == GBN_EINVAL
    assert lib.gbn_selftest_wait_timeout(0, ctypes.c_void_p(16), None) == GBN_EINVAL
    assert lib.gbn_selftest_wait_timeout(1 << 40, ctypes.c_void_p(16), None) == GBN_EINVAL
    if not torch.cuda.is_available():
        v = ctypes.c_uint(5)
        assert lib.gbn_read_faults(ctypes.byref(v), 0) == GBN_EDEVICE


def test_workspace_query(lib):
    from normalization_layers_fwd_gb300._lib import SIZE_MAX
    assert lib.gbn_bwd_workspace_bytes(5, 10, 10, 1, 0, 0) == SIZE_MAX
    assert lib.gbn_bwd_workspace_bytes(0, 10, 10, 3, 0, 0) == SIZE_MAX
    assert lib.gbn_bwd_workspace_bytes(0, -1, 10, 1, 0, 0) == SIZE_MAX
    assert lib.gbn_bwd_workspace_bytes(0, 0, 10, 1, 0, 0) == 0


def test_missing_library_fails_loudly():
    from normalization_layers_fwd_gb300 import _lib
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.load("/nonexistent/libgbnorm.so")


def test_binding_rejects_host_tensors():
    import torch
    from normalization_layers_fwd_gb300 import _lib
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        _lib.rmsnorm_fwd(x, torch.ones(8))
