"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/proj.h declares, and rejects bad arguments with the
documented status before touching a device."""
import ctypes

import numpy as np
import pytest

from gemv_projection_layers_gb300 import binding as B
from gemv_projection_layers_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.load()


def test_every_declared_function_is_exported(lib):
    names = B.header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n


def test_argument_errors_before_any_device_call(lib):
    # Wrong layer / shape / dtype / NULL weights: no CUDA call is made.
    assert lib.proj_prepare(7, 16, 2304, 8192, 0) is None
    assert B.proj_last_status() == B.PROJ_EINVAL
    assert lib.proj_prepare(B.PROJ_O, 16, 8192, 1000, B.PROJ_BF16) is None
    assert B.proj_last_status() == B.PROJ_EINVAL
    assert lib.proj_prepare(B.PROJ_ROUTER, 16, 256, 8192, B.PROJ_BF16) is None
    assert B.proj_last_status() == B.PROJ_EINVAL
    assert lib.proj_prepare(B.PROJ_O, None, 8192, 1024, B.PROJ_BF16) is None
    assert B.proj_last_status() == B.PROJ_EINVAL
    assert lib.proj_prepare(B.PROJ_O, 8, 8192, 1024, B.PROJ_BF16) is None
    assert B.proj_last_status() == B.PROJ_EALIGN
    st = ctypes.c_int(-1)
    assert lib.proj_prepare_ex(B.PROJ_O, 16, 8192, 1024, B.PROJ_BF16, 1 << 5, 0,
                               ctypes.byref(st)) is None
    assert st.value == B.PROJ_EINVAL
    # NULL handles
    assert lib.proj_run(None, 16, 1, 16, None) == B.PROJ_EINVAL
    assert lib.proj_run_host(None, 16, 1, 16, None) == B.PROJ_EINVAL
    assert lib.proj_out_features(None, 1) == -1
    assert lib.proj_info(None, None) == B.PROJ_EINVAL
    assert lib.proj_describe(None, 1, None, 0) == B.PROJ_EINVAL
    assert lib.proj_unpack_weights(None, 0, 16, None) == B.PROJ_EINVAL
    assert lib.proj_device_status(None, None, None) == B.PROJ_EINVAL
    lib.proj_destroy(None)
    # read floor argument checks
    assert lib.proj_read_floor(None, 16, 16, 0, 0, None) == B.PROJ_EINVAL
    assert lib.proj_read_floor(16, 15, 16, 0, 0, None) == B.PROJ_EINVAL
    assert lib.proj_read_floor(16, 16, 16, 0, 2, None) == B.PROJ_EINVAL
    assert lib.proj_read_floor(16, 16, 16, 0, 8, None) == B.PROJ_EINVAL
    assert lib.proj_read_floor(16, 16, 16, 0, -1, None) == B.PROJ_EINVAL
    assert lib.proj_read_floor(8, 16, 16, 0, 0, None) == B.PROJ_EALIGN
    # FMA probe argument checks
    assert lib.proj_fma_peak(None, 16, 0, None, None) == B.PROJ_EINVAL
    assert lib.proj_fma_peak(16, 0, 4, None, None) == B.PROJ_EINVAL
    assert lib.proj_fma_peak(16, (1 << 24) + 1, 4, None, None) == B.PROJ_EINVAL
    assert lib.proj_fma_peak(16, 16, -1, None, None) == B.PROJ_EINVAL
    assert lib.proj_fma_peak(18, 16, 4, None, None) == B.PROJ_EALIGN


def test_status_strings(lib):
    for s in range(7):
        assert B.status_string(s)
    assert B.status_string(99) == "unknown status"
    with pytest.raises(B.ProjError):
        B.proj_run(0, 16, 1, 16)


def test_binding_constants_match_the_header():
    """Every PROJ_* constant the binding defines has the header's value
    (enumerators written `NAME = value` and `#define NAME value`)."""
    import re
    text = open(B.HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    declared = {}
    for name, val in re.findall(r"\b(PROJ_[A-Z0-9_]+)\s*=\s*([0-9]+u?(?:\s*<<\s*[0-9]+)?)", text):
        declared[name] = eval(val.replace("u", ""))
    for name, val in re.findall(r"#define\s+(PROJ_[A-Z0-9_]+)\s+([0-9]+)", text):
        declared[name] = int(val)
    consts = {n: getattr(B, n) for n in dir(B) if n.startswith("PROJ_") and isinstance(getattr(B, n), int)}
    assert len(consts) >= 30
    for n, v in consts.items():
        assert n in declared, n
        assert declared[n] == v, (n, declared[n], v)
