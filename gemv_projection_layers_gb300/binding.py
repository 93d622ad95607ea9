"""ctypes binding of libproj (include/proj.h): same names, argument
marshalling only.  Every step of the projection runs in the library's CUDA
kernels; if the library is missing this module raises instead of falling
back to anything else.

Pointer arguments accept an int (raw address), a torch tensor (its
data_ptr()) or a numpy array (host address).  Stream arguments accept None
(legacy default stream), an int handle or a torch.cuda.Stream.  Calls that
return a status raise ProjError on anything but PROJ_OK.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libproj.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "proj.h")

PROJ_QKV_GATE, PROJ_O, PROJ_POOLER, PROJ_UNPOOLER, PROJ_ROUTER = range(5)
PROJ_BF16, PROJ_FP32 = 0, 1
PROJ_ENCODE_EXPWIN12 = 1
(PROJ_OK, PROJ_EINVAL, PROJ_EUNSUPPORTED, PROJ_EALIGN, PROJ_ENOMEM, PROJ_ECUDA,
 PROJ_EDEVICE) = range(7)
PROJ_VARIANT_AUTO, PROJ_VARIANT_DENSE, PROJ_VARIANT_EXPWIN12, PROJ_VARIANT_PLANES3 = range(4)
PROJ_REDUCE_AUTO, PROJ_REDUCE_OWNER, PROJ_REDUCE_DISTRIBUTED = range(3)
(PROJ_KERNEL_AUTO, PROJ_KERNEL_GEMV, PROJ_KERNEL_TILE, PROJ_KERNEL_CLUSTER, PROJ_KERNEL_GEMV_REG,
 PROJ_KERNEL_MMA, PROJ_KERNEL_GEMV_SPLITK, PROJ_KERNEL_PAIR, PROJ_KERNEL_ROWS) = range(9)
PROJ_UNPACK_FRAG16 = 16  # proj_unpack_weights: the few-token GEMV's fragment-order copy
PROJ_UNPACK_RC12 = 32  # proj_unpack_weights: the register GEMV's 12-bit row-chunk copy
PROJ_UNPACK_FRAG12 = 64  # proj_unpack_weights: the warp-MMA GEMV's 12-bit fragment copy
PROJ_UNPACK_RUNS = 128  # proj_unpack_weights: the row-run GEMV's copy (all N rows)
PROJ_UNPACK_RUNS_SLICE = 256  # proj_unpack_weights: the unpooler's row-run copy of its slice
PROJ_READ_PDL = 4  # proj_read_floor mode flag: launched as a programmatic dependent launch

LAYER_INDEX = {"qkv_gate": 0, "o": 1, "pooler": 2, "unpooler": 3, "router": 4}


class ProjError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})"
                         + (f" [{last_cuda_error()}]" if status == PROJ_ECUDA else ""))


class NativeLibraryMissing(ImportError):
    pass


class proj_run_opts(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("grid", ctypes.c_int),
                ("reduce", ctypes.c_int), ("kernel", ctypes.c_int), ("groups", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("stamps", ctypes.c_void_p)]


class proj_info_t(ctypes.Structure):
    _fields_ = [("layer", ctypes.c_int), ("dtype", ctypes.c_int),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("m_max", ctypes.c_int64),
                ("expwin12", ctypes.c_int), ("expwin12_declined", ctypes.c_int),
                ("expwin12_e0", ctypes.c_int),
                ("expwin12_escapes", ctypes.c_int64), ("expwin12_bytes", ctypes.c_int64),
                ("dense_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("num_sms", ctypes.c_int), ("reserved", ctypes.c_int * 7)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libproj.so (raises NativeLibraryMissing if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise NativeLibraryMissing(
            f"{LIB_PATH} is missing: build it with `python -m gemv_projection_layers_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
    lib.proj_prepare.restype = vp
    lib.proj_prepare.argtypes = [i32, vp, i64, i64, i32]
    lib.proj_prepare_ex.restype = vp
    lib.proj_prepare_ex.argtypes = [i32, vp, i64, i64, i32, u32, i64, ctypes.POINTER(i32)]
    lib.proj_run.restype = i32
    lib.proj_run.argtypes = [vp, vp, i64, vp, vp]
    lib.proj_run_ex.restype = i32
    lib.proj_run_ex.argtypes = [vp, vp, i64, vp, vp, ctypes.POINTER(proj_run_opts)]
    lib.proj_run_host.restype = i32
    lib.proj_run_host.argtypes = [vp, vp, i64, vp, vp]
    lib.proj_out_features.restype = i64
    lib.proj_out_features.argtypes = [vp, i64]
    lib.proj_info.restype = i32
    lib.proj_info.argtypes = [vp, ctypes.POINTER(proj_info_t)]
    lib.proj_describe.restype = i32
    lib.proj_describe.argtypes = [vp, i64, ctypes.c_char_p, ctypes.c_size_t]
    lib.proj_describe_ex.restype = i32
    lib.proj_describe_ex.argtypes = [vp, i64, ctypes.POINTER(proj_run_opts), ctypes.c_char_p,
                                     ctypes.c_size_t]
    lib.proj_unpack_weights.restype = i32
    lib.proj_unpack_weights.argtypes = [vp, i32, vp, vp]
    lib.proj_device_status.restype = i32
    lib.proj_device_status.argtypes = [vp, vp, ctypes.POINTER(u32)]
    lib.proj_destroy.restype = None
    lib.proj_destroy.argtypes = [vp]
    lib.proj_last_status.restype = i32
    lib.proj_last_status.argtypes = []
    lib.proj_status_string.restype = ctypes.c_char_p
    lib.proj_status_string.argtypes = [i32]
    lib.proj_last_cuda_error.restype = ctypes.c_char_p
    lib.proj_last_cuda_error.argtypes = []
    lib.proj_read_floor.restype = i32
    lib.proj_read_floor.argtypes = [vp, i64, vp, i32, i32, vp]
    lib.proj_fma_peak.restype = i32
    lib.proj_fma_peak.argtypes = [vp, i32, i32, vp, ctypes.POINTER(ctypes.c_double)]
    lib.proj_num_sms.restype = i32
    lib.proj_num_sms.argtypes = []
    lib.proj_gemv_static.argtypes = [vp, i32, i64, i64, vp, i64, vp, vp]
    lib.proj_gemv_static.restype = i32
    lib.proj_gemv_static_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.proj_gemv_static_status.restype = i32
    _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions include/proj.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(proj_[a-z_0-9]+)\s*\(", text)))


# ------------------------------------------------------------ marshalling --

def _addr(p) -> int | None:
    if p is None:
        return None
    if isinstance(p, int):
        return p
    if hasattr(p, "data_ptr"):
        return int(p.data_ptr())
    if hasattr(p, "ctypes"):
        return int(p.ctypes.data)
    raise TypeError(f"cannot take the address of {type(p)!r}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError(f"not a stream: {type(s)!r}")


def _check(status: int, what: str) -> None:
    if status != PROJ_OK:
        raise ProjError(status, what)


# ---------------------------------------------------------------- the ABI --

def proj_prepare(layer: int, W, N: int, K: int, dtype: int) -> int:
    h = load().proj_prepare(int(layer), _addr(W), int(N), int(K), int(dtype))
    if not h:
        raise ProjError(proj_last_status(), "proj_prepare")
    return h


def proj_prepare_ex(layer: int, W, N: int, K: int, dtype: int, flags: int = 0,
                    m_max: int = 0) -> int:
    st = ctypes.c_int(0)
    h = load().proj_prepare_ex(int(layer), _addr(W), int(N), int(K), int(dtype), int(flags),
                               int(m_max), ctypes.byref(st))
    if not h:
        raise ProjError(st.value, "proj_prepare_ex")
    return h


def proj_run(h: int, x, m: int, out, stream=None) -> None:
    _check(load().proj_run(h, _addr(x), int(m), _addr(out), _stream(stream)), "proj_run")


def proj_run_ex(h: int, x, m: int, out, stream=None, variant: int = PROJ_VARIANT_AUTO,
                grid: int = 0, reduce: int = PROJ_REDUCE_AUTO,
                kernel: int = PROJ_KERNEL_AUTO, groups: int = 0, tile_n: int = 0,
                stamps=None) -> None:
    opts = proj_run_opts(int(variant), int(grid), int(reduce), int(kernel), int(groups),
                         int(tile_n), _addr(stamps))
    _check(load().proj_run_ex(h, _addr(x), int(m), _addr(out), _stream(stream),
                              ctypes.byref(opts)), "proj_run_ex")


def proj_run_host(h: int, x_host, m: int, out_host, stream=None) -> None:
    _check(load().proj_run_host(h, _addr(x_host), int(m), _addr(out_host), _stream(stream)),
           "proj_run_host")


def proj_out_features(h: int, m: int) -> int:
    return int(load().proj_out_features(h, int(m)))


def proj_info(h: int) -> dict:
    info = proj_info_t()
    _check(load().proj_info(h, ctypes.byref(info)), "proj_info")
    return {name: getattr(info, name) for name, _ in proj_info_t._fields_ if name != "reserved"}


def proj_describe(h: int, m: int) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(load().proj_describe(h, int(m), buf, 256), "proj_describe")
    return buf.value.decode()


def proj_describe_ex(h: int, m: int, variant: int = PROJ_VARIANT_AUTO, grid: int = 0,
                     reduce: int = PROJ_REDUCE_AUTO, kernel: int = PROJ_KERNEL_AUTO,
                     groups: int = 0, tile_n: int = 0) -> str:
    opts = proj_run_opts(int(variant), int(grid), int(reduce), int(kernel), int(groups),
                         int(tile_n))
    buf = ctypes.create_string_buffer(256)
    _check(load().proj_describe_ex(h, int(m), ctypes.byref(opts), buf, 256), "proj_describe_ex")
    return buf.value.decode()


def proj_unpack_weights(h: int, variant: int, W_out, stream=None) -> None:
    _check(load().proj_unpack_weights(h, int(variant), _addr(W_out), _stream(stream)),
           "proj_unpack_weights")


def proj_device_status(h: int, stream=None) -> int:
    code = ctypes.c_uint32(0)
    st = load().proj_device_status(h, _stream(stream), ctypes.byref(code))
    if st not in (PROJ_OK, PROJ_EDEVICE):
        raise ProjError(st, "proj_device_status")
    return int(code.value)


def proj_destroy(h: int) -> None:
    if h:
        load().proj_destroy(h)


def proj_last_status() -> int:
    return int(load().proj_last_status())


def status_string(status: int) -> str:
    return load().proj_status_string(int(status)).decode()


proj_status_string = status_string


def last_cuda_error() -> str:
    return load().proj_last_cuda_error().decode()


proj_last_cuda_error = last_cuda_error


def proj_read_floor(buf, nbytes: int, sink, grid: int = 0, mode: int = 0, stream=None) -> None:
    _check(load().proj_read_floor(_addr(buf), int(nbytes), _addr(sink), int(grid), int(mode),
                                  _stream(stream)), "proj_read_floor")


def proj_fma_peak(sink, iters: int, grid: int = 0, stream=None) -> float:
    """Enqueue the FP32 FMA probe; returns the launch's FLOPs."""
    flops = ctypes.c_double(0.0)
    _check(load().proj_fma_peak(_addr(sink), int(iters), int(grid), _stream(stream),
                                ctypes.byref(flops)), "proj_fma_peak")
    return float(flops.value)


def proj_num_sms() -> int:
    return int(load().proj_num_sms())


def proj_gemv_static(W, w_dtype: int, N: int, K: int, x, m: int, out, stream=None) -> None:
    """Allocation-free GEMV (m <= 2) on caller-owned row-major weights; see
    proj.h for the limits and for the shared static scratch."""
    st = load().proj_gemv_static(_addr(W), int(w_dtype), int(N), int(K), _addr(x), int(m),
                                 _addr(out), _stream(stream))
    if st != PROJ_OK:
        raise ProjError(st, f"proj_gemv_static ({last_cuda_error()})")


def proj_gemv_static_status(stream=None) -> int:
    """Status word of the last proj_gemv_static call on the current device
    (synchronises `stream`); 0 when every bounded wait completed."""
    code = ctypes.c_uint32(0)
    st = load().proj_gemv_static_status(_stream(stream), ctypes.byref(code))
    if st not in (PROJ_OK, PROJ_EDEVICE):
        raise ProjError(st, f"proj_gemv_static_status ({last_cuda_error()})")
    return int(code.value)
