"""GB300-native dense projections (out = x @ W.T) behind a C ABI.

The compute runs in libproj.so (CUDA kernels for sm_103a); this package
holds its ctypes binding (`binding`, same names as include/proj.h), the
build script (`build`) and the seeded synthetic workloads (`workloads`).
"""
from . import workloads  # noqa: F401
from .binding import *  # noqa: F401,F403
from .binding import ProjError, NativeLibraryMissing, load, LIB_PATH  # noqa: F401
