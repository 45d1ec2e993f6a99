"""GB300 (sm_103a) library for the hot path of OSCAR-style 2-bit rotated KV-cache serving.

The compute lives in liboscar.so (hand-written CUDA behind the C ABI of include/oscar.h);
this package is a ctypes binding (_native), a torch-facing cache handle (cache), the
offline calibration step (calibrate) and seeded synthetic workloads (workloads).
"""
from . import _native
from ._native import OSCAR_FORMAT_BF16, OSCAR_FORMAT_INT2, OSCAR_FORMAT_INT2_CM, OscarError
from .cache import KVCache

__all__ = ["KVCache", "OscarError", "OSCAR_FORMAT_INT2", "OSCAR_FORMAT_INT2_CM", "OSCAR_FORMAT_BF16", "_native"]
