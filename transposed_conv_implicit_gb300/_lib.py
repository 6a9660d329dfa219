"""ctypes loader and signatures for libconvgb300.so (the C ABI in include/conv_gb300.h).

The library is loaded on first use.  If it has not been built, every call
raises: there is no CPU or library fallback behind this package.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libconvgb300.so")

_lock = threading.Lock()
_lib = None

# conv_status_t
CONV_OK = 0
CONV_ERR_INVALID_VALUE = 1
CONV_ERR_NOT_SUPPORTED = 2
CONV_ERR_MISALIGNED = 3
CONV_ERR_WORKSPACE_TOO_SMALL = 4
CONV_ERR_CUDA = 5
CONV_ERR_DEVICE_TIMEOUT = 6
CONV_STATUS_BYTES = 256
CONV_NOALLOC_SCRATCH_BYTES = 8 << 20

# conv_dtype_t / conv_epilogue_t
DTYPE_CODES = {"bf16": 0, "f16": 1, "f8e4m3": 2}
EPILOGUE_CODES = {"none": 0, "relu": 1, "silu": 2}

# Every symbol the headers declare (checked by the CPU tests).
EXPORTS = (
    "conv_status_string", "conv2d_packed_filter_bytes", "conv2d_pack_filter",
    "conv2d_workspace_size", "conv2d_fwd", "conv2d_fwd_packed",
    "conv_transposed_packed_filter_bytes", "conv_transposed_workspace_size",
    "conv_transposed_pack_filter", "conv_transposed", "conv_transposed_packed",
    "conv_check_device_status", "conv_testing_set_wait_fault", "conv_testing_im2col_tile",
    "conv_testing_fwd_plan", "conv2d_fwd_noalloc", "conv_testing_reload_tuning",
    "conv_testing_cache_stats", "conv_streamk_workspace_size",
    "conv_transposed_packed_filter_bytes_dilated", "conv_transposed_workspace_size_dilated",
    "conv_transposed_pack_filter_dilated",
)


class ExtensionMissing(RuntimeError):
    pass


def _declare(lib):
    P, I, F, Z, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_ulonglong
    IP = ctypes.POINTER(ctypes.c_int)
    lib.conv_status_string.argtypes = [I]
    lib.conv_status_string.restype = ctypes.c_char_p
    lib.conv2d_packed_filter_bytes.argtypes = [I, I, I, I, I]
    lib.conv2d_packed_filter_bytes.restype = Z
    lib.conv2d_workspace_size.argtypes = [I, I, I, I, I]
    lib.conv2d_workspace_size.restype = Z
    lib.conv_streamk_workspace_size.argtypes = []
    lib.conv_streamk_workspace_size.restype = Z
    lib.conv2d_pack_filter.argtypes = [P, I, I, I, I, I, I, P, Z, P]
    lib.conv2d_pack_filter.restype = I
    fwd_tail = [IP, IP, IP, I, I, P, F, I, P, Z, P]
    lib.conv2d_fwd.argtypes = [P, I, I, I, I, I, P, I, I, I, I, P, I, I, I] + fwd_tail
    lib.conv2d_fwd.restype = I
    lib.conv2d_fwd_packed.argtypes = [P, I, I, I, I, I, P, I, I, I, P, I, I, I] + fwd_tail
    lib.conv2d_fwd_packed.restype = I
    lib.conv_transposed_packed_filter_bytes.argtypes = [I, I, I, I, IP, IP, I]
    lib.conv_transposed_packed_filter_bytes.restype = Z
    lib.conv_transposed_workspace_size.argtypes = [I, I, I, I, IP, IP, I]
    lib.conv_transposed_workspace_size.restype = Z
    lib.conv_transposed_pack_filter.argtypes = [P, I, I, I, I, IP, IP, I, P, Z, P]
    lib.conv_transposed_pack_filter.restype = I
    lib.conv_transposed_packed_filter_bytes_dilated.argtypes = [I, I, I, I, IP, IP, IP, I]
    lib.conv_transposed_packed_filter_bytes_dilated.restype = Z
    lib.conv_transposed_workspace_size_dilated.argtypes = [I, I, I, I, IP, IP, IP, I]
    lib.conv_transposed_workspace_size_dilated.restype = Z
    lib.conv_transposed_pack_filter_dilated.argtypes = [P, I, I, I, I, IP, IP, IP, I, P, Z, P]
    lib.conv_transposed_pack_filter_dilated.restype = I
    tr_tail = [IP, IP, IP, I, P, F, I, P, Z, P]
    lib.conv_transposed.argtypes = [P, I, I, I, I, I, P, I, I, I, P, I, I, I] + tr_tail
    lib.conv_transposed.restype = I
    lib.conv_transposed_packed.argtypes = [P, I, I, I, I, I, P, I, I, I, P, I, I, I] + tr_tail
    lib.conv_transposed_packed.restype = I
    lib.conv2d_fwd_noalloc.argtypes = [P, I, I, I, I, I, P, I, I, I, I, P, I, I, I,
                                       IP, IP, IP, I, I, P, F, I, P]
    lib.conv2d_fwd_noalloc.restype = I
    lib.conv_check_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint)]
    lib.conv_check_device_status.restype = I
    lib.conv_testing_set_wait_fault.argtypes = [I, U64]
    lib.conv_testing_set_wait_fault.restype = None
    lib.conv_testing_im2col_tile.argtypes = [P, I, I, I, I, I, I, I, IP, IP, I, I, I, I, P, IP, P, P]
    lib.conv_testing_im2col_tile.restype = I
    lib.conv_testing_fwd_plan.argtypes = [I, I, I, I, I, I, I, I, IP, IP, I, I, Z, IP]
    lib.conv_testing_fwd_plan.restype = I
    lib.conv_testing_reload_tuning.argtypes = []
    lib.conv_testing_reload_tuning.restype = None
    lib.conv_testing_cache_stats.argtypes = [ctypes.POINTER(U64), ctypes.POINTER(U64)]
    lib.conv_testing_cache_stats.restype = None
    return lib


def lib():
    """The loaded library; raises ExtensionMissing if it was never built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ExtensionMissing(
                    "libconvgb300.so is not built (expected at %s); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def pair(v):
    a = (ctypes.c_int * 2)(*(int(x) for x in v))
    return a
