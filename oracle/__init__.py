"""CPU oracle for NHWC conv2d and transposed conv (fp64, single thread).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, compiled with gcc -O2, no
fast-math, no threads); this module compiles it on demand and wraps it with
numpy arrays.  See ``oracle.c`` for the definitions and the pages they follow:
"dispatch_amd_4wave_conv2d" (residual, layouts, gates),
"dispatch_fused_im2col_conv2d_apple" (GEMM view, filter layouts) and
"conv_transposed_gpu" (transposed conv as backward-data, RSFC filter).

Every function is pinned by ``tests/test_oracle_pins.py`` to something other
than itself; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

BF16, F16, F8E4M3 = 0, 1, 2
ACT_NONE, ACT_RELU, ACT_SILU = 0, 1, 2
DTYPE_CODES = {"bf16": BF16, "f16": F16, "f8e4m3": F8E4M3}
ACT_CODES = {"none": ACT_NONE, "relu": ACT_RELU, "silu": ACT_SILU}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc -O2, one thread, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, dbl, P = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.oracle_decode_one.argtypes = [ctypes.c_uint32, i32]
            lib.oracle_decode_one.restype = dbl
            lib.oracle_decode.argtypes = [P, i32, i64, P]
            lib.oracle_decode.restype = i32
            lib.oracle_activation.argtypes = [dbl, i32]
            lib.oracle_activation.restype = dbl
            conv_args = [P, i64, i64, i64, i64, P, i64, i64, i64]
            geo = [i32] * 6 + [i64, i64, i32, P, dbl, i32]
            fwd_args = [P, i64, i64, i64, i64, i64, P, i64, i64, i64]  # + groups after C
            lib.oracle_conv2d_fwd.argtypes = fwd_args + [i32] + geo + [P]
            lib.oracle_conv2d_fwd.restype = i32
            lib.oracle_conv2d_fwd_points.argtypes = fwd_args + [i32] + geo + [P, i64, P]
            lib.oracle_conv2d_fwd_points.restype = i32
            lib.oracle_conv_transposed.argtypes = conv_args + geo + [P]
            lib.oracle_conv_transposed.restype = i32
            lib.oracle_conv_transposed_points.argtypes = conv_args + geo + [P, i64, P]
            lib.oracle_conv_transposed_points.restype = i32
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def decode(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Decode raw storage bits (uint16 for bf16/f16, uint8 for fp8-e4m3) to fp64."""
    code = DTYPE_CODES[dtype]
    want = np.uint8 if code == F8E4M3 else np.uint16
    raw = np.ascontiguousarray(raw).view(want)
    out = np.empty(raw.shape, dtype=np.float64)
    if _load().oracle_decode(_ptr(raw), code, raw.size, _ptr(out)) != 0:
        raise ValueError("bad dtype")
    return out


def decode_one(bits: int, dtype: str) -> float:
    return _load().oracle_decode_one(bits, DTYPE_CODES[dtype])


def activation(v: float, act: str) -> float:
    return _load().oracle_activation(v, ACT_CODES[act])


def fwd_out_size(h, r, stride, pad, dil):
    """Forward output extent floor((h + 2p - d(r-1) - 1)/s) + 1."""
    return (h + 2 * pad - dil * (r - 1) - 1) // stride + 1


def _res_args(source, shape):
    if source is None:
        return 0, None, np.zeros(1)
    src = _f64(source)
    if src.shape != tuple(shape):
        raise ValueError("source shape %s != output shape %s" % (src.shape, tuple(shape)))
    return 1, src, src


def conv2d_fwd(x, w, *, filter_is_fcrs, stride=(1, 1), padding=(0, 0), dilation=(1, 1),
               source=None, beta=0.0, act="none", out_hw=None, groups=1) -> np.ndarray:
    """Forward NHWC conv over fp64 arrays. x: [N,H,W,C]; w: FCRS [F,C/G,R,S] or RSCF
    [R,S,C/G,F] for G = ``groups`` channel groups."""
    x, w = _f64(x), _f64(w)
    N, H, W, C = x.shape
    if filter_is_fcrs:
        F, C2, R, S = w.shape
    else:
        R, S, C2, F = w.shape
    if C2 * groups != C or F % groups != 0:
        raise ValueError("filter channels do not match the input and groups")
    sh, sw = stride
    ph, pw = padding
    dh, dw = dilation
    Ho, Wo = out_hw if out_hw is not None else (fwd_out_size(H, R, sh, ph, dh),
                                               fwd_out_size(W, S, sw, pw, dw))
    y = np.empty((N, Ho, Wo, F), dtype=np.float64)
    has_res, _, src = _res_args(source, y.shape)
    rc = _load().oracle_conv2d_fwd(_ptr(x), N, H, W, C, int(groups), _ptr(w), R, S, F,
                                   int(bool(filter_is_fcrs)),
                                   sh, sw, ph, pw, dh, dw, Ho, Wo, has_res, _ptr(src), float(beta),
                                   ACT_CODES[act], _ptr(y))
    if rc != 0:
        raise ValueError("oracle_conv2d_fwd rejected its arguments")
    return y


def conv2d_fwd_points(x, w, pts, *, filter_is_fcrs, stride=(1, 1), padding=(0, 0),
                      dilation=(1, 1), source=None, beta=0.0, act="none", out_hw=None, groups=1):
    """Forward conv evaluated only at flat NHWC output indices ``pts``."""
    x, w = _f64(x), _f64(w)
    N, H, W, C = x.shape
    if filter_is_fcrs:
        F, _, R, S = w.shape
    else:
        R, S, _, F = w.shape
    sh, sw = stride
    ph, pw = padding
    dh, dw = dilation
    Ho, Wo = out_hw if out_hw is not None else (fwd_out_size(H, R, sh, ph, dh),
                                               fwd_out_size(W, S, sw, pw, dw))
    pts = np.ascontiguousarray(pts, dtype=np.int64)
    out = np.empty(pts.shape, dtype=np.float64)
    has_res, _, src = _res_args(source, (N, Ho, Wo, F))
    rc = _load().oracle_conv2d_fwd_points(_ptr(x), N, H, W, C, int(groups), _ptr(w), R, S, F,
                                          int(bool(filter_is_fcrs)), sh, sw, ph, pw, dh, dw, Ho, Wo,
                                          has_res, _ptr(src), float(beta), ACT_CODES[act],
                                          _ptr(pts), pts.size, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_conv2d_fwd_points rejected its arguments")
    return out


def conv_transposed(x, w_rsfc, *, out_hw, stride=(1, 1), padding=(0, 0), dilation=(1, 1),
                    source=None, beta=0.0, act="none") -> np.ndarray:
    """Transposed NHWC conv (scatter form). x: [N,H,W,C]; w_rsfc: [R,S,F,C]."""
    x, w = _f64(x), _f64(w_rsfc)
    N, H, W, C = x.shape
    R, S, F, C2 = w.shape
    if C2 != C:
        raise ValueError("filter C mismatch")
    Ho, Wo = out_hw
    y = np.empty((N, Ho, Wo, F), dtype=np.float64)
    has_res, _, src = _res_args(source, y.shape)
    rc = _load().oracle_conv_transposed(_ptr(x), N, H, W, C, _ptr(w), R, S, F,
                                        stride[0], stride[1], padding[0], padding[1],
                                        dilation[0], dilation[1], Ho, Wo, has_res, _ptr(src),
                                        float(beta), ACT_CODES[act], _ptr(y))
    if rc != 0:
        raise ValueError("oracle_conv_transposed rejected its arguments")
    return y


def conv_transposed_points(x, w_rsfc, pts, *, out_hw, stride=(1, 1), padding=(0, 0),
                           dilation=(1, 1), source=None, beta=0.0, act="none"):
    """Transposed conv evaluated only at flat NHWC output indices ``pts``."""
    x, w = _f64(x), _f64(w_rsfc)
    N, H, W, C = x.shape
    R, S, F, _ = w.shape
    Ho, Wo = out_hw
    pts = np.ascontiguousarray(pts, dtype=np.int64)
    out = np.empty(pts.shape, dtype=np.float64)
    has_res, _, src = _res_args(source, (N, Ho, Wo, F))
    rc = _load().oracle_conv_transposed_points(_ptr(x), N, H, W, C, _ptr(w), R, S, F,
                                               stride[0], stride[1], padding[0], padding[1],
                                               dilation[0], dilation[1], Ho, Wo, has_res,
                                               _ptr(src), float(beta), ACT_CODES[act],
                                               _ptr(pts), pts.size, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_conv_transposed_points rejected its arguments")
    return out


def tolerance(oracle_vals, K, max_a, max_b, dtype):
    """Per-element parity bound |gpu - oracle| <= rel*|oracle| + 2e-3*sqrt(K)*max|a|*max|b|,
    rel = 1e-2 for bf16/f16 inputs and 2e-2 for fp8-e4m3 inputs."""
    rel = 2e-2 if dtype == "f8e4m3" else 1e-2
    return rel * np.abs(oracle_vals) + 2e-3 * np.sqrt(K) * max_a * max_b
