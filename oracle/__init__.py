"""CPU oracle for the row-wise normalization path (ctypes over ``oracle.c``).

TEST INFRASTRUCTURE ONLY.  The product package never imports this module;
only ``tests/``, the smoke check in ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

Arrays are numpy: binary32 data as ``float32``, binary16 and bfloat16 data as
raw ``uint16`` bit patterns (dtype codes 0 = f32, 1 = f16, 2 = bf16).
Statistics come back in double.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, F16, BF16 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra=()) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc."""
    cmd = ["gcc", *_CFLAGS, *extra, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> str:
    """Build liboracle.so next to the source if missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            compile_oracle()
    return _LIB_PATH


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _declare(lib):
    lib.orc_layernorm.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                  ctypes.c_float]
    lib.orc_rmsnorm.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _I64, _I64, ctypes.c_float]
    lib.orc_add_rmsnorm.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                    ctypes.c_float]
    lib.orc_batchnorm_train.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _I64, _I64, _I64, ctypes.c_float, ctypes.c_float]
    lib.orc_batchnorm_infer.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                        _I64, ctypes.c_float]
    lib.orc_batchnorm_backward.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                           _I64, _I64, _I64]
    lib.orc_softmax.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _I64, _I64]
    for name in ("orc_layernorm", "orc_rmsnorm", "orc_add_rmsnorm", "orc_batchnorm_train",
                 "orc_batchnorm_infer", "orc_batchnorm_backward", "orc_softmax"):
        getattr(lib, name).restype = ctypes.c_int
    lib.orc_f16_bits_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_f16_bits_to_double.restype = ctypes.c_double
    lib.orc_bf16_bits_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_bits_to_double.restype = ctypes.c_double
    lib.orc_double_to_f16_bits.argtypes = [ctypes.c_double]
    lib.orc_double_to_f16_bits.restype = ctypes.c_uint16
    lib.orc_double_to_bf16_bits.argtypes = [ctypes.c_double]
    lib.orc_double_to_bf16_bits.restype = ctypes.c_uint16
    lib.orc_double_to_f32.argtypes = [ctypes.c_double]
    lib.orc_double_to_f32.restype = ctypes.c_float
    return lib


def load_library(path: str):
    """Load an oracle shared library (the default one or a test variant)."""
    return _declare(ctypes.CDLL(path))


def lib():
    global _lib
    if _lib is None:
        path = build()
        with _lock:
            if _lib is None:
                _lib = load_library(path)
    return _lib


class Oracle:
    """Numpy front end over one loaded oracle library."""

    def __init__(self, library=None):
        self._l = library if library is not None else lib()

    # ---- scalar IEEE helpers -------------------------------------------------
    def f16_to_double(self, bits: int) -> float:
        return self._l.orc_f16_bits_to_double(bits)

    def bf16_to_double(self, bits: int) -> float:
        return self._l.orc_bf16_bits_to_double(bits)

    def double_to_f16(self, v: float) -> int:
        return self._l.orc_double_to_f16_bits(v)

    def double_to_bf16(self, v: float) -> int:
        return self._l.orc_double_to_bf16_bits(v)

    def double_to_f32(self, v: float) -> float:
        return self._l.orc_double_to_f32(v)

    # ---- operators -----------------------------------------------------------
    def layernorm(self, dt, x, gamma=None, beta=None, eps=1e-5, wide=False):
        x = _check(dt, x)
        rows, n = x.shape
        y = np.empty_like(x)
        yw = np.empty(x.shape, np.float64) if wide else None
        mean = np.empty(rows, np.float64)
        rstd = np.empty(rows, np.float64)
        rc = self._l.orc_layernorm(dt, _ptr(x), _ptr(_check(dt, gamma, n)),
                                   _ptr(_check(dt, beta, n)), _ptr(y), _ptr(yw), _ptr(mean),
                                   _ptr(rstd), rows, n, eps)
        _rc(rc)
        return {"y": y, "y_wide": yw, "mean": mean, "rstd": rstd}

    def rmsnorm(self, dt, x, w=None, eps=1e-6, wide=False):
        x = _check(dt, x)
        rows, n = x.shape
        y = np.empty_like(x)
        yw = np.empty(x.shape, np.float64) if wide else None
        rstd = np.empty(rows, np.float64)
        rc = self._l.orc_rmsnorm(dt, _ptr(x), _ptr(_check(dt, w, n)), _ptr(y), _ptr(yw),
                                 _ptr(rstd), rows, n, eps)
        _rc(rc)
        return {"y": y, "y_wide": yw, "rstd": rstd}

    def add_rmsnorm(self, dt, x, residual, w=None, eps=1e-6, wide=False):
        x = _check(dt, x)
        residual = _check(dt, residual)
        assert residual.shape == x.shape
        rows, n = x.shape
        res_out = np.empty_like(x)
        y = np.empty_like(x)
        yw = np.empty(x.shape, np.float64) if wide else None
        rstd = np.empty(rows, np.float64)
        rc = self._l.orc_add_rmsnorm(dt, _ptr(x), _ptr(residual), _ptr(_check(dt, w, n)),
                                     _ptr(res_out), _ptr(y), _ptr(yw), _ptr(rstd), rows, n,
                                     eps)
        _rc(rc)
        return {"residual_out": res_out, "y": y, "y_wide": yw, "rstd": rstd}

    def batchnorm_train(self, dt, x, gamma=None, beta=None, running_mean=None,
                        running_var=None, eps=1e-5, momentum=0.1, wide=False):
        """x is [batch, C, HW...] (NCHW, spatial dims flattened)."""
        x = np.ascontiguousarray(x)
        batch, c = x.shape[0], x.shape[1]
        hw = int(np.prod(x.shape[2:])) if x.ndim > 2 else 1
        x = _check(dt, x.reshape(batch, c, hw))
        y = np.empty_like(x)
        yw = np.empty(x.shape, np.float64) if wide else None
        smean = np.empty(c, np.float64)
        srstd = np.empty(c, np.float64)
        rm = None if running_mean is None else np.array(running_mean, np.float64)
        rv = None if running_var is None else np.array(running_var, np.float64)
        rc = self._l.orc_batchnorm_train(dt, _ptr(x), _ptr(_check(dt, gamma, c)),
                                         _ptr(_check(dt, beta, c)), _ptr(y), _ptr(yw),
                                         _ptr(smean), _ptr(srstd), _ptr(rm), _ptr(rv),
                                         batch, c, hw, eps, momentum)
        _rc(rc)
        return {"y": y, "y_wide": yw, "save_mean": smean, "save_rstd": srstd,
                "running_mean": rm, "running_var": rv}

    def batchnorm_infer(self, dt, x, running_mean, running_var, gamma=None, beta=None,
                        eps=1e-5, wide=False):
        """x is [batch, C, HW...]; running statistics are binary32 [C]."""
        x = np.ascontiguousarray(x)
        batch, c = x.shape[0], x.shape[1]
        hw = int(np.prod(x.shape[2:])) if x.ndim > 2 else 1
        x = _check(dt, x.reshape(batch, c, hw))
        rm = np.ascontiguousarray(running_mean, np.float32)
        rv = np.ascontiguousarray(running_var, np.float32)
        assert rm.shape == (c,) and rv.shape == (c,)
        y = np.empty_like(x)
        yw = np.empty(x.shape, np.float64) if wide else None
        rc = self._l.orc_batchnorm_infer(dt, _ptr(x), _ptr(_check(dt, gamma, c)),
                                         _ptr(_check(dt, beta, c)), _ptr(y), _ptr(yw),
                                         _ptr(rm), _ptr(rv), batch, c, hw, eps)
        _rc(rc)
        return {"y": y, "y_wide": yw}

    def batchnorm_backward(self, dt, dy, x, mean, rstd, gamma=None, wide=False):
        """dy, x are [batch, C, HW...]; mean/rstd are the saved per-channel
        statistics (any float array of shape [C], widened to double)."""
        x = np.ascontiguousarray(x)
        batch, c = x.shape[0], x.shape[1]
        hw = int(np.prod(x.shape[2:])) if x.ndim > 2 else 1
        x = _check(dt, x.reshape(batch, c, hw))
        dy = _check(dt, np.ascontiguousarray(dy).reshape(batch, c, hw))
        mean = np.ascontiguousarray(mean, np.float64)
        rstd = np.ascontiguousarray(rstd, np.float64)
        assert mean.shape == (c,) and rstd.shape == (c,)
        dx = np.empty_like(x)
        dxw = np.empty(x.shape, np.float64) if wide else None
        dg = np.empty(c, np.float64)
        db = np.empty(c, np.float64)
        rc = self._l.orc_batchnorm_backward(dt, _ptr(dy), _ptr(x), _ptr(_check(dt, gamma, c)),
                                            _ptr(mean), _ptr(rstd), _ptr(dx), _ptr(dxw),
                                            _ptr(dg), _ptr(db), batch, c, hw)
        _rc(rc)
        return {"dx": dx, "dx_wide": dxw, "dgamma": dg, "dbeta": db}

    def softmax(self, dt, x, wide=False):
        x = _check(dt, x)
        rows, n = x.shape
        y = np.empty_like(x)
        yw = np.empty(x.shape, np.float64) if wide else None
        m = np.empty(rows, np.float64)
        d = np.empty(rows, np.float64)
        rc = self._l.orc_softmax(dt, _ptr(x), _ptr(y), _ptr(yw), _ptr(m), _ptr(d), rows, n)
        _rc(rc)
        return {"y": y, "y_wide": yw, "row_max": m, "row_sum": d}


def _check(dt, a, n=None):
    if a is None:
        return None
    want = np.float32 if dt == F32 else np.uint16
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"dtype code {dt} wants numpy {np.dtype(want).name}, got {a.dtype}")
    if n is not None and a.shape != (n,):
        raise ValueError(f"parameter shape {a.shape} != ({n},)")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rc(rc):
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
