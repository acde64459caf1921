"""Double-precision CPU oracle for LayerNorm, RMSNorm and BatchNorm, and for the
activation with fused dropout.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library and
its Python binding never touch it, and it shares no code with them.

The arithmetic lives in ``norm_oracle.c`` (plain loops in double, written from
the attorch normalization articles; see that file's header for the sources and
the readings taken).  This module compiles it with gcc into ``_build/`` and
exposes numpy-friendly wrappers.  All arrays are float64 and C-contiguous;
masks are uint32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "norm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "liboracle.so")

ACT_NONE, ACT_RELU, ACT_GELU, ACT_SILU, ACT_MISH, ACT_LEAKY_RELU, ACT_ELU = 0, 1, 2, 3, 4, 5, 6
ACT_SIGMOID, ACT_CELU, ACT_SELU, ACT_RELU6, ACT_HARDTANH = 7, 8, 9, 10, 11

# -ffp-contract=off keeps a*b+c as two roundings on every host (gcc fuses them by
# default on aarch64), so the oracle gives the same bits here and on the GPU machine.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-D_DEFAULT_SOURCE"]

_lock = threading.Lock()


def build(src: str = _SRC, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc; return ``out``."""
    with _lock:
        if (not force and os.path.exists(out)
                and os.path.getmtime(out) >= os.path.getmtime(src)
                and os.path.getmtime(out) >= os.path.getmtime(
                    os.path.join(_HERE, "norm_oracle.h"))):
            return out
        os.makedirs(os.path.dirname(out), exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-I", _HERE, src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
        return out


_D = ctypes.POINTER(ctypes.c_double)
_U32 = ctypes.POINTER(ctypes.c_uint32)
_I64 = ctypes.c_int64


def _ptr(a, kind=_D):
    if a is None:
        return None
    return a.ctypes.data_as(kind)


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a copy
    built from a modified source by the mutation tests)."""

    def __init__(self, lib_path: str | None = None):
        self.lib_path = lib_path or build()
        lib = ctypes.CDLL(self.lib_path)
        lib.oracle_layernorm_fwd.argtypes = [_I64, _I64, _D, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_layernorm_bwd.argtypes = [_I64, _I64, _D, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_layernorm_cf_fwd.argtypes = [_I64, _I64, _I64, _D, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_layernorm_cf_bwd.argtypes = [_I64, _I64, _I64, _D, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_rmsnorm_fwd.argtypes = [_I64, _I64, _D, _D, _D, ctypes.c_double, _D, _D]
        lib.oracle_rmsnorm_bwd.argtypes = [_I64, _I64, _D, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_batchnorm_fwd.argtypes = [_I64, _I64, _I64, _D, _D, _D, _D,
                                             ctypes.c_double, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_double, _D, _D,
                                             _D, _D, _D, _U32, _D]
        lib.oracle_batchnorm_bwd.argtypes = [_I64, _I64, _I64, _D, _D, _D, _D, _D,
                                             _D, _D, ctypes.c_double, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, _U32, _D, _D, _D, _D]
        _U8 = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_philox4x32_10.argtypes = [_U32, _U32, _U32]
        lib.oracle_dropout_mask.argtypes = [_I64, _I64, ctypes.c_double, ctypes.c_uint32, _U8]
        lib.oracle_act_dropout_fwd.argtypes = [_I64, _I64, _D, ctypes.c_int, ctypes.c_double,
                                               ctypes.c_double, ctypes.c_uint32, _D]
        lib.oracle_act_dropout_bwd.argtypes = [_I64, _I64, _D, _D, ctypes.c_int, ctypes.c_double,
                                               ctypes.c_double, ctypes.c_uint32, _D]
        for f in ("oracle_layernorm_fwd", "oracle_layernorm_bwd", "oracle_layernorm_cf_fwd",
                  "oracle_layernorm_cf_bwd", "oracle_rmsnorm_fwd",
                  "oracle_rmsnorm_bwd", "oracle_batchnorm_fwd", "oracle_batchnorm_bwd",
                  "oracle_philox4x32_10", "oracle_dropout_mask", "oracle_act_dropout_fwd",
                  "oracle_act_dropout_bwd"):
            getattr(lib, f).restype = None
        self.lib = lib

    # -- row norms ---------------------------------------------------------
    def layernorm_fwd(self, x, w=None, b=None, eps=1e-5):
        """Returns (y, mean, rstd) for x of shape [rows, cols]."""
        x = _f64(x)
        rows, cols = x.shape
        w, b = _f64(w), _f64(b)
        y = np.empty_like(x)
        mean = np.empty(rows)
        rstd = np.empty(rows)
        self.lib.oracle_layernorm_fwd(rows, cols, _ptr(x), _ptr(w), _ptr(b), eps,
                                      _ptr(y), _ptr(mean), _ptr(rstd))
        return y, mean, rstd

    def layernorm_bwd(self, dy, x, w=None, eps=1e-5):
        """Returns (dx, dw, db)."""
        dy, x, w = _f64(dy), _f64(x), _f64(w)
        rows, cols = x.shape
        dx = np.empty_like(x)
        dw = np.empty(cols)
        db = np.empty(cols)
        self.lib.oracle_layernorm_bwd(rows, cols, _ptr(dy), _ptr(x), _ptr(w), eps,
                                      _ptr(dx), _ptr(dw), _ptr(db))
        return dx, dw, db

    def layernorm_cf_fwd(self, x, w=None, b=None, eps=1e-6):
        """Channels-first LayerNorm: x of shape [n, c, l]; returns (y, mean, rstd),
        mean and rstd of shape [n, l]."""
        x = _f64(x)
        n, c, l = x.shape
        w, b = _f64(w), _f64(b)
        y = np.empty_like(x)
        mean = np.empty((n, l))
        rstd = np.empty((n, l))
        self.lib.oracle_layernorm_cf_fwd(n, c, l, _ptr(x), _ptr(w), _ptr(b), eps, _ptr(y),
                                         _ptr(mean), _ptr(rstd))
        return y, mean, rstd

    def layernorm_cf_bwd(self, dy, x, w=None, eps=1e-6):
        """Returns (dx, dw, db) of the channels-first LayerNorm."""
        dy, x, w = _f64(dy), _f64(x), _f64(w)
        n, c, l = x.shape
        dx = np.empty_like(x)
        dw = np.empty(c)
        db = np.empty(c)
        self.lib.oracle_layernorm_cf_bwd(n, c, l, _ptr(dy), _ptr(x), _ptr(w), eps, _ptr(dx),
                                         _ptr(dw), _ptr(db))
        return dx, dw, db

    def rmsnorm_fwd(self, x, w=None, eps=1e-6, b=None):
        """Returns (y, rstd); b is the optional bias."""
        x, w, b = _f64(x), _f64(w), _f64(b)
        rows, cols = x.shape
        y = np.empty_like(x)
        rstd = np.empty(rows)
        self.lib.oracle_rmsnorm_fwd(rows, cols, _ptr(x), _ptr(w), _ptr(b), eps, _ptr(y), _ptr(rstd))
        return y, rstd

    def rmsnorm_bwd(self, dy, x, w=None, eps=1e-6, with_db=False):
        """Returns (dx, dw), or (dx, dw, db) with with_db (the bias gradient)."""
        dy, x, w = _f64(dy), _f64(x), _f64(w)
        rows, cols = x.shape
        dx = np.empty_like(x)
        dw = np.empty(cols)
        db = np.empty(cols) if with_db else None
        self.lib.oracle_rmsnorm_bwd(rows, cols, _ptr(dy), _ptr(x), _ptr(w), eps,
                                    _ptr(dx), _ptr(dw), _ptr(db))
        return (dx, dw, db) if with_db else (dx, dw)

    # -- BatchNorm -----------------------------------------------------------
    @staticmethod
    def mask_words(n, c, l):
        return n * c * ((l + 31) // 32)

    def batchnorm_fwd(self, x, res=None, w=None, b=None, eps=1e-5, momentum=0.1,
                      training=True, act=ACT_NONE, running_mean=None,
                      running_var=None, want_mask=False, want_z=False, act_param=0.0):
        """x: [n, c, l].  Returns a dict with y, save_mean, save_rstd,
        running_mean, running_var (updated copies, or None), mask (uint32 or
        None) and z (pre-activation, or None)."""
        x = _f64(x)
        n, c, l = x.shape
        res, w, b = _f64(res), _f64(w), _f64(b)
        rm = None if running_mean is None else np.array(running_mean, dtype=np.float64)
        rv = None if running_var is None else np.array(running_var, dtype=np.float64)
        y = np.empty_like(x)
        sm = np.empty(c)
        sr = np.empty(c)
        mask = np.zeros(self.mask_words(n, c, l), dtype=np.uint32) if want_mask else None
        z = np.empty_like(x) if want_z else None
        self.lib.oracle_batchnorm_fwd(n, c, l, _ptr(x), _ptr(res), _ptr(w), _ptr(b),
                                      eps, momentum, int(bool(training)), int(act), float(act_param),
                                      _ptr(rm), _ptr(rv), _ptr(y), _ptr(sm), _ptr(sr),
                                      _ptr(mask, _U32), _ptr(z))
        return dict(y=y, save_mean=sm, save_rstd=sr, running_mean=rm,
                    running_var=rv, mask=mask, z=z)

    def batchnorm_bwd(self, dy, x, res=None, w=None, b=None, running_mean=None,
                      running_var=None, eps=1e-5, training=True, act=ACT_NONE,
                      mask=None, act_param=0.0):
        """Returns (dx, dres, dw, db)."""
        dy, x = _f64(dy), _f64(x)
        n, c, l = x.shape
        res, w, b = _f64(res), _f64(w), _f64(b)
        rm, rv = _f64(running_mean), _f64(running_var)
        mask = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint32)
        dx = np.empty_like(x)
        dres = np.empty_like(x)
        dw = np.empty(c)
        db = np.empty(c)
        self.lib.oracle_batchnorm_bwd(n, c, l, _ptr(dy), _ptr(x), _ptr(res), _ptr(w),
                                      _ptr(b), _ptr(rm), _ptr(rv), eps,
                                      int(bool(training)), int(act), float(act_param), _ptr(mask, _U32),
                                      _ptr(dx), _ptr(dres), _ptr(dw), _ptr(db))
        return dx, dres, dw, db


    # -- activation with fused dropout ---------------------------------------
    def philox4x32_10(self, ctr, key):
        """The four 32-bit output words of Philox4x32-10 for a counter of four
        words and a key of two."""
        c = np.ascontiguousarray(ctr, dtype=np.uint32)
        k = np.ascontiguousarray(key, dtype=np.uint32)
        out = np.empty(4, dtype=np.uint32)
        self.lib.oracle_philox4x32_10(_ptr(c, _U32), _ptr(k, _U32), _ptr(out, _U32))
        return out

    def dropout_mask(self, count, drop_p, seed, first=0):
        """uint8 keep flags of elements first .. first+count-1."""
        keep = np.empty(int(count), dtype=np.uint8)
        self.lib.oracle_dropout_mask(int(count), int(first), float(drop_p), int(seed) & 0xFFFFFFFF,
                                     keep.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
        return keep

    def act_dropout_fwd(self, x, act, drop_p, seed, first=0, act_param=0.0):
        """y = act(x) / (1 - p) where kept, 0 where dropped; x (flattened) holds
        the tensor's elements first, first+1, ..."""
        x = _f64(x)
        y = np.empty_like(x)
        self.lib.oracle_act_dropout_fwd(x.size, int(first), _ptr(x), int(act), float(act_param),
                                        float(drop_p),
                                        int(seed) & 0xFFFFFFFF, _ptr(y))
        return y

    def act_dropout_bwd(self, dy, x, act, drop_p, seed, first=0, act_param=0.0):
        """dx = dy / (1 - p) * act'(x) where kept, 0 where dropped."""
        dy, x = _f64(dy), _f64(x)
        dx = np.empty_like(x)
        self.lib.oracle_act_dropout_bwd(x.size, int(first), _ptr(dy), _ptr(x), int(act),
                                        float(act_param), float(drop_p),
                                        int(seed) & 0xFFFFFFFF, _ptr(dx))
        return dx


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from the committed source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
