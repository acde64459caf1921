"""ctypes binding of libnorm's C ABI (include/libnorm.h).

Argument marshalling only: every function takes torch tensors (device memory
allocated by the caller), derives the sizes and the dtype code from them, and
calls the C entry point of the same name on the current torch CUDA stream (or
the stream given).  Every step of the computation runs in libnorm's kernels.
A non-OK status raises NrmError.  There is no fallback: if libnorm.so is not
built the first call raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libnorm.so")

NRM_OK, NRM_ERR_INVALID_ARG, NRM_ERR_UNSUPPORTED, NRM_ERR_WORKSPACE, NRM_ERR_CUDA, NRM_ERR_TIMEOUT = range(6)
NRM_F32, NRM_F16, NRM_BF16 = 0, 1, 2
NRM_ACT_NONE, NRM_ACT_RELU, NRM_ACT_GELU, NRM_ACT_SILU, NRM_ACT_MISH = 0, 1, 2, 3, 4
NRM_ACT_LEAKY_RELU, NRM_ACT_ELU, NRM_ACT_SIGMOID, NRM_ACT_CELU, NRM_ACT_SELU = 5, 6, 7, 8, 9
NRM_ACT_RELU6, NRM_ACT_HARDTANH = 10, 11
NRM_OP_LAYERNORM_BWD, NRM_OP_RMSNORM_BWD, NRM_OP_LAYERNORM_CF_BWD = 1, 2, 3

ACTS = {"none": NRM_ACT_NONE, "relu": NRM_ACT_RELU, "gelu": NRM_ACT_GELU, "silu": NRM_ACT_SILU,
        "mish": NRM_ACT_MISH, "leaky_relu": NRM_ACT_LEAKY_RELU, "elu": NRM_ACT_ELU,
        "sigmoid": NRM_ACT_SIGMOID, "celu": NRM_ACT_CELU, "selu": NRM_ACT_SELU,
        "relu6": NRM_ACT_RELU6, "hardtanh": NRM_ACT_HARDTANH}

# Every symbol the header declares (checked by the CPU tests).
EXPORTS = ("nrm_layernorm_fwd", "nrm_layernorm_bwd", "nrm_layernorm_bwd_noalloc",
           "nrm_layernorm_cf_fwd", "nrm_layernorm_cf_bwd",
           "nrm_rmsnorm_fwd", "nrm_rmsnorm_bwd", "nrm_layernorm_fwd_ex", "nrm_layernorm_bwd_ex",
           "nrm_rmsnorm_fwd_ex", "nrm_rmsnorm_bwd_ex",
           "nrm_batchnorm_fwd", "nrm_batchnorm_bwd", "nrm_act_dropout_fwd", "nrm_act_dropout_bwd",
           "nrm_workspace_bytes",
           "nrm_batchnorm_workspace_bytes",
           "nrm_act_mask_words", "nrm_sync_status", "nrm_status_str",
           "nrm_last_error_message", "nrm_version", "nrm_test_expire_peer_waits")


class NrmError(RuntimeError):
    def __init__(self, status: int, func: str, message: str):
        self.status = status
        super().__init__(f"{func}: status {status}: {message}")


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_I = ctypes.c_int
_lib = None


def load(path: str | None = None):
    """Loads libnorm.so (once) and declares the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libnorm is not built ({p} is missing); run "
                          "`python -m normalization_layernorm_rmsnorm_gb300.build`")
    lib = ctypes.CDLL(p)
    sig = {
        "nrm_layernorm_fwd": [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _P],
        "nrm_layernorm_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _P, ctypes.c_size_t, _P],
        "nrm_layernorm_bwd_noalloc": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _P],
        "nrm_layernorm_cf_fwd": [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _I, _P],
        "nrm_layernorm_cf_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _P, ctypes.c_size_t,
                                 _P],
        "nrm_rmsnorm_fwd": [_P, _P, _P, _P, _P, _I64, _I64, _F, _I, _P],
        "nrm_layernorm_fwd_ex": [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P],
        "nrm_layernorm_bwd_ex": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _I, _P, ctypes.c_size_t, _P],
        "nrm_rmsnorm_fwd_ex": [_P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P],
        "nrm_rmsnorm_bwd_ex": [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _I, _P, ctypes.c_size_t, _P],
        "nrm_rmsnorm_bwd": [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I, _P, ctypes.c_size_t, _P],
        "nrm_batchnorm_fwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, _I,
                              _I, _F, _I, _P, ctypes.c_size_t, _P],
        "nrm_batchnorm_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I,
                              _I, _F, _I, _P, ctypes.c_size_t, _P],
        "nrm_act_dropout_fwd": [_P, _P, _I64, _I, _F, _F, ctypes.c_uint32, _I, _P],
        "nrm_act_dropout_bwd": [_P, _P, _P, _I64, _I, _F, _F, ctypes.c_uint32, _I, _P],
        "nrm_workspace_bytes": [_I, _I64, _I64, _I],
        "nrm_batchnorm_workspace_bytes": [_I64, _I64, _I64, _I],
        "nrm_act_mask_words": [_I64, _I64, _I64],
        "nrm_sync_status": [_P],
        "nrm_status_str": [_I],
        "nrm_last_error_message": [],
        "nrm_version": [],
        "nrm_test_expire_peer_waits": [ctypes.c_uint64],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = _I
    lib.nrm_workspace_bytes.restype = ctypes.c_size_t
    lib.nrm_batchnorm_workspace_bytes.restype = ctypes.c_size_t
    lib.nrm_act_mask_words.restype = ctypes.c_int64
    lib.nrm_status_str.restype = ctypes.c_char_p
    lib.nrm_last_error_message.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: NRM_F32, torch.float16: NRM_F16, torch.bfloat16: NRM_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, func: str):
    if status != NRM_OK:
        msg = load().nrm_last_error_message().decode()
        raise NrmError(status, func, msg)


def _act(act) -> int:
    return ACTS[act] if isinstance(act, str) else int(act)


def _rows_cols(x):
    cols = x.shape[-1] if x.dim() > 0 else 1
    rows = x.numel() // cols if cols else 0
    return rows, cols


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def nrm_layernorm_fwd(x, w, b, y, mean, rstd, eps, stream=None):
    rows, cols = _rows_cols(x)
    _check(load().nrm_layernorm_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(mean), _ptr(rstd),
                                    rows, cols, eps, _dtype_code(x), _stream(stream)),
           "nrm_layernorm_fwd")


def nrm_layernorm_bwd(dy, x, w, mean, rstd, dx, dw, db, workspace, stream=None):
    rows, cols = _rows_cols(x)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().nrm_layernorm_bwd(_ptr(dy), _ptr(x), _ptr(w), _ptr(mean), _ptr(rstd), _ptr(dx),
                                    _ptr(dw), _ptr(db), rows, cols, _dtype_code(x), _ptr(workspace),
                                    ws_bytes, _stream(stream)),
           "nrm_layernorm_bwd")


def nrm_layernorm_cf_fwd(x, w, b, y, mean, rstd, eps, stream=None):
    """LayerNorm over the channels of x[n, c, *spatial]; mean, rstd hold n * prod(spatial)
    floats (or are None)."""
    n, c, l = _ncl(x)
    _check(load().nrm_layernorm_cf_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(mean), _ptr(rstd),
                                       n, c, l, eps, _dtype_code(x), _stream(stream)),
           "nrm_layernorm_cf_fwd")


def nrm_layernorm_cf_bwd(dy, x, w, mean, rstd, dx, dw, db, workspace, stream=None):
    n, c, l = _ncl(x)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().nrm_layernorm_cf_bwd(_ptr(dy), _ptr(x), _ptr(w), _ptr(mean), _ptr(rstd), _ptr(dx),
                                       _ptr(dw), _ptr(db), n, c, l, _dtype_code(x), _ptr(workspace),
                                       ws_bytes, _stream(stream)),
           "nrm_layernorm_cf_bwd")


def nrm_layernorm_bwd_noalloc(dy, x, w, mean, rstd, dx, dw, db, stream=None):
    """LayerNorm backward for callers that cannot allocate: no workspace; the
    library's static device scratch holds the dw/db partial rows."""
    rows, cols = _rows_cols(x)
    _check(load().nrm_layernorm_bwd_noalloc(_ptr(dy), _ptr(x), _ptr(w), _ptr(mean), _ptr(rstd),
                                            _ptr(dx), _ptr(dw), _ptr(db), rows, cols,
                                            _dtype_code(x), _stream(stream)),
           "nrm_layernorm_bwd_noalloc")


def nrm_rmsnorm_fwd(x, w, y, rstd, eps, stream=None, b=None):
    """RMSNorm of the rows of x; b is the optional bias."""
    rows, cols = _rows_cols(x)
    _check(load().nrm_rmsnorm_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(rstd), rows, cols, eps,
                                  _dtype_code(x), _stream(stream)),
           "nrm_rmsnorm_fwd")


def nrm_layernorm_fwd_ex(x, w, b, y, mean, rstd, eps, stream=None):
    """LayerNorm with y in its own dtype (x's, or float32 for a 16-bit x)."""
    rows, cols = _rows_cols(x)
    _check(load().nrm_layernorm_fwd_ex(_ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(mean), _ptr(rstd), rows,
                                       cols, eps, _dtype_code(x), _dtype_code(y), _stream(stream)),
           "nrm_layernorm_fwd_ex")


def nrm_layernorm_bwd_ex(dy, x, w, mean, rstd, dx, dw, db, workspace, stream=None):
    """LayerNorm backward with dy in its own dtype (the forward's y dtype)."""
    rows, cols = _rows_cols(x)
    _check(load().nrm_layernorm_bwd_ex(_ptr(dy), _ptr(x), _ptr(w), _ptr(mean), _ptr(rstd), _ptr(dx),
                                       _ptr(dw), _ptr(db), rows, cols, _dtype_code(x), _dtype_code(dy),
                                       _ptr(workspace), _ws(workspace), _stream(stream)),
           "nrm_layernorm_bwd_ex")


def nrm_rmsnorm_fwd_ex(x, w, y, rstd, eps, stream=None, b=None):
    """RMSNorm with y in its own dtype (x's, or float32 for a 16-bit x)."""
    rows, cols = _rows_cols(x)
    _check(load().nrm_rmsnorm_fwd_ex(_ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(rstd), rows, cols, eps,
                                     _dtype_code(x), _dtype_code(y), _stream(stream)),
           "nrm_rmsnorm_fwd_ex")


def nrm_rmsnorm_bwd_ex(dy, x, w, rstd, dx, dw, workspace, stream=None, db=None):
    """RMSNorm backward with dy in its own dtype (the forward's y dtype)."""
    rows, cols = _rows_cols(x)
    _check(load().nrm_rmsnorm_bwd_ex(_ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw), _ptr(db),
                                     rows, cols, _dtype_code(x), _dtype_code(dy), _ptr(workspace),
                                     _ws(workspace), _stream(stream)),
           "nrm_rmsnorm_bwd_ex")


def nrm_rmsnorm_bwd(dy, x, w, rstd, dx, dw, workspace, stream=None, db=None):
    """RMSNorm backward; db receives the bias gradient when given."""
    rows, cols = _rows_cols(x)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().nrm_rmsnorm_bwd(_ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw), _ptr(db),
                                  rows, cols, _dtype_code(x), _ptr(workspace), ws_bytes,
                                  _stream(stream)),
           "nrm_rmsnorm_bwd")


def _ncl(x):
    if x.dim() < 2:
        raise ValueError("input needs at least [n, c] (NCHW-like, channels second)")
    n, c = x.shape[0], x.shape[1]
    l = 1
    for s in x.shape[2:]:
        l *= s
    return n, c, l


def _ws(workspace):
    return 0 if workspace is None else workspace.numel() * workspace.element_size()


def nrm_batchnorm_fwd(x, residual, w, b, y, running_mean, running_var, save_mean, save_rstd,
                      act_mask, eps, momentum, training, act, workspace, stream=None, act_param=0.0):
    n, c, l = _ncl(x)
    _check(load().nrm_batchnorm_fwd(_ptr(x), _ptr(residual), _ptr(w), _ptr(b), _ptr(y),
                                    _ptr(running_mean), _ptr(running_var), _ptr(save_mean),
                                    _ptr(save_rstd), _ptr(act_mask), n, c, l, eps, momentum,
                                    int(bool(training)), _act(act), float(act_param), _dtype_code(x),
                                    _ptr(workspace), _ws(workspace), _stream(stream)),
           "nrm_batchnorm_fwd")


def nrm_batchnorm_bwd(dy, x, residual, w, b, save_mean, save_rstd, act_mask, dx, dres, dw, db,
                      training, act, workspace, stream=None, act_param=0.0):
    n, c, l = _ncl(x)
    _check(load().nrm_batchnorm_bwd(_ptr(dy), _ptr(x), _ptr(residual), _ptr(w), _ptr(b),
                                    _ptr(save_mean), _ptr(save_rstd), _ptr(act_mask), _ptr(dx),
                                    _ptr(dres), _ptr(dw), _ptr(db), n, c, l,
                                    int(bool(training)), _act(act), float(act_param), _dtype_code(x),
                                    _ptr(workspace), _ws(workspace), _stream(stream)),
           "nrm_batchnorm_bwd")


def nrm_batchnorm_workspace_bytes(n: int, c: int, l: int, dtype_code: int) -> int:
    return int(load().nrm_batchnorm_workspace_bytes(n, c, l, dtype_code))


def batchnorm_workspace(x):
    """A device workspace large enough for BatchNorm calls on x ([n, c, ...])."""
    import torch
    n, c, l = _ncl(x)
    nbytes = nrm_batchnorm_workspace_bytes(n, c, l, _dtype_code(x))
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)


def nrm_workspace_bytes(op: int, rows: int, cols: int, dtype_code: int) -> int:
    return int(load().nrm_workspace_bytes(op, rows, cols, dtype_code))


def nrm_act_dropout_fwd(x, y, act, drop_p, seed, stream=None, act_param=0.0):
    """y = act(x) / (1 - drop_p) where kept, else 0 (mask rebuilt from seed and offset)."""
    _check(load().nrm_act_dropout_fwd(_ptr(x), _ptr(y), x.numel(), _act(act), float(act_param), float(drop_p),
                                      int(seed) & 0xFFFFFFFF, _dtype_code(x), _stream(stream)),
           "nrm_act_dropout_fwd")


def nrm_act_dropout_bwd(dy, x, dx, act, drop_p, seed, stream=None, act_param=0.0):
    """dx = dy / (1 - drop_p) * act'(x) where kept, else 0."""
    _check(load().nrm_act_dropout_bwd(_ptr(dy), _ptr(x), _ptr(dx), x.numel(), _act(act), float(act_param),
                                      float(drop_p),
                                      int(seed) & 0xFFFFFFFF, _dtype_code(x), _stream(stream)),
           "nrm_act_dropout_bwd")


def nrm_act_mask_words(n: int, c: int, l: int) -> int:
    return int(load().nrm_act_mask_words(n, c, l))


def nrm_sync_status(stream=None):
    _check(load().nrm_sync_status(_stream(stream)), "nrm_sync_status")


def nrm_status_str(status: int) -> str:
    return load().nrm_status_str(status).decode()


def nrm_version() -> int:
    return int(load().nrm_version())


def nrm_last_error_message() -> str:
    return load().nrm_last_error_message().decode()


def nrm_test_expire_peer_waits(limit_ns: int):
    """Test hook: the next training BatchNorm call on this thread whose kernel
    waits for the other CTAs of a channel waits for one CTA too many and gives
    up after limit_ns (its outputs are then undefined; nrm_sync_status reports
    NRM_ERR_TIMEOUT)."""
    _check(load().nrm_test_expire_peer_waits(int(limit_ns)), "nrm_test_expire_peer_waits")
