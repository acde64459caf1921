"""Seeded synthetic inputs for the normalization workloads.

This module is the one piece shared by the CUDA path's tests and bench and by
the CPU oracle's tests: it only draws random numbers and rounds them to the
storage dtype.  It holds none of the normalization arithmetic.

Generator: counter-based.  Each tensor has a 64-bit key derived from
(seed, stream id) with the splitmix64 finaliser; element i's uniform is the
finaliser applied to key + (i+1)*0x9E3779B97F4A7C15, top 53 bits, shifted by
half an ulp so it lies in (0, 1).  Normals use the Box-Muller cosine branch on
uniforms 2i and 2i+1 of the tensor's stream.  Values are formed in float64,
rounded to float32, then rounded to nearest-even into fp16 or bf16 where the
workload stores that dtype.  The oracle consumes exactly the rounded values.

Workloads (the shapes of the models the articles use: LLaMA-style RMSNorm,
ViT LayerNorm, ResNet BatchNorm+ReLU) are in ``CONFIGS``.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_CHUNK = 1 << 20
_POOL = None


def _pool():
    """Thread pool for chunked generation (numpy ufuncs release the GIL)."""
    global _POOL
    if _POOL is None:
        _POOL = concurrent.futures.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _chunked(count: int, fn) -> None:
    list(_pool().map(lambda lo: fn(lo, min(count, lo + _CHUNK)), range(0, count, _CHUNK)))


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array, in place (wrapping arithmetic)."""
    t = np.empty_like(z)
    np.right_shift(z, np.uint64(30), out=t)
    np.bitwise_xor(z, t, out=z)
    np.multiply(z, np.uint64(0xBF58476D1CE4E5B9), out=z)
    np.right_shift(z, np.uint64(27), out=t)
    np.bitwise_xor(z, t, out=z)
    np.multiply(z, np.uint64(0x94D049BB133111EB), out=z)
    np.right_shift(z, np.uint64(31), out=t)
    np.bitwise_xor(z, t, out=z)
    return z


def _mix_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return _mix_int(_mix_int(seed * _GOLDEN + 0x632BE59BD9B4E019) + stream * _GOLDEN)


def _uniform_into(out: np.ndarray, key: np.uint64, start: int, stride: int) -> None:
    """out[k] = uniform number (start + k*stride) of the stream with ``key``."""
    count = out.shape[0]
    ctr = np.arange(count, dtype=np.uint64)
    np.multiply(ctr, np.uint64(stride), out=ctr)
    np.add(ctr, np.uint64(start + 1), out=ctr)
    np.multiply(ctr, np.uint64(_GOLDEN), out=ctr)
    np.add(ctr, key, out=ctr)
    _mix(ctr)
    np.right_shift(ctr, np.uint64(11), out=ctr)
    np.copyto(out, ctr, casting="unsafe")
    out += 0.5
    out *= 2.0 ** -53


def uniform(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Uniforms in (0, 1), float64, elements [start, start+count) of a stream."""
    key = np.uint64(stream_key(seed, stream))
    out = np.empty(count, dtype=np.float64)

    def chunk(lo, hi):
        with np.errstate(over="ignore"):
            _uniform_into(out[lo:hi], key, start + lo, 1)
    _chunked(count, chunk)
    return out


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """Standard normals, float64 (Box-Muller, cosine branch on uniforms 2i, 2i+1)."""
    key = np.uint64(stream_key(seed, stream))
    out = np.empty(count, dtype=np.float64)

    def chunk(lo, hi):
        o = out[lo:hi]
        v = np.empty(hi - lo, dtype=np.float64)
        with np.errstate(over="ignore"):
            _uniform_into(o, key, 2 * lo, 2)
            _uniform_into(v, key, 2 * lo + 1, 2)
        np.log(o, out=o)
        o *= -2.0
        np.sqrt(o, out=o)
        v *= 2.0 * math.pi
        np.cos(v, out=v)
        o *= v
    _chunked(count, chunk)
    return out


# ---------------------------------------------------------------------------
# storage dtypes
# ---------------------------------------------------------------------------

DTYPES = ("f32", "f16", "bf16")


def round_bf16_bits(a32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    bits = np.ascontiguousarray(a32, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return ((bits + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(b16: np.ndarray) -> np.ndarray:
    return (b16.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclasses.dataclass
class Tensor:
    """A host tensor in its storage dtype.  ``data`` is float32, float16, or
    uint16 holding bf16 bit patterns."""
    data: np.ndarray
    dtype: str

    @property
    def shape(self):
        return self.data.shape

    @property
    def nbytes(self):
        return self.data.nbytes

    def f64(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f64(self.data)
        return self.data.astype(np.float64)

    def torch(self, device="cpu"):
        import torch
        t = torch.from_numpy(np.ascontiguousarray(self.data))
        if self.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.to(device)


def store(values: np.ndarray, dtype: str, shape) -> Tensor:
    """Round float64 values to float32, then to the storage dtype."""
    src = np.ascontiguousarray(values, dtype=np.float64).reshape(-1)
    count = src.shape[0]
    np_dt = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]
    out = np.empty(count, dtype=np_dt)

    def chunk(lo, hi):
        a32 = src[lo:hi].astype(np.float32)
        if dtype == "f32":
            out[lo:hi] = a32
        elif dtype == "f16":
            out[lo:hi] = a32.astype(np.float16)
        else:
            out[lo:hi] = round_bf16_bits(a32)
    _chunked(count, chunk)
    return Tensor(out.reshape(shape), dtype)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

# stream ids, one per tensor role
S_X, S_W, S_B, S_DY, S_RES, S_OFF, S_SCALE = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class RowConfig:
    name: str
    kind: str            # "layernorm" | "rmsnorm"
    rows: int
    cols: int
    dtype: str
    eps: float
    seed: int
    x_mean: float = 0.0
    x_std: float = 1.0
    w_std: float = 0.1   # weight = 1 + w_std * N(0,1)
    b_std: float = 0.1   # bias = b_std * N(0,1) (LayerNorm only)
    outlier_cols: tuple = ()
    outlier_scale: float = 1.0
    affine: bool = True


@dataclasses.dataclass(frozen=True)
class BnConfig:
    name: str
    n: int
    c: int
    l: int
    dtype: str
    eps: float
    momentum: float
    seed: int
    act: str             # "none" | "relu" | "gelu"
    residual: bool
    x_kind: str          # "offset_scale": off_c + scale_c*N ; "scale": N*s_c
    off_range: tuple = (-1.0, 1.0)
    scale_range: tuple = (0.5, 2.0)
    w_std: float = 0.0   # weight = 1 + w_std*N(0,1); 0 gives weight = 1
    b_std: float = 0.0   # bias = b_std*N(0,1); 0 gives bias = 0
    training: bool = True


CONFIGS = {
    "ln_f32_64x256": RowConfig("ln_f32_64x256", "layernorm", 64, 256, "f32", 1e-5, 0),
    "rms_bf16_16384x4096": RowConfig(
        "rms_bf16_16384x4096", "rmsnorm", 16384, 4096, "bf16", 1e-6, 1,
        w_std=0.02, outlier_cols=tuple(7 + 512 * k for k in range(8)), outlier_scale=20.0),
    "ln_f16_25216x768": RowConfig(
        "ln_f16_25216x768", "layernorm", 25216, 768, "f16", 1e-6, 2, x_mean=0.3, x_std=1.5),
    "bn_f32_256x64x56x56_res_relu": BnConfig(
        "bn_f32_256x64x56x56_res_relu", 256, 64, 56 * 56, "f32", 1e-5, 0.1, 3,
        act="relu", residual=True, x_kind="offset_scale"),
    "bn_f16_128x512x7x7_gelu": BnConfig(
        "bn_f16_128x512x7x7_gelu", 128, 512, 7 * 7, "f16", 1e-5, 0.1, 4,
        act="gelu", residual=False, x_kind="scale", scale_range=(0.5, 3.0),
        w_std=0.1, b_std=0.1),
}

# The small case the oracle finishes in milliseconds, then the four full-size
# workloads in the order they are quoted.
SMALL = "ln_f32_64x256"
FULL = ("rms_bf16_16384x4096", "ln_f16_25216x768",
        "bn_f32_256x64x56x56_res_relu", "bn_f16_128x512x7x7_gelu")


def row_inputs(cfg: RowConfig, rows: int | None = None):
    """x, w, b (LayerNorm only), dy for a row-norm workload.  ``rows`` takes the
    first rows of the same streams (a bounded sample of the workload)."""
    rows = cfg.rows if rows is None else rows
    R, N = rows, cfg.cols
    x = normal(cfg.seed, S_X, R * N).reshape(R, N) * cfg.x_std + cfg.x_mean
    if cfg.outlier_cols:
        x[:, list(cfg.outlier_cols)] *= cfg.outlier_scale
    out = {"x": store(x, cfg.dtype, (R, N))}
    if cfg.affine:
        out["w"] = store(1.0 + cfg.w_std * normal(cfg.seed, S_W, N), cfg.dtype, (N,))
        if cfg.kind == "layernorm":
            out["b"] = store(cfg.b_std * normal(cfg.seed, S_B, N), cfg.dtype, (N,))
    out["dy"] = store(normal(cfg.seed, S_DY, R * N), cfg.dtype, (R, N))
    return out


def bn_inputs(cfg: BnConfig, channels: int | None = None):
    """x, residual, w, b, dy, running_mean, running_var for a BatchNorm workload.
    ``channels`` keeps the first channels (a bounded sample of the workload)."""
    C = cfg.c if channels is None else channels
    n, l = cfg.n, cfg.l
    z = normal(cfg.seed, S_X, n * cfg.c * l).reshape(n, cfg.c, l)[:, :C, :]
    lo, hi = cfg.scale_range
    scale = lo + (hi - lo) * uniform(cfg.seed, S_SCALE, cfg.c)[:C]
    if cfg.x_kind == "offset_scale":
        olo, ohi = cfg.off_range
        off = olo + (ohi - olo) * uniform(cfg.seed, S_OFF, cfg.c)[:C]
        x = off[None, :, None] + scale[None, :, None] * z
    elif cfg.x_kind == "scale":
        x = z * scale[None, :, None]
    else:
        raise ValueError(cfg.x_kind)
    out = {"x": store(x, cfg.dtype, (n, C, l))}
    if cfg.residual:
        r = normal(cfg.seed, S_RES, n * cfg.c * l).reshape(n, cfg.c, l)[:, :C, :]
        out["res"] = store(r, cfg.dtype, (n, C, l))
    w = np.ones(C) if cfg.w_std == 0 else 1.0 + cfg.w_std * normal(cfg.seed, S_W, cfg.c)[:C]
    b = np.zeros(C) if cfg.b_std == 0 else cfg.b_std * normal(cfg.seed, S_B, cfg.c)[:C]
    out["w"] = store(w, "f32", (C,))
    out["b"] = store(b, "f32", (C,))
    d = normal(cfg.seed, S_DY, n * cfg.c * l).reshape(n, cfg.c, l)[:, :C, :]
    out["dy"] = store(d, cfg.dtype, (n, C, l))
    out["running_mean"] = store(np.zeros(C), "f32", (C,))
    out["running_var"] = store(np.ones(C), "f32", (C,))
    return out


def random_tensor(seed: int, stream: int, shape, dtype: str, mean=0.0, std=1.0) -> Tensor:
    """A normal tensor of any shape (for odd-shape and edge-case tests)."""
    count = int(np.prod(shape)) if len(shape) else 1
    return store(mean + std * normal(seed, stream, count), dtype, shape)
