"""LayerNorm over the channels of an NCHW tensor (channels first) through
libnorm's C ABI against the CPU oracle, element by element: ConvNeXt-like
shapes on the 16-byte vector path and on the unaligned scalar path, a
multi-tile grid with ragged tiles, absent affine parameters, and an empty
tensor."""
import numpy as np
import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import DT_CODE, STAT_TOL, TOL, assert_close, empty, host, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()


def _inputs(n, c, l, dtype, seed, affine=True):
    x = synth.random_tensor(seed, 1, (n, c, l), dtype, mean=0.3, std=1.5)
    dy = synth.random_tensor(seed, 2, (n, c, l), dtype)
    w = synth.store(1 + 0.1 * synth.normal(seed, 3, c), dtype, (c,)) if affine else None
    b = synth.store(0.1 * synth.normal(seed, 4, c), dtype, (c,)) if affine else None
    return x, dy, w, b


def _run(x, dy, w, b, dtype, eps, stat_offset=0):
    n, c, l = x.shape
    xt, dyt = x.torch("cuda"), dy.torch("cuda")
    wt = w.torch("cuda") if w is not None else None
    bt = b.torch("cuda") if b is not None else None
    y = empty((n, c, l), dtype)
    # stat_offset floats in: saved statistics that are not 16-byte aligned
    mean = torch.empty(n * l + stat_offset, device="cuda")[stat_offset:].view(n, l)
    rstd = torch.empty(n * l + stat_offset, device="cuda")[stat_offset:].view(n, l)
    nrm.nrm_layernorm_cf_fwd(xt, wt, bt, y, mean, rstd, eps)
    dx = empty((n, c, l), dtype)
    dw = empty((c,), dtype)
    db = empty((c,), dtype)
    ws = workspace(nrm.NRM_OP_LAYERNORM_CF_BWD, n * l, c, DT_CODE[dtype])
    nrm.nrm_layernorm_cf_bwd(dyt, xt, wt, mean, rstd, dx, dw, db, ws)
    nrm.nrm_sync_status()
    return {k: host(v) for k, v in dict(y=y, mean=mean, rstd=rstd, dx=dx, dw=dw, db=db).items()}


def _check(orc, x, dy, w, b, dtype, eps, tag, stat_offset=0):
    got = _run(x, dy, w, b, dtype, eps, stat_offset)
    wf = w.f64() if w is not None else None
    bf = b.f64() if b is not None else None
    y, mean, rstd = orc.layernorm_cf_fwd(x.f64(), wf, bf, eps=eps)
    dx, dw, db = orc.layernorm_cf_bwd(dy.f64(), x.f64(), wf, eps=eps)
    tol = TOL[dtype]
    assert_close(got["mean"], mean, STAT_TOL, tag + " mean")
    assert_close(got["rstd"], rstd, STAT_TOL, tag + " rstd")
    assert_close(got["y"], y, tol, tag + " y")
    assert_close(got["dx"], dx, tol, tag + " dx")
    assert_close(got["dw"], dw, tol, tag + " dw")
    assert_close(got["db"], db, tol, tag + " db")


CASES = [
    # (dtype, n, c, l): ConvNeXt stage shapes (channels of 56x56 ... 7x7 maps) and odd ones
    ("f16", 8, 96, 3136),    # vector path, 12 tiles per sample, a ragged last tile
    ("bf16", 4, 768, 49),    # 98-byte planes: the scalar path
    ("f32", 4, 192, 784),    # vector path, f32
    ("f32", 3, 5, 33),       # scalar, few channels, ragged tile
    ("bf16", 2, 384, 196),   # 392-byte planes (not a multiple of 16): the scalar path
    ("f16", 1, 3, 8),        # one tile, three channels
    ("f16", 3, 257, 200),    # two channel boxes (the second one past c), positions past l
    ("bf16", 2, 1024, 64),   # too many channels for a shared-memory tile: the register kernel
    ("f32", 5, 300, 36),     # 144-byte planes, two boxes of 150 channels
]


@pytest.mark.parametrize("case", CASES, ids=[f"{d}-{n}x{c}x{l}" for d, n, c, l in CASES])
def test_layernorm_cf(orc, case):
    dtype, n, c, l = case
    x, dy, w, b = _inputs(n, c, l, dtype, seed=n * 1000 + c + l)
    _check(orc, x, dy, w, b, dtype, 1e-6, f"cf {dtype} [{n},{c},{l}]")


def test_layernorm_cf_without_affine(orc):
    x, dy, _, _ = _inputs(2, 64, 1024, "f32", seed=11, affine=False)
    _check(orc, x, dy, None, None, "f32", 1e-5, "cf no affine")


def test_layernorm_cf_unaligned_saved_statistics(orc):
    # saved mean/rstd 4-byte but not 16-byte aligned: the backward cannot bulk-copy them
    x, dy, w, b = _inputs(4, 96, 784, "f16", seed=13)
    _check(orc, x, dy, w, b, "f16", 1e-6, "cf unaligned stats", stat_offset=1)


def test_layernorm_cf_many_tiles_per_cta(orc):
    # more tiles than resident CTAs: the backward's persistent CTAs each sum
    # several tiles into their dw/db partial rows
    x, dy, w, b = _inputs(64, 32, 3136, "bf16", seed=12)
    _check(orc, x, dy, w, b, "bf16", 1e-6, "cf many tiles")


def test_layernorm_cf_empty_gives_zero_grads():
    c = 16
    x = torch.empty((0, c, 5), dtype=torch.float32, device="cuda")
    dw = torch.full((c,), 7.0, device="cuda")
    db = torch.full((c,), 7.0, device="cuda")
    mean = torch.empty((0, 5), device="cuda")
    nrm.nrm_layernorm_cf_fwd(x, None, None, torch.empty_like(x), mean, mean, 1e-5)
    nrm.nrm_layernorm_cf_bwd(x, x, None, mean, mean, torch.empty_like(x), dw, db, None)
    nrm.nrm_sync_status()
    assert torch.count_nonzero(dw).item() == 0 and torch.count_nonzero(db).item() == 0


def test_layernorm_cf_bench_size(orc):
    # the benchmarked workload itself (ConvNeXt-T's 96 channels of 56x56, batch
    # 128, fp16, same seeds), every element against the oracle
    x, dy, w, b = _inputs(128, 96, 3136, "f16", seed=31)
    _check(orc, x, dy, w, b, "f16", 1e-6, "cf bench size")
