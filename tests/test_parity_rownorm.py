"""LayerNorm / RMSNorm through libnorm's C ABI against the CPU oracle, element by
element: the full-size workloads (LLaMA-style RMSNorm bf16 [16384, 4096] with
outlier columns, ViT-B LayerNorm fp16 [25216, 768]), the small fp32 case, and
odd shapes that exercise every kernel path (register-resident vector path,
unaligned scalar path, two-pass wide-row path, ragged tails)."""
import numpy as np
import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import (DT_CODE, STAT_TOL, TOL, assert_close, compare_row, dev, empty, host, oracle_row, run_row, workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()


@pytest.mark.parametrize("name", ["ln_f32_64x256", "rms_bf16_16384x4096", "ln_f16_25216x768"])
def test_row_workloads_full_size(orc, name):
    cfg = synth.CONFIGS[name]
    inp = synth.row_inputs(cfg)
    got = run_row(cfg.kind, inp, cfg.dtype, cfg.eps)
    want = oracle_row(orc, cfg.kind, inp, cfg.eps)
    compare_row(got, want, cfg.dtype, name)


def test_row_wide_workload_full_size(orc):
    # the wide-row workload timed beside the step, LayerNorm fp16 [2048, 65536]:
    # rows above the register and ring kernels' widths, one 1024-thread CTA each
    cfg = synth.RowConfig("wide", "layernorm", 2048, 65536, "f16", 1e-5, seed=43, x_mean=0.3, x_std=1.5)
    inp = synth.row_inputs(cfg)
    got = run_row(cfg.kind, inp, cfg.dtype, cfg.eps)
    want = oracle_row(orc, cfg.kind, inp, cfg.eps)
    compare_row(got, want, cfg.dtype, "ln f16 [2048,65536]")


ODD_COLS = [1, 7, 8, 33, 64, 100, 256, 768, 1023, 1025, 2048, 4097, 8200, 40000]


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("cols", ODD_COLS)
def test_row_odd_shapes(orc, kind, dtype, cols):
    rows = 37 if cols < 8192 else 5
    cfg = synth.RowConfig("odd", kind, rows, cols, dtype, 1e-5, seed=100 + cols,
                          x_mean=0.5, x_std=2.0)
    inp = synth.row_inputs(cfg)
    got = run_row(kind, inp, dtype, cfg.eps)
    want = oracle_row(orc, kind, inp, cfg.eps)
    compare_row(got, want, dtype, f"{kind} {dtype} [{rows},{cols}]")


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_row_misaligned_pointers_use_scalar_path(orc, kind, dtype):
    # cols a multiple of 16 bytes, but every tensor starts one element past a
    # 16-byte boundary: the kernels must take the unaligned path
    rows, cols = 50, 512
    cfg = synth.RowConfig("mis", kind, rows, cols, dtype, 1e-5, seed=7)
    inp = synth.row_inputs(cfg)

    def shifted(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")
        view = buf[1:1 + t.numel()].view(t.shape)
        view.copy_(t)
        return view

    x = shifted(dev(inp["x"]))
    dy = shifted(dev(inp["dy"]))
    w = shifted(dev(inp["w"]))
    b = shifted(dev(inp["b"])) if kind == "layernorm" else None
    y = shifted(empty((rows, cols), dtype))
    dx = shifted(empty((rows, cols), dtype))
    dw = shifted(empty((cols,), dtype))
    db = shifted(empty((cols,), dtype)) if kind == "layernorm" else None
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    if kind == "layernorm":
        nrm.nrm_layernorm_fwd(x, w, b, y, mean, rstd, cfg.eps)
        ws = workspace(nrm.NRM_OP_LAYERNORM_BWD, rows, cols, DT_CODE[dtype])
        nrm.nrm_layernorm_bwd(dy, x, w, mean, rstd, dx, dw, db, ws)
    else:
        nrm.nrm_rmsnorm_fwd(x, w, y, rstd, cfg.eps)
        ws = workspace(nrm.NRM_OP_RMSNORM_BWD, rows, cols, DT_CODE[dtype])
        nrm.nrm_rmsnorm_bwd(dy, x, w, rstd, dx, dw, ws)
    nrm.nrm_sync_status()
    got = dict(y=host(y), dx=host(dx), dw=host(dw), rstd=host(rstd))
    if kind == "layernorm":
        got.update(mean=host(mean), db=host(db))
    compare_row(got, oracle_row(orc, kind, inp, cfg.eps), dtype, f"misaligned {kind} {dtype}")


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_row_without_affine_and_gradients(orc, kind):
    cfg = synth.RowConfig("noaff", kind, 300, 384, "bf16", 1e-5, seed=11)
    inp = synth.row_inputs(cfg)
    got = run_row(kind, inp, "bf16", cfg.eps, with_w=False, with_b=False, want_dw=False,
                  want_db=False)
    want = oracle_row(orc, kind, inp, cfg.eps, with_w=False, with_b=False)
    compare_row(got, want, "bf16", f"{kind} without affine")


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_row_zero_rows_gives_zero_gradients(kind):
    cols = 96
    x = torch.empty((0, cols), dtype=torch.float16, device="cuda")
    dy = torch.empty_like(x)
    dx = torch.empty_like(x)
    w = torch.ones(cols, dtype=torch.float16, device="cuda")
    dw = torch.full((cols,), 7.0, dtype=torch.float16, device="cuda")
    db = torch.full((cols,), 7.0, dtype=torch.float16, device="cuda")
    stats = torch.empty(0, device="cuda")
    if kind == "layernorm":
        nrm.nrm_layernorm_bwd(dy, x, w, stats, stats, dx, dw, db, None)
    else:
        nrm.nrm_rmsnorm_bwd(dy, x, w, stats, dx, dw, None)
    nrm.nrm_sync_status()
    assert (dw == 0).all()
    if kind == "layernorm":
        assert (db == 0).all()


def test_constant_rows(orc):
    # a constant row has variance 0: y = b, rstd = eps^-1/2
    rows, cols = 9, 640
    x = torch.full((rows, cols), 3.25, dtype=torch.float32, device="cuda")
    w = torch.linspace(0.5, 1.5, cols, device="cuda")
    b = torch.linspace(-1, 1, cols, device="cuda")
    y = torch.empty_like(x)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    nrm.nrm_layernorm_fwd(x, w, b, y, mean, rstd, 1e-4)
    nrm.nrm_sync_status()
    want_y, want_mean, want_rstd = orc.layernorm_fwd(host(x), host(w), host(b), 1e-4)
    np.testing.assert_allclose(host(y), want_y, atol=1e-5, rtol=1e-5)
    np.testing.assert_allclose(host(rstd), want_rstd, rtol=1e-5)


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("dtype,rows,cols", [("f16", 20011, 256), ("f32", 3001, 1024), ("bf16", 613, 8192)])
def test_row_backward_ring_many_chunks(orc, kind, dtype, rows, cols):
    # aligned rows the backward streams through shared memory: several chunks
    # per CTA and a ragged last chunk
    cfg = synth.RowConfig("ring", kind, rows, cols, dtype, 1e-5, seed=rows + cols, x_mean=-0.3, x_std=1.7)
    inp = synth.row_inputs(cfg)
    got = run_row(kind, inp, dtype, cfg.eps)
    want = oracle_row(orc, kind, inp, cfg.eps)
    compare_row(got, want, dtype, f"{kind} {dtype} [{rows},{cols}]")


RMS_BIAS = [(300, 256), (300, 768), (97, 1023), (5, 40000), (2000, 4096)]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", RMS_BIAS, ids=[f"{r}x{c}" for r, c in RMS_BIAS])
def test_rmsnorm_with_bias(orc, dtype, shape):
    # the ring backward (aligned rows), the register kernels (1023 columns are
    # not 16-byte rows), the wide-row kernels (40000 columns)
    rows, cols = shape
    check_rmsnorm_bias(orc, dtype, rows, cols, 60 + cols % 97)


def check_rmsnorm_bias(orc, dtype, rows, cols, seed):
    """RMSNorm with its optional bias, forward and backward (db), against the oracle."""
    inp = {
        "x": synth.random_tensor(seed, 1, (rows, cols), dtype, std=1.3),
        "w": synth.store(1 + 0.1 * synth.normal(seed, 2, cols), dtype, (cols,)),
        "b": synth.store(0.2 * synth.normal(seed, 3, cols), dtype, (cols,)),
        "dy": synth.random_tensor(seed, 4, (rows, cols), dtype),
    }
    got = run_row("rmsnorm", inp, dtype, 1e-6)
    want = oracle_row(orc, "rmsnorm", inp, 1e-6)
    assert "db" in got
    compare_row(got, want, dtype, f"rms+bias {dtype} [{rows},{cols}]")


F32OUT = [(300, 768), (97, 1023), (64, 4096), (5, 40000), (25216, 768)]  # the last: the bench workload's size


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", F32OUT, ids=[f"{r}x{c}" for r, c in F32OUT])
def test_row_f32_output(orc, kind, dtype, shape):
    rows, cols = shape
    check_f32_output(orc, kind, dtype, rows, cols, 80 + cols % 91)


def check_f32_output(orc, kind, dtype, rows, cols, seed):
    """The autocast_to_fp32-style option: a 16-bit x, y (and so dy) in float32;
    y meets the fp32 bound, dx/dw/db (stored 16-bit) the 16-bit one."""
    x = synth.random_tensor(seed, 1, (rows, cols), dtype, mean=0.2, std=1.3)
    w = synth.store(1 + 0.1 * synth.normal(seed, 2, cols), dtype, (cols,))
    b = synth.store(0.1 * synth.normal(seed, 3, cols), dtype, (cols,))
    dy = synth.random_tensor(seed, 4, (rows, cols), "f32")
    xt, wt, bt, dyt = x.torch("cuda"), w.torch("cuda"), b.torch("cuda"), dy.torch("cuda")
    y = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    dx = empty((rows, cols), dtype)
    dw = empty((cols,), dtype)
    db = empty((cols,), dtype)
    if kind == "layernorm":
        nrm.nrm_layernorm_fwd_ex(xt, wt, bt, y, mean, rstd, 1e-5)
        ws = workspace(nrm.NRM_OP_LAYERNORM_BWD, rows, cols, DT_CODE[dtype])
        nrm.nrm_layernorm_bwd_ex(dyt, xt, wt, mean, rstd, dx, dw, db, ws)
        yo, mo, ro = orc.layernorm_fwd(x.f64(), w.f64(), b.f64(), 1e-5)
        dxo, dwo, dbo = orc.layernorm_bwd(dy.f64(), x.f64(), w.f64(), 1e-5)
    else:
        nrm.nrm_rmsnorm_fwd_ex(xt, wt, y, rstd, 1e-5, b=bt)
        ws = workspace(nrm.NRM_OP_RMSNORM_BWD, rows, cols, DT_CODE[dtype])
        nrm.nrm_rmsnorm_bwd_ex(dyt, xt, wt, rstd, dx, dw, ws, db=db)
        yo, ro = orc.rmsnorm_fwd(x.f64(), w.f64(), 1e-5, b=b.f64())
        dxo, dwo, dbo = orc.rmsnorm_bwd(dy.f64(), x.f64(), w.f64(), 1e-5, with_db=True)
    nrm.nrm_sync_status()
    tag = f"{kind} {dtype}->f32 [{rows},{cols}]"
    assert_close(host(y), yo, TOL["f32"], tag + " y")
    assert_close(host(rstd), ro, STAT_TOL, tag + " rstd")
    if kind == "layernorm":
        assert_close(host(mean), mo, STAT_TOL, tag + " mean")
    assert_close(host(dx), dxo, TOL[dtype], tag + " dx")
    assert_close(host(dw), dwo, TOL[dtype], tag + " dw")
    assert_close(host(db), dbo, TOL[dtype], tag + " db")
