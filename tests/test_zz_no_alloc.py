"""nrm_layernorm_bwd_noalloc: the LayerNorm backward for callers that cannot
allocate device memory (code running under another framework's allocator,
loops that must never enter cudaMalloc after start-up, C callers holding only
device pointers).  It keeps the dw/db partial rows in the library's own static
device array instead of a caller workspace.

Checked through the C ABI against the CPU oracle and against nrm_layernorm_bwd
(the entry point with a workspace), with the parity tolerances, on two calls in
a row (the second call finds the previous call's partial sums still in the
shared array).  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh
process."""
import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import DT_CODE, TOL, assert_close, host, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()


def _inputs(rows, cols, dtype, seed):
    cfg = synth.RowConfig("noalloc", "layernorm", rows, cols, dtype, 1e-5, seed, x_mean=0.2, x_std=1.3)
    inp = synth.row_inputs(cfg)
    x, w, b, dy = (inp[k].torch("cuda") for k in ("x", "w", "b", "dy"))
    y = torch.empty_like(x)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    nrm.nrm_layernorm_fwd(x, w, b, y, mean, rstd, cfg.eps)
    return x, w, dy, mean, rstd, inp, cfg.eps


@pytest.mark.parametrize("dtype,rows,cols", [
    ("f16", 25216, 768),     # ViT-B tokens
    ("bf16", 2048, 4096),    # wide rows, register path
    ("f32", 300, 1000),      # vector path, ragged groups
    ("bf16", 64, 12000),     # wide-row kernel
    ("f16", 37, 1025),       # unaligned scalar path
])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(orc, dtype, rows, cols):
    x, w, dy, mean, rstd, inp, eps = _inputs(rows, cols, dtype, seed=rows + cols)
    dx_o, dw_o, db_o = orc.layernorm_bwd(inp["dy"].f64(), inp["x"].f64(), inp["w"].f64(), eps)
    dx_ref = torch.empty_like(x)
    dw_ref = torch.empty_like(w)
    db_ref = torch.empty_like(w)
    ws = workspace(nrm.NRM_OP_LAYERNORM_BWD, rows, cols, DT_CODE[dtype])
    nrm.nrm_layernorm_bwd(dy, x, w, mean, rstd, dx_ref, dw_ref, db_ref, ws)
    nrm.nrm_sync_status()
    tol = TOL[dtype]
    for call in range(2):
        dx = torch.full_like(x, 7.0)
        dw = torch.full_like(w, 7.0)
        db = torch.full_like(w, 7.0)
        nrm.nrm_layernorm_bwd_noalloc(dy, x, w, mean, rstd, dx, dw, db)
        nrm.nrm_sync_status()
        tag = f"noalloc call {call + 1} {dtype} [{rows},{cols}]"
        assert_close(host(dx), dx_o, tol, tag + " dx vs oracle")
        assert_close(host(dw), dw_o, tol, tag + " dw vs oracle")
        assert_close(host(db), db_o, tol, tag + " db vs oracle")
        assert_close(host(dx), host(dx_ref), tol, tag + " dx")
        assert_close(host(dw), host(dw_ref), tol, tag + " dw")
        assert_close(host(db), host(db_ref), tol, tag + " db")


def test_noalloc_rejects_rows_wider_than_its_scratch():
    cols = 65537
    x = torch.zeros(2, cols, device="cuda")
    st = torch.zeros(2, device="cuda")
    with pytest.raises(nrm.NrmError) as e:
        nrm.nrm_layernorm_bwd_noalloc(x, x, None, st, st, torch.empty_like(x),
                                      torch.empty(cols, device="cuda"), None)
    assert e.value.status == nrm.NRM_ERR_UNSUPPORTED
    assert "65536" in str(e.value)
