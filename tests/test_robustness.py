"""Robustness of libnorm on the GPU (compute-sanitizer is closed on this machine, so
these stand in for it):
  * bitwise determinism: two runs of every entry point give identical bytes;
  * canary guards: every output lives inside a larger buffer whose guard
    regions must be untouched after the call (out-of-bounds writes);
  * argument errors with a live context: bad calls return a status, enqueue
    nothing, and the next good call still works."""
import numpy as np
import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import DT_CODE, TORCH_DT

pytestmark = pytest.mark.gpu

GUARD = 1024  # bytes of guard on each side


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()


class Guarded:
    """A tensor view inside a byte buffer with canary-filled guard regions.
    `offset` (bytes) shifts the view off 16-byte alignment when not 0."""

    def __init__(self, shape, dtype, offset=0):
        numel = int(np.prod(shape)) if len(shape) else 1
        es = torch.empty(0, dtype=dtype).element_size()
        offset -= offset % es  # a view must start on an element boundary
        self.buf = torch.full((GUARD * 2 + numel * es + offset,), 0x5A, dtype=torch.uint8, device="cuda")
        start = GUARD + offset
        self.t = self.buf[start:start + numel * es].view(dtype).view(shape)
        self.start, self.end = start, start + numel * es

    def check(self, what):
        b = self.buf.cpu().numpy()
        assert (b[:self.start] == 0x5A).all(), f"{what}: write before the tensor"
        assert (b[self.end:] == 0x5A).all(), f"{what}: write after the tensor"


def _row_run(kind, dtype, rows, cols, offset, seed):
    cfg = synth.RowConfig("g", kind, rows, cols, dtype, 1e-5, seed)
    inp = synth.row_inputs(cfg)
    td = TORCH_DT[dtype]
    x = inp["x"].torch("cuda")
    dy = inp["dy"].torch("cuda")
    w = inp["w"].torch("cuda")
    b = inp["b"].torch("cuda") if kind == "layernorm" else None
    outs = {k: Guarded(s, t, offset) for k, s, t in (
        ("y", (rows, cols), td), ("dx", (rows, cols), td), ("dw", (cols,), td), ("db", (cols,), td),
        ("mean", (rows,), torch.float32), ("rstd", (rows,), torch.float32))}
    op = nrm.NRM_OP_LAYERNORM_BWD if kind == "layernorm" else nrm.NRM_OP_RMSNORM_BWD
    nws = nrm.nrm_workspace_bytes(op, rows, cols, DT_CODE[dtype])
    ws = Guarded((nws // 4,), torch.float32)
    o = {k: g.t for k, g in outs.items()}
    if kind == "layernorm":
        nrm.nrm_layernorm_fwd(x, w, b, o["y"], o["mean"], o["rstd"], 1e-5)
        nrm.nrm_layernorm_bwd(dy, x, w, o["mean"], o["rstd"], o["dx"], o["dw"], o["db"], ws.t)
    else:
        nrm.nrm_rmsnorm_fwd(x, w, o["y"], o["rstd"], 1e-5)
        nrm.nrm_rmsnorm_bwd(dy, x, w, o["rstd"], o["dx"], o["dw"], ws.t)
    nrm.nrm_sync_status()
    for k, g in outs.items():
        if kind == "rmsnorm" and k in ("db", "mean"):
            continue
        g.check(f"{kind} {dtype} [{rows},{cols}] {k}")
    ws.check("workspace")
    return {k: g.t.clone() for k, g in outs.items()}


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("dtype,rows,cols,offset", [
    ("f32", 33, 1000, 0), ("f16", 257, 768, 0), ("bf16", 64, 4096, 0), ("bf16", 5, 4097, 2),
    ("f16", 3, 33000, 0), ("f32", 100, 7, 4), ("bf16", 1000, 64, 0),
])
def test_row_guards_and_determinism(kind, dtype, rows, cols, offset):
    a = _row_run(kind, dtype, rows, cols, offset, seed=rows + cols)
    b = _row_run(kind, dtype, rows, cols, offset, seed=rows + cols)
    for k in a:
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), f"{k} differs between runs"


def _bn_run(dtype, n, c, l, act, res, training, mask, offset):
    cfg = synth.BnConfig("g", n, c, l, dtype, 1e-5, 0.1, n + c + l, act=act, residual=res,
                         x_kind="offset_scale", w_std=0.1, b_std=0.1)
    inp = synth.bn_inputs(cfg)
    td = TORCH_DT[dtype]
    x = inp["x"].torch("cuda")
    r = inp["res"].torch("cuda") if res else None
    w, b_ = inp["w"].torch("cuda"), inp["b"].torch("cuda")
    dy = inp["dy"].torch("cuda")
    rm = Guarded((c,), torch.float32)
    rv = Guarded((c,), torch.float32)
    rm.t.zero_()
    rv.t.fill_(1.0)
    outs = {k: Guarded(s, t, offset) for k, s, t in (
        ("y", (n, c, l), td), ("dx", (n, c, l), td), ("dres", (n, c, l), td),
        ("sm", (c,), torch.float32), ("sr", (c,), torch.float32), ("dw", (c,), torch.float32),
        ("db", (c,), torch.float32))}
    mk = Guarded((nrm.nrm_act_mask_words(n, c, l),), torch.int32) if mask else None
    o = {k: g.t for k, g in outs.items()}
    nws = nrm.nrm_batchnorm_workspace_bytes(n, c, l, DT_CODE[dtype])
    ws = Guarded((nws,), torch.uint8)
    nrm.nrm_batchnorm_fwd(x, r, w, b_, o["y"], rm.t, rv.t, o["sm"], o["sr"], mk.t if mk else None,
                          1e-5, 0.1, training, act, ws.t)
    nrm.nrm_batchnorm_bwd(dy, x, r, w, b_, o["sm"], o["sr"], mk.t if mk else None, o["dx"], o["dres"],
                          o["dw"], o["db"], training, act, ws.t)
    nrm.nrm_sync_status()
    for k, g in list(outs.items()) + [("rm", rm), ("rv", rv), ("ws", ws)] + ([("mask", mk)] if mk else []):
        g.check(f"bn {dtype} [{n},{c},{l}] {act} {k}")
    got = {k: g.t.clone() for k, g in outs.items()}
    got["rm"], got["rv"] = rm.t.clone(), rv.t.clone()
    if mk:
        got["mask"] = mk.t.clone()
    return got


@pytest.mark.parametrize("dtype,n,c,l,act,res,training,mask,offset", [
    ("f32", 4, 3, 3136, "relu", True, True, True, 0),
    ("f32", 3, 5, 49, "relu", True, True, True, 4),
    ("f16", 16, 8, 49, "gelu", False, True, False, 0),
    ("bf16", 2, 3, 70, "relu", False, False, True, 2),
    ("f32", 128, 2, 12544, "none", True, True, False, 0),
    ("f16", 7, 3, 33, "relu", True, False, False, 0),
    ("bf16", 9, 8, 7, "relu", True, True, True, 0),     # channel groups, cluster of 8
    ("f32", 33, 12, 9, "gelu", True, False, False, 0),  # channel groups, an empty CTA
])
def test_bn_guards_and_determinism(dtype, n, c, l, act, res, training, mask, offset):
    a = _bn_run(dtype, n, c, l, act, res, training, mask, offset)
    b = _bn_run(dtype, n, c, l, act, res, training, mask, offset)
    for k in a:
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), f"{k} differs between runs"


def _cf_run(dtype, n, c, l, offset, seed):
    td = TORCH_DT[dtype]
    x = synth.random_tensor(seed, 1, (n, c, l), dtype, mean=0.2, std=1.3).torch("cuda")
    dy = synth.random_tensor(seed, 2, (n, c, l), dtype).torch("cuda")
    w = synth.store(1 + 0.1 * synth.normal(seed, 3, c), dtype, (c,)).torch("cuda")
    b = synth.store(0.1 * synth.normal(seed, 4, c), dtype, (c,)).torch("cuda")
    outs = {k: Guarded(sh, t, offset) for k, sh, t in (
        ("y", (n, c, l), td), ("dx", (n, c, l), td), ("dw", (c,), td), ("db", (c,), td),
        ("mean", (n, l), torch.float32), ("rstd", (n, l), torch.float32))}
    nws = nrm.nrm_workspace_bytes(nrm.NRM_OP_LAYERNORM_CF_BWD, n * l, c, DT_CODE[dtype])
    ws = Guarded((nws // 4,), torch.float32)
    o = {k: g.t for k, g in outs.items()}
    nrm.nrm_layernorm_cf_fwd(x, w, b, o["y"], o["mean"], o["rstd"], 1e-6)
    nrm.nrm_layernorm_cf_bwd(dy, x, w, o["mean"], o["rstd"], o["dx"], o["dw"], o["db"], ws.t)
    nrm.nrm_sync_status()
    for k, g in list(outs.items()) + [("ws", ws)]:
        g.check(f"cf {dtype} [{n},{c},{l}] {k}")
    return {k: g.t.clone() for k, g in outs.items()}


@pytest.mark.parametrize("dtype,n,c,l,offset", [
    ("f16", 4, 96, 3136, 0),   # TMA ring, ragged last tile
    ("f32", 3, 300, 36, 0),    # two channel boxes
    ("f16", 3, 257, 200, 0),   # second box past c
    ("bf16", 4, 384, 196, 0),  # register kernel (unaligned planes)
    ("f16", 2, 96, 784, 4),    # unaligned outputs: the register kernel
])
def test_cf_guards_and_determinism(dtype, n, c, l, offset):
    a = _cf_run(dtype, n, c, l, offset, seed=n + c + l)
    b = _cf_run(dtype, n, c, l, offset, seed=n + c + l)
    for k in a:
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), f"{k} differs between runs"


@pytest.mark.parametrize("dtype,count,act,offset", [
    ("f16", 100_003, "gelu", 0), ("f32", 4099, "selu", 4), ("bf16", 65_541, "leaky_relu", 2),
    ("f16", 7, "mish", 0),
])
def test_dropout_guards_and_determinism(dtype, count, act, offset):
    td = TORCH_DT[dtype]
    x = synth.random_tensor(5, 1, (count,), dtype).torch("cuda")
    dy = synth.random_tensor(5, 2, (count,), dtype).torch("cuda")
    runs = []
    for _ in range(2):
        y = Guarded((count,), td, offset)
        dx = Guarded((count,), td, offset)
        nrm.nrm_act_dropout_fwd(x, y.t, act, 0.3, 12345, act_param=0.1)
        nrm.nrm_act_dropout_bwd(dy, x, dx.t, act, 0.3, 12345, act_param=0.1)
        nrm.nrm_sync_status()
        y.check(f"dropout {dtype} {count} y")
        dx.check(f"dropout {dtype} {count} dx")
        runs.append((y.t.clone(), dx.t.clone()))
    for (a, b) in zip(runs[0], runs[1]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), "dropout differs between runs"


def test_rmsnorm_bias_guards_and_determinism():
    rows, cols = 300, 768
    outs = []
    for _ in range(2):
        x = synth.random_tensor(9, 1, (rows, cols), "bf16").torch("cuda")
        dy = synth.random_tensor(9, 2, (rows, cols), "bf16").torch("cuda")
        w = synth.store(1 + 0.1 * synth.normal(9, 3, cols), "bf16", (cols,)).torch("cuda")
        b = synth.store(0.1 * synth.normal(9, 4, cols), "bf16", (cols,)).torch("cuda")
        g = {k: Guarded(sh, t) for k, sh, t in (
            ("y", (rows, cols), torch.bfloat16), ("dx", (rows, cols), torch.bfloat16),
            ("dw", (cols,), torch.bfloat16), ("db", (cols,), torch.bfloat16), ("rstd", (rows,), torch.float32))}
        ws = Guarded((nrm.nrm_workspace_bytes(nrm.NRM_OP_RMSNORM_BWD, rows, cols, nrm.NRM_BF16) // 4,),
                     torch.float32)
        nrm.nrm_rmsnorm_fwd(x, w, g["y"].t, g["rstd"].t, 1e-6, b=b)
        nrm.nrm_rmsnorm_bwd(dy, x, w, g["rstd"].t, g["dx"].t, g["dw"].t, ws.t, db=g["db"].t)
        nrm.nrm_sync_status()
        for k, v in list(g.items()) + [("ws", ws)]:
            v.check(f"rms bias {k}")
        outs.append({k: v.t.clone() for k, v in g.items()})
    for k in outs[0]:
        assert torch.equal(outs[0][k].view(torch.uint8), outs[1][k].view(torch.uint8)), f"{k} differs"


def test_errors_leave_the_context_usable():
    lib = nrm.load()
    x = torch.randn(64, 256, device="cuda")
    y = torch.empty_like(x)
    # short workspace
    dw = torch.empty(256, device="cuda")
    ws = torch.empty(4, device="cuda")
    st = torch.empty(64, device="cuda")
    with pytest.raises(nrm.NrmError) as e:
        nrm.nrm_rmsnorm_bwd(x, x, None, st, y, dw, ws)
    assert e.value.status == nrm.NRM_ERR_WORKSPACE
    # null output
    assert lib.nrm_layernorm_fwd(x.data_ptr(), None, None, None, None, None, 64, 256, 1e-5,
                                 nrm.NRM_F32, None) == nrm.NRM_ERR_INVALID_ARG
    # misaligned element pointer
    assert lib.nrm_layernorm_fwd(x.data_ptr() + 2, None, None, y.data_ptr(), None, None, 64, 256,
                                 1e-5, nrm.NRM_F32, None) == nrm.NRM_ERR_INVALID_ARG
    # the next good call works
    nrm.nrm_rmsnorm_fwd(x, None, y, st, 1e-5)
    nrm.nrm_sync_status()
    ref = x / torch.sqrt((x * x).mean(1, keepdim=True) + 1e-5)
    assert torch.allclose(y, ref, atol=1e-5, rtol=1e-5)


def test_streams_are_respected():
    # work enqueued on a side stream is complete once that stream has synchronised
    s = torch.cuda.Stream()
    x = torch.randn(4096, 1024, device="cuda", dtype=torch.bfloat16)
    y = torch.zeros_like(x)
    rstd = torch.empty(4096, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        nrm.nrm_rmsnorm_fwd(x, None, y, rstd, 1e-6)
    s.synchronize()
    xf = x.float()
    ref = xf * torch.rsqrt((xf * xf).mean(1, keepdim=True) + 1e-6)
    err = (y.float() - ref).abs()
    assert bool((err <= 2e-2 + 1e-2 * ref.abs()).all())
