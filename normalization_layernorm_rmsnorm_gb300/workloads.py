"""The bench's workloads as a list of C-ABI calls on device-resident inputs.

Each Call wraps one libnorm entry point with its tensors, its algorithmic bytes
(every input read once, every output written once, saved statistics, ReLU mask
bits: the bytes that must cross HBM) and the kernels it launches.  Used by
bench.py and by profile_case (the driver of the ncu captures).
"""
from __future__ import annotations


def nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


class Call:
    def __init__(self, workload, phase, kernel, fn, nbytes_, launches, inputs, outputs):
        self.workload = workload
        self.phase = phase
        self.kernel = kernel
        self.fn = fn
        self.bytes = nbytes_
        self.launches = launches
        self.inputs = inputs      # device tensors a user would upload
        self.outputs = outputs    # device tensors a user would download
        self.times_ms: list[float] = []


def build_calls(dev, names=None):
    """The calls of one bench step (or only those of the workloads in `names`)."""
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth

    calls = []

    def f32(n):
        return torch.empty(n, dtype=torch.float32, device=dev)

    def want(name):
        return names is None or name in names

    # ---- LayerNorm f32 [64, 256]: the small case (latency-bound, a few µs) ----
    cfg = synth.CONFIGS["ln_f32_64x256"]
    if want(cfg.name):
        calls += _ln(cfg, dev, f32)
    # ---- RMSNorm bf16 [16384, 4096] ----
    cfg = synth.CONFIGS["rms_bf16_16384x4096"]
    if want(cfg.name):
        calls += _rms(cfg, dev, f32)
    cfg = synth.CONFIGS["ln_f16_25216x768"]
    if want(cfg.name):
        calls += _ln(cfg, dev, f32)
    cfg = synth.CONFIGS["bn_f32_256x64x56x56_res_relu"]
    if want(cfg.name) or want(cfg.name + "_eval"):
        calls += [c for c in _bn_res_relu(cfg, dev, f32) if want(c.workload)]
    cfg = synth.CONFIGS["bn_f16_128x512x7x7_gelu"]
    if want(cfg.name):
        calls += _bn_gelu(cfg, dev, f32)
    return calls


# Workloads of the operations built beyond the step, timed beside it (not part
# of the step's bytes or time): LayerNorm over the channels of an NCHW tensor,
# as in ConvNeXt-T's stem and first downsampling layer (96 channels of 56x56),
# and GELU with fused dropout on a ViT-B MLP hidden activation (128 images x 197
# tokens x 3072 features).
DROPOUT_WORKLOAD = "act_dropout_gelu_f16_25216x3072"
DROPOUT_P = 0.1
DROPOUT_SEED = 2024
# and the ViT-B LayerNorm with its output (and so dy) kept in float32
F32OUT_WORKLOAD = "ln_f16_to_f32_25216x768"
# and rows too wide for the register and ring kernels (above 32768 fp16 values
# forward, 16384 backward), which take one 1024-thread CTA per row
WIDE_WORKLOAD = "ln_f16_2048x65536"
EXTRA = ("ln_cf_f16_128x96x56x56", DROPOUT_WORKLOAD, F32OUT_WORKLOAD, WIDE_WORKLOAD)


def build_extra_calls(dev, names=None):
    import torch

    calls = []

    def f32(n):
        return torch.empty(n, dtype=torch.float32, device=dev)

    if names is None or EXTRA[0] in names:
        calls += _ln_cf(EXTRA[0], 128, 96, 56 * 56, dev, f32)
    if names is None or DROPOUT_WORKLOAD in names:
        calls += _act_dropout(DROPOUT_WORKLOAD, 25216, 3072, dev)
    if names is None or F32OUT_WORKLOAD in names:
        calls += _ln_f32out(F32OUT_WORKLOAD, 25216, 768, dev, f32)
    if names is None or WIDE_WORKLOAD in names:
        calls += _ln_wide(WIDE_WORKLOAD, 2048, 65536, dev, f32)
    return calls


def _rms(cfg, dev, f32):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    calls = []
    inp = synth.row_inputs(cfg)
    x, w, dy = (inp[k].torch(dev) for k in ("x", "w", "dy"))
    y, dx, dw = torch.empty_like(x), torch.empty_like(x), torch.empty_like(w)
    rstd = f32(cfg.rows)
    ws = f32(nrm.nrm_workspace_bytes(nrm.NRM_OP_RMSNORM_BWD, cfg.rows, cfg.cols, nrm.NRM_BF16) // 4)
    calls.append(Call(cfg.name, "fwd", "row_fwd_kernel<bf16,rms>",
                      lambda x=x, w=w, y=y, r=rstd, e=cfg.eps: nrm.nrm_rmsnorm_fwd(x, w, y, r, e),
                      nbytes(x, y, w, rstd), 1, [x, w], [y, rstd]))
    calls.append(Call(cfg.name, "bwd", "row_bwd_ring_kernel<bf16,rms>+colsum",
                      lambda: nrm.nrm_rmsnorm_bwd(dy, x, w, rstd, dx, dw, ws),
                      nbytes(dy, x, w, rstd, dx, dw), 2, [dy], [dx, dw]))

    return calls


def _ln(cfg, dev, f32):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    calls = []
    inp = synth.row_inputs(cfg)
    lx, lw, lb, ldy = (inp[k].torch(dev) for k in ("x", "w", "b", "dy"))
    ly, ldx, ldw, ldb = torch.empty_like(lx), torch.empty_like(lx), torch.empty_like(lw), torch.empty_like(lb)
    lmean, lrstd = f32(cfg.rows), f32(cfg.rows)
    code = {"f32": nrm.NRM_F32, "f16": nrm.NRM_F16, "bf16": nrm.NRM_BF16}[cfg.dtype]
    lws = f32(nrm.nrm_workspace_bytes(nrm.NRM_OP_LAYERNORM_BWD, cfg.rows, cfg.cols, code) // 4)
    dt = cfg.dtype
    calls.append(Call(cfg.name, "fwd", f"row_fwd_kernel<{dt},ln>",
                      lambda e=cfg.eps: nrm.nrm_layernorm_fwd(lx, lw, lb, ly, lmean, lrstd, e),
                      nbytes(lx, lw, lb, ly, lmean, lrstd), 1, [lx, lw, lb], [ly, lmean, lrstd]))
    calls.append(Call(cfg.name, "bwd", f"row_bwd_ring_kernel<{dt},ln>+colsum",
                      lambda: nrm.nrm_layernorm_bwd(ldy, lx, lw, lmean, lrstd, ldx, ldw, ldb, lws),
                      nbytes(ldy, lx, lw, lmean, lrstd, ldx, ldw, ldb), 2, [ldy], [ldx, ldw, ldb]))

    return calls


def _bn_res_relu(cfg, dev, f32):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    calls = []
    inp = synth.bn_inputs(cfg)
    bx, bres, bw, bb, bdy = (inp[k].torch(dev) for k in ("x", "res", "w", "b", "dy"))
    brm, brv = inp["running_mean"].torch(dev), inp["running_var"].torch(dev)
    n, c, l = cfg.n, cfg.c, cfg.l
    by, bdx, bdres = torch.empty_like(bx), torch.empty_like(bx), torch.empty_like(bx)
    bsm, bsr, bdw, bdb = f32(c), f32(c), f32(c), f32(c)
    bmask = torch.empty(nrm.nrm_act_mask_words(n, c, l), dtype=torch.int32, device=dev)
    bws = nrm.batchnorm_workspace(bx)
    calls.append(Call(cfg.name, "fwd", "bn_fwd_train_kernel<f32,relu>",
                      lambda: nrm.nrm_batchnorm_fwd(bx, bres, bw, bb, by, brm, brv, bsm, bsr, bmask,
                                                    cfg.eps, cfg.momentum, True, "relu", bws),
                      nbytes(bx, bres, by, bmask, bw, bb, bsm, bsr) + 2 * nbytes(brm, brv), 1,
                      [bx, bres, bw, bb, brm, brv], [by, bmask, bsm, bsr, brm, brv]))
    calls.append(Call(cfg.name, "bwd", "bn_bwd_train_kernel<f32,relu>",
                      lambda: nrm.nrm_batchnorm_bwd(bdy, bx, bres, bw, bb, bsm, bsr, bmask, bdx, bdres,
                                                    bdw, bdb, True, "relu", bws),
                      nbytes(bdy, bx, bmask, bw, bb, bsm, bsr, bdx, bdres, bdw, bdb), 1,
                      [bdy], [bdx, bdres, bdw, bdb]))
    erm = synth.store(0.3 * synth.normal(cfg.seed, 20, c), "f32", (c,)).torch(dev)
    erv = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,)).torch(dev)
    esm, esr = f32(c), f32(c)
    eval_name = cfg.name + "_eval"
    calls.append(Call(eval_name, "fwd", "bn_fwd_eval_stream_kernel<f32,relu>",
                      lambda: nrm.nrm_batchnorm_fwd(bx, bres, bw, bb, by, erm, erv, esm, esr, bmask,
                                                    cfg.eps, cfg.momentum, False, "relu", bws),
                      nbytes(bx, bres, by, bmask, bw, bb, erm, erv, esm, esr), 1,
                      [erm, erv], [by, bmask]))
    calls.append(Call(eval_name, "bwd", "bn_bwd_eval_kernel<f32,relu>",
                      lambda: nrm.nrm_batchnorm_bwd(bdy, bx, bres, bw, bb, esm, esr, bmask, bdx, bdres,
                                                    bdw, bdb, False, "relu", bws),
                      nbytes(bdy, bx, bmask, bw, bb, esm, esr, bdx, bdres, bdw, bdb), 1,
                      [], [bdx, bdres, bdw, bdb]))

    return calls


def _bn_gelu(cfg, dev, f32):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    calls = []
    inp = synth.bn_inputs(cfg)
    gx, gw, gb, gdy = (inp[k].torch(dev) for k in ("x", "w", "b", "dy"))
    grm, grv = inp["running_mean"].torch(dev), inp["running_var"].torch(dev)
    c = cfg.c
    gy, gdx = torch.empty_like(gx), torch.empty_like(gx)
    gsm, gsr, gdw, gdb = f32(c), f32(c), f32(c), f32(c)
    gws = nrm.batchnorm_workspace(gx)
    calls.append(Call(cfg.name, "fwd", "bn_fwd_group_kernel<f16,train>",
                      lambda: nrm.nrm_batchnorm_fwd(gx, None, gw, gb, gy, grm, grv, gsm, gsr, None,
                                                    cfg.eps, cfg.momentum, True, "gelu", gws),
                      nbytes(gx, gy, gw, gb, gsm, gsr) + 2 * nbytes(grm, grv), 1,
                      [gx, gw, gb, grm, grv], [gy, gsm, gsr, grm, grv]))
    calls.append(Call(cfg.name, "bwd", "bn_bwd_group_kernel<f16,train>",
                      lambda: nrm.nrm_batchnorm_bwd(gdy, gx, None, gw, gb, gsm, gsr, None, gdx, None,
                                                    gdw, gdb, True, "gelu", gws),
                      nbytes(gdy, gx, gw, gb, gsm, gsr, gdx, gdw, gdb), 1,
                      [gdy], [gdx, gdw, gdb]))
    return calls


def _ln_cf(name, n, c, l, dev, f32, kernels=("lncf_fwd_ring_kernel<f16>", "lncf_bwd_ring_kernel<f16>+colsum")):
    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    seed = 31
    x = synth.random_tensor(seed, 1, (n, c, l), "f16", mean=0.3, std=1.5).torch(dev)
    dy = synth.random_tensor(seed, 2, (n, c, l), "f16").torch(dev)
    w = synth.store(1 + 0.1 * synth.normal(seed, 3, c), "f16", (c,)).torch(dev)
    b = synth.store(0.1 * synth.normal(seed, 4, c), "f16", (c,)).torch(dev)
    y, dx = x.new_empty(x.shape), x.new_empty(x.shape)
    dw, db = w.new_empty(c), w.new_empty(c)
    mean, rstd = f32(n * l), f32(n * l)
    ws = f32(nrm.nrm_workspace_bytes(nrm.NRM_OP_LAYERNORM_CF_BWD, n * l, c, nrm.NRM_F16) // 4)
    return [
        Call(name, "fwd", kernels[0],
             lambda: nrm.nrm_layernorm_cf_fwd(x, w, b, y, mean, rstd, 1e-6),
             nbytes(x, w, b, y, mean, rstd), 1, [x, w, b], [y, mean, rstd]),
        Call(name, "bwd", kernels[1],
             lambda: nrm.nrm_layernorm_cf_bwd(dy, x, w, mean, rstd, dx, dw, db, ws),
             nbytes(dy, x, w, mean, rstd, dx, dw, db), 2, [dy], [dx, dw, db]),
    ]


def _act_dropout(name, rows, cols, dev):
    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    seed = 37
    x = synth.random_tensor(seed, 1, (rows, cols), "f16").torch(dev)
    dy = synth.random_tensor(seed, 2, (rows, cols), "f16").torch(dev)
    y, dx = x.new_empty(x.shape), x.new_empty(x.shape)
    p, s = DROPOUT_P, DROPOUT_SEED
    return [
        Call(name, "fwd", "act_dropout_vec_kernel<f16,gelu>",
             lambda: nrm.nrm_act_dropout_fwd(x, y, "gelu", p, s), nbytes(x, y), 1, [x], [y]),
        Call(name, "bwd", "act_dropout_vec_kernel<f16,gelu,bwd>",
             lambda: nrm.nrm_act_dropout_bwd(dy, x, dx, "gelu", p, s), nbytes(dy, x, dx), 1, [dy], [dx]),
    ]


def _ln_f32out(name, rows, cols, dev, f32):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    seed = 41
    x = synth.random_tensor(seed, 1, (rows, cols), "f16", mean=0.3, std=1.5).torch(dev)
    w = synth.store(1 + 0.1 * synth.normal(seed, 2, cols), "f16", (cols,)).torch(dev)
    b = synth.store(0.1 * synth.normal(seed, 3, cols), "f16", (cols,)).torch(dev)
    dy = synth.random_tensor(seed, 4, (rows, cols), "f32").torch(dev)
    y = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    dx, dw, db = x.new_empty(x.shape), w.new_empty(cols), b.new_empty(cols)
    mean, rstd = f32(rows), f32(rows)
    ws = f32(nrm.nrm_workspace_bytes(nrm.NRM_OP_LAYERNORM_BWD, rows, cols, nrm.NRM_F16) // 4)
    return [
        Call(name, "fwd", "row_fwd_kernel<f16,ln,f32 out>",
             lambda: nrm.nrm_layernorm_fwd_ex(x, w, b, y, mean, rstd, 1e-6),
             nbytes(x, w, b, y, mean, rstd), 1, [x, w, b], [y, mean, rstd]),
        Call(name, "bwd", "row_bwd_ring_kernel<f16,ln,f32 dy>+colsum",
             lambda: nrm.nrm_layernorm_bwd_ex(dy, x, w, mean, rstd, dx, dw, db, ws),
             nbytes(dy, x, w, mean, rstd, dx, dw, db), 2, [dy], [dx, dw, db]),
    ]


def _ln_wide(name, rows, cols, dev, f32):
    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    seed = 43
    x = synth.random_tensor(seed, 1, (rows, cols), "f16", mean=0.3, std=1.5).torch(dev)
    w = synth.store(1 + 0.1 * synth.normal(seed, 2, cols), "f16", (cols,)).torch(dev)
    b = synth.store(0.1 * synth.normal(seed, 3, cols), "f16", (cols,)).torch(dev)
    dy = synth.random_tensor(seed, 4, (rows, cols), "f16").torch(dev)
    y, dx, dw, db = x.new_empty(x.shape), x.new_empty(x.shape), w.new_empty(cols), b.new_empty(cols)
    mean, rstd = f32(rows), f32(rows)
    ws = f32(nrm.nrm_workspace_bytes(nrm.NRM_OP_LAYERNORM_BWD, rows, cols, nrm.NRM_F16) // 4)
    return [
        Call(name, "fwd", "row_fwd_wide_kernel<f16,ln>",
             lambda: nrm.nrm_layernorm_fwd(x, w, b, y, mean, rstd, 1e-5),
             nbytes(x, w, b, y, mean, rstd), 1, [x, w, b], [y, mean, rstd]),
        Call(name, "bwd", "row_bwd_wide_sums+cols_kernel<f16,ln>+colsum",
             lambda: nrm.nrm_layernorm_bwd(dy, x, w, mean, rstd, dx, dw, db, ws),
             nbytes(dy, x, w, mean, rstd, dx, dw, db), 3, [dy], [dx, dw, db]),
    ]


# Shapes that take the paths no bench workload reaches, run only by
# profile_case for their ncu captures: rows that are not 16-byte multiples (the
# scalar register kernels), BatchNorm eval with 8192 channels (a 64 KB
# coefficient table in the streamed eval forward; the ring eval backward), channels-first planes that are not 16-byte multiples (the register
# kernels), an unaligned activation-dropout tensor (the scalar kernel) and
# unaligned rows too wide for the register kernels (the one-kernel wide
# backward).
PROFILE_ONLY = ("ln_f16_65536x1023", "bn_f32_64x8192x8x8_eval", "ln_cf_f16_2048x768x7x7",
                "act_dropout_gelu_f16_unaligned_67108863", "ln_f16_2048x65537")


def build_profile_calls(dev, names):
    import torch

    def f32(n):
        return torch.empty(n, dtype=torch.float32, device=dev)

    calls = []
    if "ln_f16_65536x1023" in names:
        calls += _ln_plain("ln_f16_65536x1023", 65536, 1023, dev, f32,
                           ("row_fwd_kernel<f16,ln,scalar>", "row_bwd_kernel<f16,ln,scalar>+colsum"))
    if "bn_f32_64x8192x8x8_eval" in names:
        calls += _bn_eval_plain("bn_f32_64x8192x8x8_eval", 64, 8192, 64, dev, f32)
    if "ln_cf_f16_2048x768x7x7" in names:
        calls += _ln_cf("ln_cf_f16_2048x768x7x7", 2048, 768, 49, dev, f32,
                        ("lncf_fwd_kernel<f16>", "lncf_bwd_kernel<f16>+colsum"))
    if "act_dropout_gelu_f16_unaligned_67108863" in names:
        calls += _act_dropout_unaligned("act_dropout_gelu_f16_unaligned_67108863", 67108863, dev)
    if "ln_f16_2048x65537" in names:
        calls += _ln_plain("ln_f16_2048x65537", 2048, 65537, dev, f32,
                           ("row_fwd_wide_kernel<f16,ln,scalar>", "row_bwd_wide_kernel<f16,ln,scalar>+colsum"))
    return calls


def _ln_plain(name, rows, cols, dev, f32, kernels):
    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    seed = 47
    x = synth.random_tensor(seed, 1, (rows, cols), "f16", mean=0.3, std=1.5).torch(dev)
    w = synth.store(1 + 0.1 * synth.normal(seed, 2, cols), "f16", (cols,)).torch(dev)
    b = synth.store(0.1 * synth.normal(seed, 3, cols), "f16", (cols,)).torch(dev)
    dy = synth.random_tensor(seed, 4, (rows, cols), "f16").torch(dev)
    y, dx, dw, db = x.new_empty(x.shape), x.new_empty(x.shape), w.new_empty(cols), b.new_empty(cols)
    mean, rstd = f32(rows), f32(rows)
    ws = f32(nrm.nrm_workspace_bytes(nrm.NRM_OP_LAYERNORM_BWD, rows, cols, nrm.NRM_F16) // 4)
    return [
        Call(name, "fwd", kernels[0], lambda: nrm.nrm_layernorm_fwd(x, w, b, y, mean, rstd, 1e-5),
             nbytes(x, w, b, y, mean, rstd), 1, [x, w, b], [y, mean, rstd]),
        Call(name, "bwd", kernels[1], lambda: nrm.nrm_layernorm_bwd(dy, x, w, mean, rstd, dx, dw, db, ws),
             nbytes(dy, x, w, mean, rstd, dx, dw, db), 2, [dy], [dx, dw, db]),
    ]


def _bn_eval_plain(name, n, c, l, dev, f32):
    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    seed = 53
    x = synth.random_tensor(seed, 1, (n, c, l), "f32", mean=0.2, std=1.4).torch(dev)
    dy = synth.random_tensor(seed, 2, (n, c, l), "f32").torch(dev)
    w = synth.store(1 + 0.2 * synth.normal(seed, 3, c), "f32", (c,)).torch(dev)
    b = synth.store(0.2 * synth.normal(seed, 4, c), "f32", (c,)).torch(dev)
    rm = synth.store(0.3 * synth.normal(seed, 5, c), "f32", (c,)).torch(dev)
    rv = synth.store(0.5 + synth.uniform(seed, 6, c), "f32", (c,)).torch(dev)
    y, dx = x.new_empty(x.shape), x.new_empty(x.shape)
    sm, sr, dw, db = f32(c), f32(c), f32(c), f32(c)
    ws = nrm.batchnorm_workspace(x)
    return [
        Call(name, "fwd", "bn_fwd_eval_stream_kernel<f32,none>",
             lambda: nrm.nrm_batchnorm_fwd(x, None, w, b, y, rm, rv, sm, sr, None, 1e-5, 0.1, False, "none", ws),
             nbytes(x, y, w, b, rm, rv, sm, sr), 1, [x, w, b, rm, rv], [y, sm, sr]),
        Call(name, "bwd", "bn_bwd_eval_kernel<f32,none>",
             lambda: nrm.nrm_batchnorm_bwd(dy, x, None, w, b, sm, sr, None, dx, None, dw, db, False, "none", ws),
             nbytes(dy, x, w, b, sm, sr, dx, dw, db), 1, [dy], [dx, dw, db]),
    ]


def _act_dropout_unaligned(name, count, dev):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import synth
    seed = 59
    # views one element into their buffers: not 16-byte aligned
    xb = torch.empty(count + 1, dtype=torch.float16, device=dev)
    dyb = torch.empty(count + 1, dtype=torch.float16, device=dev)
    xb[1:] = synth.random_tensor(seed, 1, (count,), "f16").torch(dev)
    dyb[1:] = synth.random_tensor(seed, 2, (count,), "f16").torch(dev)
    x, dy = xb[1:], dyb[1:]
    y = torch.empty(count + 1, dtype=torch.float16, device=dev)[1:]
    dx = torch.empty(count + 1, dtype=torch.float16, device=dev)[1:]
    p, s = DROPOUT_P, DROPOUT_SEED
    return [
        Call(name, "fwd", "act_dropout_scalar_kernel<f16,gelu>",
             lambda: nrm.nrm_act_dropout_fwd(x, y, "gelu", p, s), nbytes(x, y), 1, [x], [y]),
        Call(name, "bwd", "act_dropout_scalar_kernel<f16,gelu,bwd>",
             lambda: nrm.nrm_act_dropout_bwd(dy, x, dx, "gelu", p, s), nbytes(dy, x, dx), 1, [dy], [dx]),
    ]
