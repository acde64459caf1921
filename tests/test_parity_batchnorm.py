"""BatchNorm (training and eval, with fused residual and ReLU / GELU) through
libnorm's C ABI against the CPU oracle, element by element: the full-size
workloads (ResNet BatchNorm2d fp32 [256,64,56,56] + residual + ReLU, fp16
[128,512,7,7] + GELU) and odd shapes that exercise every path (vector and
scalar, clusters of 1 to 16 CTAs, channels larger than the shared-memory
staging budget, ragged mask words)."""
import numpy as np
import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import compare_bn, oracle_bn, run_bn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()


@pytest.mark.parametrize("training", [True, False], ids=["train", "eval"])
@pytest.mark.parametrize("name", ["bn_f32_256x64x56x56_res_relu", "bn_f16_128x512x7x7_gelu"])
def test_bn_workloads_full_size(orc, name, training):
    cfg = synth.CONFIGS[name]
    inp = synth.bn_inputs(cfg)
    if not training:
        # eval reads running statistics: use non-trivial ones
        c = cfg.c
        inp["running_mean"] = synth.store(0.3 * synth.normal(cfg.seed, 20, c), "f32", (c,))
        inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
    use_mask = cfg.act == "relu"
    got = run_bn(inp, cfg.dtype, cfg.eps, cfg.momentum, training, cfg.act, cfg.residual, use_mask)
    want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, training, cfg.act, cfg.residual)
    compare_bn(got, want, cfg.dtype, training, cfg.act, f"{name} training={training}")


ODD = [
    # (n, c, l)
    (2, 3, 1),
    (3, 5, 49),
    (4, 2, 70),
    (1, 3, 300),
    (5, 7, 33),
    (8, 4, 64),
    (64, 3, 3136),      # vector path, several CTAs per channel
    (128, 2, 12544),    # fp32 channel of 6.4 MB: larger than the staging budget
    (3, 1, 100003),     # one channel, odd length
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", ODD, ids=[f"{n}x{c}x{l}" for n, c, l in ODD])
def test_bn_odd_shapes(orc, dtype, shape):
    n, c, l = shape
    idx = ODD.index(shape)
    acts = ["none", "relu", "gelu", "silu", "mish"]
    for training in (True, False):
        act = acts[(idx + 2 * int(training)) % len(acts)]
        with_res = (idx % 2 == 0)
        cfg = synth.BnConfig("odd", n, c, l, dtype, 1e-5, 0.1, seed=200 + idx, act=act,
                             residual=with_res, x_kind="offset_scale", w_std=0.2, b_std=0.2)
        inp = synth.bn_inputs(cfg)
        if not training:
            inp["running_mean"] = synth.store(0.2 * synth.normal(cfg.seed, 20, c), "f32", (c,))
            inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
        use_mask = act == "relu" and idx % 3 != 0
        got = run_bn(inp, dtype, cfg.eps, cfg.momentum, training, act, with_res, use_mask)
        want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, training, act, with_res)
        compare_bn(got, want, dtype, training, act,
                   f"bn {dtype} {shape} training={training} act={act} res={with_res} mask={use_mask}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bn_eval_forward_both_paths(orc, dtype):
    # the eval forward streams through registers with a per-CTA table of up to
    # 16384 channels' coefficients in dynamic shared memory (above 48 KB, 6144
    # channels, with the opt-in size); more channels take the ring kernel.  All
    # three, with the ReLU mask and a residual, with a ragged last block per segment
    for n, c, l in ((3, 4096, 40), (2, 8200, 24), (2, 16400, 8)):
        cfg = synth.BnConfig("evc", n, c, l, dtype, 1e-5, 0.1, seed=640 + c % 97, act="relu",
                             residual=True, x_kind="offset_scale", w_std=0.2, b_std=0.2)
        inp = synth.bn_inputs(cfg)
        inp["running_mean"] = synth.store(0.2 * synth.normal(cfg.seed, 20, c), "f32", (c,))
        inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
        got = run_bn(inp, dtype, cfg.eps, cfg.momentum, False, "relu", True, True)
        want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, False, "relu", True)
        compare_bn(got, want, dtype, False, "relu", f"bn eval {dtype} [{n},{c},{l}]")


@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_bn_without_affine_or_running_stats(orc, act):
    n, c, l = 6, 5, 200
    cfg = synth.BnConfig("noaff", n, c, l, "f32", 1e-5, 0.1, seed=300, act=act, residual=True,
                         x_kind="offset_scale")
    inp = synth.bn_inputs(cfg)
    x = inp["x"].torch("cuda")
    res = inp["res"].torch("cuda")
    dy = inp["dy"].torch("cuda")
    y = torch.empty_like(x)
    sm = torch.empty(c, device="cuda")
    sr = torch.empty(c, device="cuda")
    ws = nrm.batchnorm_workspace(x)
    nrm.nrm_batchnorm_fwd(x, res, None, None, y, None, None, sm, sr, None, 1e-5, 0.1, True, act, ws)
    dx = torch.empty_like(x)
    nrm.nrm_batchnorm_bwd(dy, x, res, None, None, sm, sr, None, dx, None, None, None, True, act, ws)
    nrm.nrm_sync_status()
    want = oracle_bn(orc, inp, 1e-5, 0.1, True, act, True, with_affine=False)
    yo = want["fwd"]["y"]
    ok = ~want["amb"] if "amb" in want else np.ones_like(yo, dtype=bool)
    err = np.abs(y.double().cpu().numpy() - yo)
    assert (err[ok] <= 1e-5 + 1e-5 * np.abs(yo[ok])).all()
    dxo = want["bwd"][0]
    err = np.abs(dx.double().cpu().numpy() - dxo)
    assert (err[ok] <= 1e-5 + 1e-5 * np.abs(dxo[ok])).all()


def test_bn_running_stats_closed_form():
    # from running_mean 0, running_var 1 and momentum m: rm = m*mean, rv = (1-m) + m*var_unbiased
    n, c, l = 16, 3, 500
    cfg = synth.BnConfig("ema", n, c, l, "f32", 1e-5, 0.1, seed=400, act="none", residual=False,
                         x_kind="offset_scale")
    inp = synth.bn_inputs(cfg)
    x = inp["x"].torch("cuda")
    y = torch.empty_like(x)
    rm = torch.zeros(c, device="cuda")
    rv = torch.ones(c, device="cuda")
    nrm.nrm_batchnorm_fwd(x, None, None, None, y, rm, rv, None, None, None, 1e-5, 0.1, True, "none",
                          nrm.batchnorm_workspace(x))
    nrm.nrm_sync_status()
    xc = inp["x"].f64().transpose(1, 0, 2).reshape(c, -1)
    np.testing.assert_allclose(rm.double().cpu().numpy(), 0.1 * xc.mean(1), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(rv.double().cpu().numpy(), 0.9 + 0.1 * xc.var(1, ddof=1), rtol=1e-5)


GROUPS = [
    # (dtype, n, c, l): segments too short for 16-byte access; G channels of a
    # sample form an aligned span (G = 16 / gcd(l*size, 16))
    ("f16", 16, 16, 49),     # G = 8, two groups
    ("bf16", 9, 8, 7),       # a 16-byte vector spans up to three channels
    ("f32", 33, 12, 9),      # G = 4; a cluster of 8 where the last CTA has no samples
    ("f32", 4, 2, 70),       # G = 2
    ("f16", 300, 8, 25),     # one group, many samples per CTA
    ("bf16", 2048, 8, 49),   # forward fits the group path, backward falls back
]


@pytest.mark.parametrize("case", GROUPS, ids=[f"{d}-{n}x{c}x{l}" for d, n, c, l in GROUPS])
def test_bn_channel_groups(orc, case):
    dtype, n, c, l = case
    idx = GROUPS.index(case)
    for training in (True, False):
        for act, with_res, use_mask in (("relu", True, True), ("gelu", False, False), ("none", True, False),
                                        ("relu", False, False), ("silu", True, False), ("mish", False, False)):
            cfg = synth.BnConfig("grp", n, c, l, dtype, 1e-5, 0.1, seed=500 + idx, act=act,
                                 residual=with_res, x_kind="offset_scale", w_std=0.2, b_std=0.2)
            inp = synth.bn_inputs(cfg)
            if not training:
                inp["running_mean"] = synth.store(0.2 * synth.normal(cfg.seed, 20, c), "f32", (c,))
                inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
            got = run_bn(inp, dtype, cfg.eps, cfg.momentum, training, act, with_res, use_mask)
            want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, training, act, with_res)
            compare_bn(got, want, dtype, training, act,
                       f"bn {dtype} {case} training={training} act={act} res={with_res} mask={use_mask}")


@pytest.mark.parametrize("act", ["silu", "mish"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bn_silu_mish_vector_path(orc, act, dtype):
    # the ring kernels with z recomputed in the backward, with and without a residual
    n, c, l = 32, 6, 1568
    for training in (True, False):
        for with_res in (False, True):
            cfg = synth.BnConfig("act", n, c, l, dtype, 1e-5, 0.1, seed=700 + int(with_res), act=act,
                                 residual=with_res, x_kind="offset_scale", w_std=0.2, b_std=0.2)
            inp = synth.bn_inputs(cfg)
            if not training:
                inp["running_mean"] = synth.store(0.2 * synth.normal(cfg.seed, 20, c), "f32", (c,))
                inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
            got = run_bn(inp, dtype, cfg.eps, cfg.momentum, training, act, with_res, False)
            want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, training, act, with_res)
            compare_bn(got, want, dtype, training, act, f"bn {dtype} {act} training={training} res={with_res}")


LEAKY_ELU = [
    # (dtype, n, c, l): the ring kernels, the channel-group kernels (7x7 maps), the scalar path
    ("f32", 32, 6, 1568),
    ("bf16", 32, 6, 1568),
    ("f16", 16, 24, 49),
    ("f32", 5, 7, 33),
]


@pytest.mark.parametrize("act", ["leaky_relu", "elu", "sigmoid", "celu", "selu", "relu6", "hardtanh"])
@pytest.mark.parametrize("case", LEAKY_ELU, ids=[f"{d}-{n}x{c}x{l}" for d, n, c, l in LEAKY_ELU])
def test_bn_leaky_relu_elu(orc, act, case):
    # the activations with a parameter (slope 0.05, alpha 1.3 / 0.7) and the
    # run-time dispatched ones (sigmoid, CELU, SELU), z recomputed in the backward
    dtype, n, c, l = case
    for training in (True, False):
        for with_res in (False, True):
            cfg = synth.BnConfig("actp", n, c, l, dtype, 1e-5, 0.1, seed=750 + int(with_res), act=act,
                                 residual=with_res, x_kind="offset_scale", w_std=0.2, b_std=0.2)
            inp = synth.bn_inputs(cfg)
            if not training:
                inp["running_mean"] = synth.store(0.2 * synth.normal(cfg.seed, 20, c), "f32", (c,))
                inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
            got = run_bn(inp, dtype, cfg.eps, cfg.momentum, training, act, with_res, False)
            want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, training, act, with_res)
            compare_bn(got, want, dtype, training, act,
                       f"bn {dtype} [{n},{c},{l}] {act} training={training} res={with_res}")


BN1D = [("f32", 4096, 64), ("f16", 4096, 64), ("bf16", 300, 24), ("f32", 50000, 8)]


@pytest.mark.parametrize("case", BN1D, ids=[f"{d}-{n}x{c}" for d, n, c in BN1D])
def test_bn1d(orc, case):
    # BatchNorm1d on [N, C] is [n, c, l] with l = 1: a sample's channels are
    # contiguous, so G channels form one 16-byte span (the channel-group path,
    # or the scalar path when a group does not fit in shared memory)
    dtype, n, c = case
    for training in (True, False):
        for act, with_res, use_mask in (("relu", True, True), ("none", False, False), ("silu", True, False)):
            cfg = synth.BnConfig("bn1d", n, c, 1, dtype, 1e-5, 0.1, seed=900 + n + c, act=act,
                                 residual=with_res, x_kind="offset_scale", w_std=0.2, b_std=0.2)
            inp = synth.bn_inputs(cfg)
            if not training:
                inp["running_mean"] = synth.store(0.2 * synth.normal(cfg.seed, 20, c), "f32", (c,))
                inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
            got = run_bn(inp, dtype, cfg.eps, cfg.momentum, training, act, with_res, use_mask)
            want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, training, act, with_res)
            compare_bn(got, want, dtype, training, act,
                       f"bn1d {dtype} [{n},{c}] training={training} act={act} res={with_res}")
