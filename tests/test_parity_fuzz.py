"""Seeded random shapes through libnorm's C ABI against the CPU oracle, element
by element, beside the hand-picked shapes of the other parity tests: row norms
with widths from 1 to 70000 (every kernel family: register, ring, wide,
scalar), also with float32 output and RMSNorm with a bias; BatchNorm with
every activation, residual and mask choice in both modes; channels-first
LayerNorm; and the activation with fused dropout at any length, probability
and pointer offset.  Each case draws its parameters from
its own seed, so a failure names a reproducible case; the comparisons and
their tolerances are those of the other parity tests."""
import math

import numpy as np
import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import compare_bn, compare_row, oracle_bn, oracle_row, run_bn, run_row
import test_parity_dropout as drop
import test_parity_layernorm_cf as cf
import test_parity_rownorm as rn

pytestmark = pytest.mark.gpu

DTYPES = ("f32", "f16", "bf16")
BN_ACTS = ("none", "relu", "gelu", "silu", "mish", "leaky_relu", "elu", "sigmoid", "celu", "selu",
           "relu6", "hardtanh")
MAX_ELEMS = 1 << 21  # per tensor: the oracle finishes each case in well under a second


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()


def _log_uniform(r, lo, hi):
    """An integer in [lo, hi], uniform in log scale."""
    return int(min(hi, max(lo, round(math.exp(r.uniform(math.log(lo), math.log(hi + 1)))))))


@pytest.mark.parametrize("case", range(48))
def test_fuzz_row_norms(orc, case):
    r = np.random.default_rng(7100 + case)
    kind = ("layernorm", "rmsnorm")[case % 2]
    dtype = DTYPES[(case // 2) % 3]
    cols = _log_uniform(r, 1, 70000)
    rows = _log_uniform(r, 1, max(1, min(20000, MAX_ELEMS // cols)))
    affine = bool(r.random() < 0.8)
    eps = float(r.choice([1e-6, 1e-5, 1e-3]))
    cfg = synth.RowConfig("fuzz", kind, rows, cols, dtype, eps, seed=7100 + case,
                          x_mean=float(r.uniform(-1, 1)), x_std=float(r.uniform(0.3, 3)),
                          affine=affine)
    inp = synth.row_inputs(cfg)
    got = run_row(kind, inp, dtype, eps, with_w=affine, with_b=affine, want_dw=affine, want_db=affine)
    want = oracle_row(orc, kind, inp, eps, with_w=affine, with_b=affine)
    compare_row(got, want, dtype, f"fuzz {case}: {kind} {dtype} [{rows},{cols}] affine={affine} eps={eps}")


@pytest.mark.parametrize("case", range(16))
def test_fuzz_row_f32_output(orc, case):
    # a 16-bit x with y and dy in float32 (the _ex entry points)
    r = np.random.default_rng(7500 + case)
    kind = ("layernorm", "rmsnorm")[case % 2]
    dtype = ("f16", "bf16")[(case // 2) % 2]
    cols = _log_uniform(r, 1, 70000)
    rows = _log_uniform(r, 1, max(1, min(20000, MAX_ELEMS // cols)))
    rn.check_f32_output(orc, kind, dtype, rows, cols, 7500 + case)


@pytest.mark.parametrize("case", range(12))
def test_fuzz_rmsnorm_bias(orc, case):
    r = np.random.default_rng(7600 + case)
    dtype = DTYPES[case % 3]
    cols = _log_uniform(r, 1, 70000)
    rows = _log_uniform(r, 1, max(1, min(20000, MAX_ELEMS // cols)))
    rn.check_rmsnorm_bias(orc, dtype, rows, cols, 7600 + case)


@pytest.mark.parametrize("case", range(48))
def test_fuzz_batchnorm(orc, case):
    # every activation with every dtype; channels of up to 2^21 elements (several CTAs each)
    r = np.random.default_rng(7200 + case)
    dtype = DTYPES[(case // len(BN_ACTS)) % 3]
    act = BN_ACTS[case % len(BN_ACTS)]
    l = _log_uniform(r, 1, 12544)
    c = _log_uniform(r, 1, 300)
    n = _log_uniform(r, 1, max(1, min(256, MAX_ELEMS // (c * l))))
    training = bool(r.random() < 0.6)
    if training and n * l < 2:
        l = 2  # training needs two values per channel
    with_res = bool(r.random() < 0.5)
    use_mask = act == "relu" and bool(r.random() < 0.7)
    cfg = synth.BnConfig("fuzz", n, c, l, dtype, 1e-5, float(r.uniform(0, 1)), seed=7200 + case, act=act,
                         residual=with_res, x_kind="offset_scale", w_std=0.2, b_std=0.2)
    inp = synth.bn_inputs(cfg)
    if not training:
        inp["running_mean"] = synth.store(0.2 * synth.normal(cfg.seed, 20, c), "f32", (c,))
        inp["running_var"] = synth.store(0.5 + synth.uniform(cfg.seed, 21, c), "f32", (c,))
    got = run_bn(inp, dtype, cfg.eps, cfg.momentum, training, act, with_res, use_mask)
    want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, training, act, with_res)
    compare_bn(got, want, dtype, training, act,
               f"fuzz {case}: bn {dtype} [{n},{c},{l}] training={training} act={act} res={with_res} "
               f"mask={use_mask}")


@pytest.mark.parametrize("case", range(24))
def test_fuzz_layernorm_channels_first(orc, case):
    r = np.random.default_rng(7300 + case)
    dtype = DTYPES[case % 3]
    c = _log_uniform(r, 1, 1200)
    l = _log_uniform(r, 1, 4000)
    n = _log_uniform(r, 1, max(1, min(16, MAX_ELEMS // (c * l))))
    affine = bool(r.random() < 0.8)
    x, dy, w, b = cf._inputs(n, c, l, dtype, seed=7300 + case, affine=affine)
    cf._check(orc, x, dy, w, b, dtype, 1e-6, f"fuzz {case}: cf {dtype} [{n},{c},{l}] affine={affine}")


@pytest.mark.parametrize("case", range(36))
def test_fuzz_activation_dropout(orc, case):
    r = np.random.default_rng(7400 + case)
    dtype = DTYPES[(case // len(drop.ACTS)) % 3]
    act = drop.ACTS[case % len(drop.ACTS)]
    count = _log_uniform(r, 1, 3 << 20)
    p = float(r.choice([0.0, 1.0, r.uniform(0, 1)], p=[0.1, 0.1, 0.8]))
    seed = int(r.integers(0, 2**32))
    offset = int(r.integers(0, 8)) if r.random() < 0.3 else 0
    x = synth.random_tensor(7400 + case, 1, (count,), dtype, std=2.0)
    dy = synth.random_tensor(7400 + case, 2, (count,), dtype)
    drop._check(orc, x, dy, act, p, seed, dtype,
                f"fuzz {case}: {act} {dtype} count={count} p={p} seed={seed} offset={offset}", offset=offset)
