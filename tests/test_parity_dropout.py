"""The activation with fused dropout through libnorm's C ABI against the CPU
oracle: keep flags bit-exact (an integer decision), values element by element
within the dtype's tolerance; the 16-byte vector path with a ragged tail, the
scalar path for unaligned tensors, in-place calls, p = 0 and p = 1, and the
benchmarked workload itself in windows at its start, middle and end."""
import numpy as np
import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import TOL, assert_close, host

pytestmark = pytest.mark.gpu

ACTS = ["none", "relu", "gelu", "silu", "mish", "leaky_relu", "elu", "sigmoid", "celu", "selu", "relu6",
        "hardtanh"]
ACT_CODE = {a: i for i, a in enumerate(ACTS)}
ACT_PARAM = {"leaky_relu": 0.05, "elu": 1.3, "celu": 0.7}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()


def _run(x, dy, act, p, seed, offset=0):
    """x, dy: synth tensors; offset > 0 runs on views that start `offset`
    elements into a larger buffer (not 16-byte aligned for offset % 8 != 0)."""
    n = x.shape[0]
    xb = torch.zeros(n + offset, dtype=x.torch("cpu").dtype, device="cuda")
    dyb = torch.zeros_like(xb)
    xb[offset:] = x.torch("cuda")
    dyb[offset:] = dy.torch("cuda")
    xt, dyt = xb[offset:], dyb[offset:]
    y = torch.empty_like(xb)[offset:]
    dx = torch.empty_like(xb)[offset:]
    prm = ACT_PARAM.get(act, 0.0)
    nrm.nrm_act_dropout_fwd(xt, y, act, p, seed, act_param=prm)
    nrm.nrm_act_dropout_bwd(dyt, xt, dx, act, p, seed, act_param=prm)
    nrm.nrm_sync_status()
    return host(y), host(dx)


def _check(orc, x, dy, act, p, seed, dtype, tag, offset=0):
    y, dx = _run(x, dy, act, p, seed, offset)
    prm = ACT_PARAM.get(act, 0.0)
    yo = orc.act_dropout_fwd(x.f64(), ACT_CODE[act], p, seed, act_param=prm)
    dxo = orc.act_dropout_bwd(dy.f64(), x.f64(), ACT_CODE[act], p, seed, act_param=prm)
    keep = orc.dropout_mask(x.shape[0], p, seed).astype(bool)
    # dropped elements are exactly zero on both passes
    assert not y[~keep].any(), f"{tag}: nonzero y at dropped elements"
    assert not dx[~keep].any(), f"{tag}: nonzero dx at dropped elements"
    assert_close(y, yo, TOL[dtype], tag + " y")
    assert_close(dx, dxo, TOL[dtype], tag + " dx")
    return keep, y


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("act", ACTS)
def test_act_dropout(orc, dtype, act):
    n = 100_003  # whole vectors and a ragged tail
    x = synth.random_tensor(7, 1, (n,), dtype, std=2.0)
    dy = synth.random_tensor(7, 2, (n,), dtype)
    _check(orc, x, dy, act, 0.1, 1234, dtype, f"{act} {dtype}")


def test_dropout_mask_bit_exact(orc):
    # act none on nonzero inputs: y != 0 exactly where the element is kept
    n = 65_541
    x = synth.store(np.abs(synth.normal(3, 1, n)) + 0.5, "f32", (n,))
    dy = synth.random_tensor(3, 2, (n,), "f32")
    for p, seed in ((0.5, 0), (0.9, 65535), (0.05, 0xDEADBEEF)):
        keep, y = _check(orc, x, dy, "none", p, seed, "f32", f"mask p={p}")
        assert ((y != 0) == keep).all(), f"keep flags differ for p={p}, seed={seed}"


def test_gelu_dense_grid_fp32(orc):
    # GELU and GELU' in fp32 on a dense grid of z in [-12, 12] (p = 0: y = GELU(z),
    # dx = GELU'(z) for dy = 1) against the oracle's exact values.  The kernels
    # take Phi from the erfc approximation of Abramowitz and Stegun 7.1.26 (erf
    # within 1.5e-7): the bound below is that, times |z|, plus fp32 rounding of
    # the reciprocal, exponential and products, and is 10x tighter than the
    # fp32 parity tolerance.
    z = np.concatenate([np.linspace(-12.0, 12.0, 1_200_001), [0.0, 1e-30, -1e-30, 1e-6, -1e-6, 40.0, -40.0]])
    x = synth.store(z, "f32", z.shape)
    dy = synth.store(np.ones_like(z), "f32", z.shape)
    y, dx = _run(x, dy, "gelu", 0.0, 1)
    zf = x.f64()
    yo = orc.act_dropout_fwd(zf, ACT_CODE["gelu"], 0.0, 1)
    dxo = orc.act_dropout_bwd(dy.f64(), zf, ACT_CODE["gelu"], 0.0, 1)
    bound = 1e-6 * np.maximum(1.0, np.abs(zf))
    ey = np.abs(y - yo)
    edx = np.abs(dx - dxo)
    assert (ey <= bound).all(), f"GELU: max error {ey.max():.3g} at z = {zf[ey.argmax()]}"
    assert (edx <= bound).all(), f"GELU': max error {edx.max():.3g} at z = {zf[edx.argmax()]}"


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("act", ["relu6", "hardtanh"])
def test_clamp_activations_at_their_ends(orc, dtype, act):
    # values across both clamps with every end present exactly (0, 6, -1, 1 and
    # the 1/256 grid on [-8, 8] are exact in fp16): y and dx against the oracle,
    # the derivative exactly 0 at the ends and nonzero strictly inside
    lo, hi = {"relu6": (0.0, 6.0), "hardtanh": (-1.0, 1.0)}[act]
    z = np.concatenate([np.linspace(-8.0, 8.0, 4097), np.repeat([lo, hi], 64)])
    x = synth.store(z, dtype, z.shape)
    dy = synth.store(np.ones_like(z), dtype, z.shape)
    keep, y = _check(orc, x, dy, act, 0.2, 31, dtype, f"{act} {dtype}")
    _, dx = _run(x, dy, act, 0.2, 31)
    xv = x.f64()
    assert not dx[(xv == lo) | (xv == hi)].any(), f"{act}: derivative at the ends must be 0"
    inside = (xv > lo) & (xv < hi)
    assert (dx[inside & keep] != 0).all() and not dx[~inside].any(), f"{act}: derivative support"
    assert (y[keep & (xv >= hi)] == y[keep & (xv >= hi)].max()).all(), f"{act}: upper clamp"


@pytest.mark.parametrize("p", [0.0, 1.0])
def test_dropout_extremes(orc, p):
    n = 4099
    x = synth.random_tensor(5, 1, (n,), "bf16")
    dy = synth.random_tensor(5, 2, (n,), "bf16")
    keep, _ = _check(orc, x, dy, "gelu", p, 77, "bf16", f"p={p}")
    assert keep.all() if p == 0.0 else not keep.any()


@pytest.mark.parametrize("offset", [1, 3])
def test_dropout_unaligned_scalar_path(orc, offset):
    n = 20_011
    x = synth.random_tensor(6, 1, (n,), "f16")
    dy = synth.random_tensor(6, 2, (n,), "f16")
    _check(orc, x, dy, "silu", 0.3, 99, "f16", f"unaligned +{offset}", offset=offset)


@pytest.mark.parametrize("n", [1, 3, 7, 8, 9, 33])
def test_dropout_tiny(orc, n):
    x = synth.random_tensor(8, 1, (n,), "f16")
    dy = synth.random_tensor(8, 2, (n,), "f16")
    _check(orc, x, dy, "mish", 0.25, 5, "f16", f"n={n}")


def test_dropout_in_place(orc):
    n = 10_000
    x = synth.random_tensor(9, 1, (n,), "f32", std=2.0)
    dy = synth.random_tensor(9, 2, (n,), "f32")
    t = x.torch("cuda")
    nrm.nrm_act_dropout_fwd(t, t, "relu", 0.2, 42)
    g = dy.torch("cuda")
    xt = x.torch("cuda")
    nrm.nrm_act_dropout_bwd(g, xt, g, "relu", 0.2, 42)
    nrm.nrm_sync_status()
    assert_close(host(t), orc.act_dropout_fwd(x.f64(), 1, 0.2, 42), TOL["f32"], "in-place y")
    assert_close(host(g), orc.act_dropout_bwd(dy.f64(), x.f64(), 1, 0.2, 42), TOL["f32"], "in-place dx")


def test_dropout_empty():
    t = torch.empty(0, device="cuda", dtype=torch.float16)
    nrm.nrm_act_dropout_fwd(t, t, "gelu", 0.5, 1)
    nrm.nrm_act_dropout_bwd(t, t, t, "gelu", 0.5, 1)
    nrm.nrm_sync_status()


def test_dropout_bench_size_windows(orc):
    # the benchmarked workload (GELU + dropout p = 0.1 on fp16 [25216, 3072],
    # the inputs the bench builds) in the bench's launch configuration; the
    # oracle checks windows at the start, the middle and the end
    from normalization_layernorm_rmsnorm_gb300 import workloads
    calls = workloads.build_extra_calls(torch.device("cuda", 0), {workloads.DROPOUT_WORKLOAD})
    fwd, bwd = calls
    fwd.fn()
    bwd.fn()
    nrm.nrm_sync_status()
    x, dy = fwd.inputs[0], bwd.inputs[0]
    y, dx = fwd.outputs[0], bwd.outputs[0]
    n = x.numel()
    p, seed = workloads.DROPOUT_P, workloads.DROPOUT_SEED
    w = 1 << 20
    for first in (0, n // 2 - 12345, n - w):
        xs = host(x.view(-1)[first:first + w])
        dys = host(dy.view(-1)[first:first + w])
        assert_close(host(y.view(-1)[first:first + w]), orc.act_dropout_fwd(xs, 2, p, seed, first=first),
                     TOL["f16"], f"bench window {first} y")
        assert_close(host(dx.view(-1)[first:first + w]),
                     orc.act_dropout_bwd(dys, xs, 2, p, seed, first=first), TOL["f16"], f"bench window {first} dx")
