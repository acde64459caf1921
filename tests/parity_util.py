"""Helpers for the GPU parity tests: run libnorm through its C ABI and the CPU
oracle on the same seeded inputs and compare element by element.

Tolerances (|gpu - oracle| <= atol + rtol*|oracle|):
  * float32 workloads' outputs and gradients, and every saved statistic
    (mean, rstd, running statistics): atol 1e-5, rtol 1e-5;
  * float16 / bfloat16 workloads' outputs and gradients: atol 2e-2, rtol 1e-2.
  BatchNorm dw/db are float32 tensors whatever the activation dtype and take
  the float32 bound.  For a 16-bit workload they also get a rounding term
  BN_SUM_K * 2^-24 * sum|t| per channel, t the summed terms (dz for db,
  dz*xhat for dw) as the oracle forms them: each term is formed in fp32 from
  16-bit inputs (exact in fp32) with a few roundings and an activation
  derivative evaluated in fp32, so a channel whose sum nearly cancels cannot
  meet an absolute 1e-5.  In training, dw also gets 4 ulps(mean) * rstd * |db|:
  the backward reads the mean the forward saved in fp32, and a mean off by d
  moves dw by d*rstd*db.

ReLU decides an integer from floating point (the mask bit z > 0).  The kernel
decides in fp32, the oracle in double, so elements whose oracle pre-activation
lies within RELU_BAND of 0 may legitimately get either decision.  There the test
accepts either branch (y in {0, z}; dx, dres from the oracle run with that bit
set either way) and compares all other elements exactly as above.
"""
from __future__ import annotations

import numpy as np
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth

TOL = {"f32": (1e-5, 1e-5), "f16": (2e-2, 1e-2), "bf16": (2e-2, 1e-2)}
# the parameter the parameterised activations are tested with (slope, alpha)
ACT_PARAM = {"leaky_relu": 0.05, "elu": 1.3, "celu": 0.7}
SELU_L, SELU_A = 1.0507009873554805, 1.6732632423543772
# activations with a kink at 0 whose branch the kernel (fp32) and the oracle
# (double) may decide differently within RELU_BAND
KINKED = ("relu", "leaky_relu", "elu", "selu")
# the clamping activations: their two ends, where either branch (z passed
# through, or the bound) is accepted within RELU_BAND
CLAMPS = {"relu6": (0.0, 6.0), "hardtanh": (-1.0, 1.0)}
STAT_TOL = (1e-5, 1e-5)
# rounding term of the BatchNorm channel sums of 16-bit workloads, in units of
# 2^-24 * sum|term| (derivation beside the tolerances in the design notes)
BN_SUM_K = 2.0
U32 = 2.0 ** -24
# largest (error - float32 bound) / (2^-24 * sum|term|) seen by compare_bn, per sum
BN_SUM_RATIO = {"db": 0.0, "dw": 0.0}
RELU_BAND = 1e-4
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def dev(t: synth.Tensor | None):
    return None if t is None else t.torch("cuda")


def host(t) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def assert_close(got, want, tol, what, mask=None):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    atol, rtol = tol
    err = np.abs(got - want)
    bad = err > atol + rtol * np.abs(want)
    if mask is not None:
        bad &= mask
    if bad.any():
        i = int(np.flatnonzero(bad.ravel())[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance "
            f"(atol {atol}, rtol {rtol}); first at flat index {i}: got {got.ravel()[i]!r}, "
            f"want {want.ravel()[i]!r}; max err {err.max():.3e}")


def empty(shape, dtype: str):
    return torch.empty(shape, dtype=TORCH_DT[dtype], device="cuda")


def workspace(op, rows, cols, dtype_code):
    nbytes = nrm.nrm_workspace_bytes(op, rows, cols, dtype_code)
    return torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")


DT_CODE = {"f32": nrm.NRM_F32, "f16": nrm.NRM_F16, "bf16": nrm.NRM_BF16}


# ---------------------------------------------------------------------------
# row norms
# ---------------------------------------------------------------------------

def run_row(kind, inp, dtype, eps, with_w=True, with_b=True, want_dw=True, want_db=True):
    """Forward then backward through libnorm.  Returns host float64 arrays."""
    x = dev(inp["x"])
    dy = dev(inp["dy"])
    w = dev(inp.get("w")) if with_w else None
    # RMSNorm takes its optional bias when the inputs carry one
    b = dev(inp.get("b")) if (with_b and (kind == "layernorm" or "b" in inp)) else None
    rows, cols = x.shape
    y = empty(x.shape, dtype)
    dx = empty(x.shape, dtype)
    rstd = torch.empty(rows, dtype=torch.float32, device="cuda")
    mean = torch.empty(rows, dtype=torch.float32, device="cuda")
    dw = empty((cols,), dtype) if want_dw else None
    db = empty((cols,), dtype) if (want_db and (kind == "layernorm" or b is not None)) else None
    if kind == "layernorm":
        nrm.nrm_layernorm_fwd(x, w, b, y, mean, rstd, eps)
        ws = workspace(nrm.NRM_OP_LAYERNORM_BWD, rows, cols, DT_CODE[dtype])
        nrm.nrm_layernorm_bwd(dy, x, w, mean, rstd, dx, dw, db, ws)
    else:
        nrm.nrm_rmsnorm_fwd(x, w, y, rstd, eps, b=b)
        ws = workspace(nrm.NRM_OP_RMSNORM_BWD, rows, cols, DT_CODE[dtype])
        nrm.nrm_rmsnorm_bwd(dy, x, w, rstd, dx, dw, ws, db=db)
    nrm.nrm_sync_status()
    out = dict(y=host(y), dx=host(dx), rstd=host(rstd))
    if kind == "layernorm":
        out["mean"] = host(mean)
    if db is not None:
        out["db"] = host(db)
    if dw is not None:
        out["dw"] = host(dw)
    return out


def oracle_row(orc, kind, inp, eps, with_w=True, with_b=True):
    x = inp["x"].f64()
    dy = inp["dy"].f64()
    w = inp["w"].f64() if (with_w and "w" in inp) else None
    b = inp["b"].f64() if (with_b and "b" in inp) else None
    if kind == "layernorm":
        y, mean, rstd = orc.layernorm_fwd(x, w, b, eps)
        dx, dw, db = orc.layernorm_bwd(dy, x, w, eps)
        return dict(y=y, mean=mean, rstd=rstd, dx=dx, dw=dw, db=db)
    y, rstd = orc.rmsnorm_fwd(x, w, eps, b=b)
    dx, dw, db = orc.rmsnorm_bwd(dy, x, w, eps, with_db=True)
    return dict(y=y, rstd=rstd, dx=dx, dw=dw, db=db)


def compare_row(got, want, dtype, tag):
    tol = TOL[dtype]
    for k in ("y", "dx", "dw", "db"):
        if k in got:
            assert_close(got[k], want[k], tol, f"{tag} {k}")
    for k in ("mean", "rstd"):
        if k in got:
            assert_close(got[k], want[k], STAT_TOL, f"{tag} {k}")


# ---------------------------------------------------------------------------
# BatchNorm
# ---------------------------------------------------------------------------

def unpack_mask(words: np.ndarray, n, c, l) -> np.ndarray:
    """Bits of the documented layout -> bool [n, c, l]."""
    per = (l + 31) // 32
    w = np.ascontiguousarray(words, dtype=np.uint32).reshape(n * c, per)
    bits = np.unpackbits(w.view(np.uint8), bitorder="little").reshape(n * c, per * 32)[:, :l]
    return bits.reshape(n, c, l).astype(bool)


def pack_mask(bits: np.ndarray) -> np.ndarray:
    n, c, l = bits.shape
    per = (l + 31) // 32
    padded = np.zeros((n * c, per * 32), dtype=np.uint8)
    padded[:, :l] = bits.reshape(n * c, l)
    return np.packbits(padded, bitorder="little").view(np.uint32).copy()


def run_bn(inp, dtype, eps, momentum, training, act, with_res, use_mask, with_affine=True):
    x = dev(inp["x"])
    n, c, l = x.shape
    res = dev(inp["res"]) if with_res else None
    w = dev(inp["w"]) if with_affine else None
    b = dev(inp["b"]) if with_affine else None
    rm = dev(inp["running_mean"]).clone()
    rv = dev(inp["running_var"]).clone()
    dy = dev(inp["dy"])
    y = empty(x.shape, dtype)
    sm = torch.empty(c, dtype=torch.float32, device="cuda")
    sr = torch.empty(c, dtype=torch.float32, device="cuda")
    mask = None
    if use_mask:
        mask = torch.full((nrm.nrm_act_mask_words(n, c, l),), 0xA5A5A5A5 - 2**32, dtype=torch.int32,
                          device="cuda")
    ws = nrm.batchnorm_workspace(x)
    prm = ACT_PARAM.get(act, 0.0)
    nrm.nrm_batchnorm_fwd(x, res, w, b, y, rm, rv, sm, sr, mask, eps, momentum, training, act, ws, act_param=prm)
    dx = empty(x.shape, dtype)
    dres = empty(x.shape, dtype)
    dw = torch.empty(c, dtype=torch.float32, device="cuda")
    db = torch.empty(c, dtype=torch.float32, device="cuda")
    nrm.nrm_batchnorm_bwd(dy, x, res, w, b, sm, sr, mask, dx, dres, dw, db, training, act, ws, act_param=prm)
    nrm.nrm_sync_status()
    out = dict(y=host(y), save_mean=host(sm), save_rstd=host(sr), running_mean=host(rm),
               running_var=host(rv), dx=host(dx), dres=host(dres), dw=host(dw), db=host(db))
    if mask is not None:
        out["mask"] = mask.cpu().numpy().view(np.uint32)
    return out


def oracle_bn(orc, inp, eps, momentum, training, act, with_res, with_affine=True):
    import oracle as oracle_mod
    a = {"none": oracle_mod.ACT_NONE, "relu": oracle_mod.ACT_RELU, "gelu": oracle_mod.ACT_GELU,
         "silu": oracle_mod.ACT_SILU, "mish": oracle_mod.ACT_MISH, "leaky_relu": oracle_mod.ACT_LEAKY_RELU,
         "elu": oracle_mod.ACT_ELU, "sigmoid": oracle_mod.ACT_SIGMOID, "celu": oracle_mod.ACT_CELU,
         "selu": oracle_mod.ACT_SELU, "relu6": oracle_mod.ACT_RELU6,
         "hardtanh": oracle_mod.ACT_HARDTANH}[act]
    prm = ACT_PARAM.get(act, 0.0)
    x = inp["x"].f64()
    res = inp["res"].f64() if with_res else None
    w = inp["w"].f64() if with_affine else None
    b = inp["b"].f64() if with_affine else None
    rm0 = inp["running_mean"].f64()
    rv0 = inp["running_var"].f64()
    dy = inp["dy"].f64()
    f = orc.batchnorm_fwd(x, res, w, b, eps, momentum, training, a, rm0, rv0,
                          want_mask=(act == "relu"), want_z=True, act_param=prm)
    bw = orc.batchnorm_bwd(dy, x, res, w, b, rm0, rv0, eps, training, a, mask=f["mask"], act_param=prm)
    out = dict(fwd=f, bwd=bw, act=a, x=x, dy=dy)
    if act in KINKED:
        z = f["z"]
        amb = np.abs(z) < RELU_BAND
        out["amb"] = amb
        # the other branch's output at the kink: relu 0 | z, leaky a*z | z, elu a*(e^z - 1) | z
        neg = {"relu": 0.0 * z, "leaky_relu": prm * z, "elu": prm * np.expm1(z),
               "selu": SELU_L * SELU_A * np.expm1(z)}[act]
        pos = SELU_L * z if act == "selu" else z
        out["y_alt"] = np.where(z > 0, neg, pos)
        if act == "relu" and amb.any():
            bits = unpack_mask(f["mask"], *x.shape)
            out["bwd_flipped"] = orc.batchnorm_bwd(dy, x, res, w, b, rm0, rv0, eps, training, a,
                                                   mask=pack_mask(bits ^ amb))
    elif act in CLAMPS:
        lo, hi = CLAMPS[act]
        z = f["z"]
        near_lo = np.abs(z - lo) < RELU_BAND
        amb = near_lo | (np.abs(z - hi) < RELU_BAND)
        out["amb"] = amb
        # the other branch: the bound where the oracle passed z through, z where it clamped
        out["y_alt"] = np.where(f["y"] == z, np.where(near_lo, lo, hi), z)
    return out


def compare_bn(got, want, dtype, training, act, tag):
    tol = TOL[dtype]
    f = want["fwd"]
    dx_a, dres_a, dw_a, db_a = want["bwd"]
    amb = want.get("amb")
    ok = None if amb is None else ~amb
    assert_close(got["y"], f["y"], tol, f"{tag} y", mask=ok)
    if amb is not None and amb.any():
        # either branch of the kink decision, within tolerance
        y_amb = got["y"][amb]
        lim = tol[0] + tol[1] * np.abs(f["z"][amb])
        e1 = np.abs(y_amb - f["y"][amb])
        e2 = np.abs(y_amb - want["y_alt"][amb])
        assert (np.minimum(e1, e2) <= lim).all(), f"{tag} y at kink ties"
    assert_close(got["save_mean"], f["save_mean"], STAT_TOL, f"{tag} save_mean")
    assert_close(got["save_rstd"], f["save_rstd"], STAT_TOL, f"{tag} save_rstd")
    if training:
        assert_close(got["running_mean"], f["running_mean"], STAT_TOL, f"{tag} running_mean")
        assert_close(got["running_var"], f["running_var"], STAT_TOL, f"{tag} running_var")
    if "mask" in got:
        n, c, l = got["y"].shape
        gb = unpack_mask(got["mask"], n, c, l)
        ob = unpack_mask(f["mask"], n, c, l)
        diff = (gb != ob) & ~amb
        assert not diff.any(), f"{tag} ReLU mask: {int(diff.sum())} bits differ outside the tie band"
        # bits past l in each segment's last word are zero
        per = (l + 31) // 32
        if l % 32:
            last = got["mask"].reshape(n * c, per)[:, -1]
            assert (last >> np.uint32(l % 32) == 0).all(), f"{tag} ReLU mask padding bits set"
    for name, g, a_ in (("dx", got["dx"], dx_a), ("dres", got["dres"], dres_a)):
        if amb is not None and amb.any() and "bwd_flipped" in want:
            b_ = want["bwd_flipped"][0 if name == "dx" else 1]
            atol, rtol = tol
            ea = np.abs(g - a_) <= atol + rtol * np.abs(a_)
            eb = np.abs(g - b_) <= atol + rtol * np.abs(b_)
            good = np.where(amb, ea | eb, ea)
            assert good.all(), f"{tag} {name}: {int((~good).sum())} elements out of tolerance"
        elif amb is not None and amb.any():
            # a tie decided the other way changes that element's derivative (1 vs
            # the slope or alpha); the per-channel sums below bound its effect
            assert_close(g, a_, tol, f"{tag} {name}", mask=~amb)
        else:
            assert_close(g, a_, tol, f"{tag} {name}")
    # per-channel sums.  Outside ReLU ties they are unique.  A tie element the
    # kernel decided the other way changes db by +-dy and dw by +-dy*xhat: with
    # the kernel's mask that set is known and the expected sums are corrected
    # by exactly those terms; without a mask only a bound can be checked.
    x = want["x"]
    corr_db = np.zeros_like(db_a)
    corr_dw = np.zeros_like(dw_a)
    slack = np.zeros_like(db_a)
    if amb is not None and amb.any():
        dy = want["dy"]
        xhat = (x - f["save_mean"][None, :, None]) * f["save_rstd"][None, :, None]
        if "mask" in got:
            n, c, l = got["y"].shape
            gb = unpack_mask(got["mask"], n, c, l)
            ob = unpack_mask(f["mask"], n, c, l)
            flip = amb & (gb != ob)
            sgn = np.where(gb, 1.0, -1.0) * flip
            corr_db = (sgn * dy).sum(axis=(0, 2))
            corr_dw = (sgn * dy * xhat).sum(axis=(0, 2))
        else:
            slack = (np.abs(dy) * amb).sum(axis=(0, 2))
            slack_w = (np.abs(dy * xhat) * amb).sum(axis=(0, 2))
    # dw, db are float32 tensors: the float32 bound, plus for 16-bit workloads
    # BN_SUM_K * 2^-24 * sum|term| of the channel's terms (dz, dz*xhat)
    atol, rtol = STAT_TOL
    ref_db = db_a + corr_db
    ref_dw = dw_a + corr_dw
    round_db = np.zeros_like(db_a)
    round_dw = np.zeros_like(dw_a)
    if dtype != "f32":
        xhat_o = (x - f["save_mean"][None, :, None]) * f["save_rstd"][None, :, None]
        round_db = U32 * np.abs(dres_a).sum(axis=(0, 2))
        round_dw = U32 * np.abs(dres_a * xhat_o).sum(axis=(0, 2))
    slack_dw = slack_w if slack.any() else slack
    if training:
        # dw is computed from the saved fp32 mean: a mean off by d moves dw by
        # d*rstd*db, and a mean held in fp32 is off by up to a few ulps (4 here)
        mu = f["save_mean"]
        ulp = np.spacing(np.abs(mu).astype(np.float32)).astype(np.float64)
        slack_dw = slack_dw + 4.0 * ulp * f["save_rstd"] * np.abs(ref_db)
    for name, g, ref, rnd, sl in (("db", got["db"], ref_db, round_db, slack),
                                  ("dw", got["dw"], ref_dw, round_dw, slack_dw)):
        err = np.abs(g - ref)
        base = atol + rtol * np.abs(ref) + sl
        if dtype != "f32":
            over = (err - base) / np.maximum(rnd, 1e-300)
            BN_SUM_RATIO[name] = max(BN_SUM_RATIO[name], float(np.max(over, initial=0.0)))
        assert (err <= base + BN_SUM_K * rnd).all(), \
            f"{tag} {name}: max err {err.max():.3e} (float32 bound + {BN_SUM_K:g} * 2^-24 * sum|term|)"
