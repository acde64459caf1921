"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on failure.
They are run against the committed oracle (test_oracle_pins.py) and against
copies with a planted mistake (test_oracle_mutations.py), which every pin set
must catch.

What pins what:
  * hand-worked fixtures in tests/golden/ (exact values derived on paper);
  * closed forms and invariants: standardised rows/channels have mean 0 and
    mean square var/(var+eps); LayerNorm and BatchNorm input gradients sum
    to 0 and sum(dx*xhat) = rstd*sum(g*xhat)*eps/(var+eps); the RMSNorm gradient satisfies
    sum(x*dx) = inv_rms*sum(g*x)*eps/(ms+eps); the running statistics follow
    the EMA with the unbiased batch variance (numpy var with ddof=1);
  * brute force on the smallest sizes, worked by hand: rows of one and two
    columns, BatchNorm channels of two elements (training and eval);
  * central finite differences of L = sum(dy * y) for every backward output;
  * independent library routines: torch.nn.functional layer_norm / rms_norm /
    batch_norm / gelu / silu / mish and torch autograd, all in float64 on the CPU;
  * the dropout generator: the published Philox4x32-10 known-answer vectors
    (tests/golden/), and binomial bounds on keep rates and on the agreement of
    masks that must be independent.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ACT = {"none": 0, "relu": 1, "gelu": 2, "silu": 3, "mish": 4, "leaky_relu": 5, "elu": 6,
       "sigmoid": 7, "celu": 8, "selu": 9, "relu6": 10, "hardtanh": 11}
# where each kinked activation's derivative jumps (finite differences keep clear of them)
KINKS = {"relu": (0.0,), "leaky_relu": (0.0,), "relu6": (0.0, 6.0), "hardtanh": (-1.0, 1.0)}
# the parameter the activations that take one are exercised with (slope, alpha)
ACT_PARAM = {"leaky_relu": 0.05, "elu": 1.3, "celu": 0.7}
ALL_ACTS = tuple(ACT)


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.abs(a - b)
    bad = err > atol + rtol * np.abs(b)
    assert not bad.any(), (f"{what}: max err {err.max():.3e} at {np.argmax(err)}; "
                           f"got {a.ravel()[np.argmax(err)]}, want {b.ravel()[np.argmax(err)]}")


def _central_diff(f, v, h):
    """Gradient of scalar f at array v by central differences."""
    g = np.zeros_like(v)
    it = np.nditer(v, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        keep = v[i]
        v[i] = keep + h
        fp = f()
        v[i] = keep - h
        fm = f()
        v[i] = keep
        g[i] = (fp - fm) / (2 * h)
    return g


# ---------------------------------------------------------------------------
# LayerNorm
# ---------------------------------------------------------------------------

def pin_layernorm_golden(o):
    d = json.load(open(os.path.join(GOLDEN, "layernorm_rmsnorm_hand_worked.json")))
    for case in d["layernorm"]:
        x = np.array([case["x"]])
        w = None if case["w"] is None else np.array(case["w"])
        b = None if case["b"] is None else np.array(case["b"])
        y, mean, rstd = o.layernorm_fwd(x, w, b, eps=case["eps"])
        _close(y[0], case["y"], 1e-15, 1e-15, "layernorm golden y")
        _close(mean[0], case["mean"], 1e-15, 0, "layernorm golden mean")
        _close(rstd[0], case["rstd"], 1e-15, 0, "layernorm golden rstd")


def pin_layernorm_standardizes(o):
    r = _rng(1)
    x = r.normal(size=(6, 37)) * r.uniform(0.1, 5, size=(6, 1)) + r.uniform(-3, 3, size=(6, 1))
    eps = 1e-3
    y, mean, rstd = o.layernorm_fwd(x, None, None, eps=eps)
    var = np.var(x, axis=1)
    _close(y.mean(axis=1), np.zeros(6), 0, 1e-13, "row mean of standardised y")
    _close((y * y).mean(axis=1), var / (var + eps), 1e-12, 0, "row mean square of y")
    _close(mean, np.mean(x, axis=1), 1e-13, 1e-13, "saved mean")


def pin_layernorm_vs_torch(o):
    import torch
    r = _rng(2)
    x = r.normal(size=(7, 33)) * 2 + 0.5
    w = 1 + 0.3 * r.normal(size=33)
    b = 0.2 * r.normal(size=33)
    y, _, rstd = o.layernorm_fwd(x, w, b, eps=1e-5)
    yt = torch.nn.functional.layer_norm(torch.from_numpy(x), (33,), torch.from_numpy(w),
                                        torch.from_numpy(b), eps=1e-5).numpy()
    _close(y, yt, 1e-12, 1e-12, "layernorm vs torch")


def pin_layernorm_bwd_fd(o):
    r = _rng(3)
    for rows, cols in ((3, 5), (2, 17)):
        x = r.normal(size=(rows, cols))
        w = 1 + 0.5 * r.normal(size=cols)
        b = 0.5 * r.normal(size=cols)
        dy = r.normal(size=(rows, cols))
        eps = 1e-3
        dx, dw, db = o.layernorm_bwd(dy, x, w, eps=eps)
        loss = lambda: float((dy * o.layernorm_fwd(x, w, b, eps=eps)[0]).sum())
        h = 1e-6
        _close(dx, _central_diff(loss, x, h), 1e-6, 1e-7, "layernorm dx vs finite differences")
        _close(dw, _central_diff(loss, w, h), 1e-6, 1e-7, "layernorm dw vs finite differences")
        _close(db, _central_diff(loss, b, h), 1e-6, 1e-7, "layernorm db vs finite differences")


def pin_layernorm_bwd_invariants(o):
    # sum_j dx_j = 0 and sum_j dx_j*xhat_j = rstd * sum(g*xhat) * eps/(var+eps)
    r = _rng(4)
    x = r.normal(size=(5, 64)) * 3 + 1
    w = 1 + 0.5 * r.normal(size=64)
    dy = r.normal(size=(5, 64))
    eps = 0.5
    dx, _, _ = o.layernorm_bwd(dy, x, w, eps=eps)
    var = x.var(1, keepdims=True)
    rstd = 1 / np.sqrt(var + eps)
    xhat = (x - x.mean(1, keepdims=True)) * rstd
    scale = np.abs(dx).sum(1)
    _close(dx.sum(1) / scale, np.zeros(5), 0, 1e-13, "sum of dx per row")
    want = (rstd * ((dy * w) * xhat).sum(1, keepdims=True) * eps / (var + eps)).ravel()
    _close((dx * xhat).sum(1), want, 1e-10, 1e-13, "sum of dx*xhat per row")


def pin_layernorm_bwd_vs_torch(o):
    import torch
    r = _rng(5)
    x = torch.tensor(r.normal(size=(4, 19)), requires_grad=True)
    w = torch.tensor(1 + 0.4 * r.normal(size=19), requires_grad=True)
    b = torch.tensor(0.3 * r.normal(size=19), requires_grad=True)
    dy = r.normal(size=(4, 19))
    y = torch.nn.functional.layer_norm(x, (19,), w, b, eps=1e-4)
    y.backward(torch.from_numpy(dy))
    dx, dw, db = o.layernorm_bwd(dy, x.detach().numpy(), w.detach().numpy(), eps=1e-4)
    _close(dx, x.grad.numpy(), 1e-11, 1e-12, "layernorm dx vs torch autograd")
    _close(dw, w.grad.numpy(), 1e-11, 1e-12, "layernorm dw vs torch autograd")
    _close(db, b.grad.numpy(), 1e-11, 1e-12, "layernorm db vs torch autograd")


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def pin_rmsnorm_golden(o):
    d = json.load(open(os.path.join(GOLDEN, "layernorm_rmsnorm_hand_worked.json")))
    for case in d["rmsnorm"]:
        y, rstd = o.rmsnorm_fwd(np.array([case["x"]]), np.array(case["w"]), eps=case["eps"])
        _close(y[0], case["y"], 1e-15, 1e-15, "rmsnorm golden y")
        _close(rstd[0], case["rstd"], 1e-15, 0, "rmsnorm golden rstd")


def pin_rmsnorm_unit_rms(o):
    r = _rng(6)
    x = r.normal(size=(6, 41)) * r.uniform(0.1, 4, size=(6, 1)) + 0.3
    eps = 1e-2
    y, rstd = o.rmsnorm_fwd(x, None, eps=eps)
    ms = np.mean(x * x, axis=1)
    _close((y * y).mean(1), ms / (ms + eps), 1e-12, 0, "row mean square of RMS-normalised y")
    # direction is preserved: y is a positive multiple of x
    _close(y / x, np.broadcast_to((y / x)[:, :1], y.shape), 1e-12, 0, "y parallel to x")


def pin_rmsnorm_vs_torch(o):
    import torch
    r = _rng(7)
    x = r.normal(size=(5, 24)) * 1.5
    w = 1 + 0.2 * r.normal(size=24)
    y, _ = o.rmsnorm_fwd(x, w, eps=1e-6)
    yt = torch.nn.functional.rms_norm(torch.from_numpy(x), (24,), torch.from_numpy(w),
                                      eps=1e-6).numpy()
    _close(y, yt, 1e-12, 1e-12, "rmsnorm vs torch")


def pin_rmsnorm_bwd_fd(o):
    r = _rng(8)
    for rows, cols in ((3, 5), (2, 17)):
        x = r.normal(size=(rows, cols))
        w = 1 + 0.5 * r.normal(size=cols)
        dy = r.normal(size=(rows, cols))
        eps = 1e-3
        dx, dw = o.rmsnorm_bwd(dy, x, w, eps=eps)
        loss = lambda: float((dy * o.rmsnorm_fwd(x, w, eps=eps)[0]).sum())
        _close(dx, _central_diff(loss, x, 1e-6), 1e-6, 1e-7, "rmsnorm dx vs finite differences")
        _close(dw, _central_diff(loss, w, 1e-6), 1e-6, 1e-7, "rmsnorm dw vs finite differences")


def pin_rmsnorm_bias(o):
    """With a bias: y is torch's rms_norm plus b; db = sum of dy over rows and
    dx, dw are those without the bias; all three against finite differences."""
    import torch
    r = _rng(33)
    x = r.normal(size=(4, 19)) * 1.2
    w = 1 + 0.2 * r.normal(size=19)
    b = 0.3 * r.normal(size=19)
    y, _ = o.rmsnorm_fwd(x, w, eps=1e-5, b=b)
    yt = torch.nn.functional.rms_norm(torch.from_numpy(x), (19,), torch.from_numpy(w), eps=1e-5).numpy()
    _close(y, yt + b, 1e-12, 1e-12, "rmsnorm with bias vs torch")
    dy = r.normal(size=(4, 19))
    dx, dw, db = o.rmsnorm_bwd(dy, x, w, eps=1e-5, with_db=True)
    dx0, dw0 = o.rmsnorm_bwd(dy, x, w, eps=1e-5)
    _close(db, dy.sum(0), 1e-15, 1e-15, "rmsnorm db = sum dy")
    assert (dx == dx0).all() and (dw == dw0).all(), "the bias must not change dx, dw"
    loss = lambda: float((dy * o.rmsnorm_fwd(x, w, eps=1e-5, b=b)[0]).sum())
    _close(db, _central_diff(loss, b, 1e-6), 1e-7, 1e-7, "rmsnorm db vs finite differences")
    _close(dx, _central_diff(loss, x, 1e-6), 1e-6, 1e-7, "rmsnorm (bias) dx vs finite differences")


def pin_rmsnorm_bwd_invariant(o):
    r = _rng(9)
    x = r.normal(size=(4, 50))
    w = 1 + 0.5 * r.normal(size=50)
    dy = r.normal(size=(4, 50))
    eps = 0.05
    dx, _ = o.rmsnorm_bwd(dy, x, w, eps=eps)
    ms = (x * x).mean(1)
    rr = 1 / np.sqrt(ms + eps)
    want = rr * ((dy * w) * x).sum(1) * eps / (ms + eps)
    _close((x * dx).sum(1), want, 1e-11, 1e-13, "sum(x*dx) closed form")


def pin_rmsnorm_bwd_vs_torch(o):
    import torch
    r = _rng(10)
    x = torch.tensor(r.normal(size=(3, 21)), requires_grad=True)
    w = torch.tensor(1 + 0.4 * r.normal(size=21), requires_grad=True)
    dy = r.normal(size=(3, 21))
    y = torch.nn.functional.rms_norm(x, (21,), w, eps=1e-5)
    y.backward(torch.from_numpy(dy))
    dx, dw = o.rmsnorm_bwd(dy, x.detach().numpy(), w.detach().numpy(), eps=1e-5)
    _close(dx, x.grad.numpy(), 1e-11, 1e-12, "rmsnorm dx vs torch autograd")
    _close(dw, w.grad.numpy(), 1e-11, 1e-12, "rmsnorm dw vs torch autograd")


# ---------------------------------------------------------------------------
# BatchNorm
# ---------------------------------------------------------------------------

def pin_batchnorm_golden(o):
    d = json.load(open(os.path.join(GOLDEN, "batchnorm_hand_worked.json")))
    for case in d["cases"]:
        shape = tuple(case["shape"])
        x = np.array(case["x"]).reshape(shape)
        res = np.array(case["res"]).reshape(shape) if "res" in case else None
        out = o.batchnorm_fwd(x, res, np.array(case["w"]), np.array(case["b"]),
                              eps=case["eps"], momentum=case["momentum"],
                              training=case.get("training", True), act=ACT[case["act"]],
                              running_mean=np.array(case["running_mean_in"]),
                              running_var=np.array(case["running_var_in"]),
                              want_mask=case["act"] == "relu")
        _close(out["y"].ravel(), case["y"], 1e-15, 1e-15, "batchnorm golden y")
        _close(out["save_mean"], case["save_mean"], 1e-15, 0, "batchnorm golden mean")
        _close(out["save_rstd"], case["save_rstd"], 1e-15, 0, "batchnorm golden rstd")
        if "running_mean" in case:
            _close(out["running_mean"], case["running_mean"], 1e-15, 0, "golden running_mean")
            _close(out["running_var"], case["running_var"], 1e-15, 0, "golden running_var")
        if "mask_words" in case:
            assert list(out["mask"]) == case["mask_words"], f"mask {list(out['mask'])}"
        if "dres_for_unit_dy" in case:
            # dz = dy * ReLU'(z) with ReLU'(0) = 0, recomputed (no mask) and from the mask
            for mask in (None, out["mask"]):
                _, dres, _, _ = o.batchnorm_bwd(np.ones(shape), x, res, np.array(case["w"]),
                                                np.array(case["b"]), eps=case["eps"],
                                                training=case.get("training", True),
                                                act=ACT[case["act"]], mask=mask)
                _close(dres.ravel(), case["dres_for_unit_dy"], 0, 0, "golden ReLU gradient")


def pin_batchnorm_standardizes_and_ema(o):
    r = _rng(11)
    n, c, l = 4, 3, 10
    x = r.normal(size=(n, c, l)) * np.array([0.5, 2, 4])[None, :, None] + np.array([-1, 0, 3])[None, :, None]
    eps = 1e-2
    out = o.batchnorm_fwd(x, eps=eps, momentum=0.1, training=True,
                          running_mean=np.zeros(c), running_var=np.ones(c))
    y = out["y"]
    xc = x.transpose(1, 0, 2).reshape(c, -1)
    yc = y.transpose(1, 0, 2).reshape(c, -1)
    var_b = np.var(xc, axis=1)
    _close(yc.mean(1), np.zeros(c), 0, 1e-13, "channel mean of y")
    _close((yc * yc).mean(1), var_b / (var_b + eps), 1e-12, 0, "channel mean square of y")
    _close(out["running_mean"], 0.1 * np.mean(xc, axis=1), 1e-13, 1e-15, "running_mean EMA")
    _close(out["running_var"], 0.9 + 0.1 * np.var(xc, axis=1, ddof=1), 1e-13, 0, "running_var EMA")


def _torch_bn_forward(x, res, w, b, rm, rv, eps, momentum, training, act):
    import torch
    F = torch.nn.functional
    xt = torch.from_numpy(x)
    z = F.batch_norm(xt, rm, rv, torch.from_numpy(w), torch.from_numpy(b),
                     training=training, momentum=momentum, eps=eps)
    if res is not None:
        z = z + torch.from_numpy(res)
    if act == "relu":
        return F.relu(z)
    if act == "gelu":
        return F.gelu(z, approximate="none")
    if act == "silu":
        return F.silu(z)
    if act == "mish":
        return F.mish(z)
    if act == "leaky_relu":
        return F.leaky_relu(z, ACT_PARAM[act])
    if act == "elu":
        return F.elu(z, ACT_PARAM[act])
    if act == "sigmoid":
        return torch.sigmoid(z)
    if act == "celu":
        return F.celu(z, ACT_PARAM[act])
    if act == "selu":
        return F.selu(z)
    if act == "relu6":
        return F.relu6(z)
    if act == "hardtanh":
        return F.hardtanh(z)
    return z


def pin_batchnorm_vs_torch(o):
    import torch
    r = _rng(12)
    n, c, l = 3, 4, 7
    for training in (True, False):
        for act in ALL_ACTS:
            for with_res in (False, True):
                x = r.normal(size=(n, c, l)) * 1.7 + 0.4
                res = r.normal(size=(n, c, l)) if with_res else None
                w = 1 + 0.3 * r.normal(size=c)
                b = 0.3 * r.normal(size=c)
                rm0 = 0.2 * r.normal(size=c)
                rv0 = 1 + 0.5 * r.uniform(size=c)
                rm_t = torch.from_numpy(rm0.copy())
                rv_t = torch.from_numpy(rv0.copy())
                yt = _torch_bn_forward(x, res, w, b, rm_t, rv_t, 1e-5, 0.1, training, act).numpy()
                out = o.batchnorm_fwd(x, res, w, b, eps=1e-5, momentum=0.1, training=training,
                                      act=ACT[act], running_mean=rm0, running_var=rv0,
                                      act_param=ACT_PARAM.get(act, 0.0))
                tag = f"batchnorm training={training} act={act} res={with_res}"
                _close(out["y"], yt, _torch_rtol(act, 1e-12), 1e-12, tag + " y vs torch")
                _close(out["running_mean"], rm_t.numpy(), 1e-13, 1e-15, tag + " running_mean")
                _close(out["running_var"], rv_t.numpy(), 1e-13, 1e-15, tag + " running_var")


def pin_gelu_values(o):
    # eval mode with running_mean 0 and running_var + eps = 1 makes z = x exactly
    z = np.array([-3.0, -1.0, 0.0, 0.5, 1.0, 2.0]).reshape(1, 1, 6)
    out = o.batchnorm_fwd(z, eps=0.25, training=False, act=ACT["gelu"],
                          running_mean=np.zeros(1), running_var=np.array([0.75]))
    phi = np.array([0.5 * (1 + math.erf(v / math.sqrt(2))) for v in z.ravel()])
    _close(out["y"].ravel(), z.ravel() * phi, 1e-15, 1e-16, "gelu = z * Phi(z)")
    # Phi(1) = 0.8413447460685429 (standard normal table)
    _close(out["y"].ravel()[4], 0.8413447460685429, 1e-15, 0, "gelu(1)")


def pin_silu_mish_values(o):
    # eval mode with running_mean 0 and running_var + eps = 1 makes z = x exactly;
    # then y = act(z) and, with w = 1 and dy = 1, dx = act'(z)
    ln3 = math.log(3.0)
    z = np.array([0.0, ln3, -ln3, math.log(math.e - 1.0), 2.0]).reshape(1, 1, 5)
    rm, rv = np.zeros(1), np.array([0.75])
    y_silu = o.batchnorm_fwd(z, eps=0.25, training=False, act=ACT["silu"], running_mean=rm,
                             running_var=rv)["y"].ravel()
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    _close(y_silu[:3], [0.0, 0.75 * ln3, -0.25 * ln3], 1e-15, 1e-16, "silu(0), silu(+-ln 3)")
    y_mish = o.batchnorm_fwd(z, eps=0.25, training=False, act=ACT["mish"], running_mean=rm,
                             running_var=rv)["y"].ravel()
    # softplus(log(e - 1)) = 1, so mish = log(e - 1) * tanh(1)
    _close(y_mish[[0, 3]], [0.0, math.log(math.e - 1.0) * math.tanh(1.0)], 1e-15, 1e-16, "mish(0), mish(log(e-1))")
    dy = np.ones_like(z)
    dx_silu = o.batchnorm_bwd(dy, z, None, np.ones(1), np.zeros(1), rm, rv, eps=0.25, training=False,
                              act=ACT["silu"])[0].ravel()
    # silu'(0) = 1/2; silu'(ln 3) = 3/4 + ln3 * 3/16
    _close(dx_silu[:2], [0.5, 0.75 + ln3 * 3.0 / 16.0], 1e-15, 1e-16, "silu'(0), silu'(ln 3)")
    dx_mish = o.batchnorm_bwd(dy, z, None, np.ones(1), np.zeros(1), rm, rv, eps=0.25, training=False,
                              act=ACT["mish"])[0].ravel()
    # mish'(0) = tanh(ln 2) = 3/5
    _close(dx_mish[0], 0.6, 1e-15, 1e-16, "mish'(0)")


def pin_leaky_relu_elu_values(o):
    # z = x as above; closed forms: leaky(-2) = -2a, elu(-ln 2) = -a/2,
    # elu'(-ln 2) = a/2, leaky'(z < 0) = a, both derivatives 1 for z > 0
    z = np.array([-2.0, -math.log(2.0), 0.5]).reshape(1, 1, 3)
    rm, rv = np.zeros(1), np.array([0.75])
    for act, a in (("leaky_relu", 0.2), ("elu", 1.7)):
        y = o.batchnorm_fwd(z, eps=0.25, training=False, act=ACT[act], running_mean=rm,
                            running_var=rv, act_param=a)["y"].ravel()
        dx = o.batchnorm_bwd(np.ones_like(z), z, None, np.ones(1), np.zeros(1), rm, rv, eps=0.25,
                             training=False, act=ACT[act], act_param=a)[0].ravel()
        if act == "leaky_relu":
            _close(y, [-2.0 * a, -math.log(2.0) * a, 0.5], 1e-15, 0, "leaky_relu values")
            _close(dx, [a, a, 1.0], 1e-15, 0, "leaky_relu derivative")
        else:
            _close(y[1:], [-a / 2.0, 0.5], 1e-15, 1e-16, "elu values")
            _close(dx[1:], [a / 2.0, 1.0], 1e-15, 1e-16, "elu derivative")


def pin_sigmoid_celu_selu_values(o):
    # z = x as above; closed forms: sigmoid(ln 3) = 3/4, sigmoid'(ln 3) = 3/16;
    # celu(-a ln 2) = -a/2, celu'(-a ln 2) = 1/2; selu(1) = L, selu'(-ln 2) = L*A/2
    rm, rv = np.zeros(1), np.array([0.75])
    lam, alp = 1.0507009873554805, 1.6732632423543772

    def run(act, zs, a=0.0):
        z = np.array(zs).reshape(1, 1, len(zs))
        y = o.batchnorm_fwd(z, eps=0.25, training=False, act=ACT[act], running_mean=rm,
                            running_var=rv, act_param=a)["y"].ravel()
        dx = o.batchnorm_bwd(np.ones_like(z), z, None, np.ones(1), np.zeros(1), rm, rv, eps=0.25,
                             training=False, act=ACT[act], act_param=a)[0].ravel()
        return y, dx
    y, dx = run("sigmoid", [math.log(3.0)])
    _close(y, [0.75], 1e-15, 0, "sigmoid(ln 3)")
    _close(dx, [3.0 / 16.0], 1e-15, 0, "sigmoid'(ln 3)")
    a = 0.8
    y, dx = run("celu", [-a * math.log(2.0), 1.5], a)
    _close(y, [-a / 2.0, 1.5], 1e-15, 1e-16, "celu values")
    _close(dx, [0.5, 1.0], 1e-15, 1e-16, "celu derivative")
    y, dx = run("selu", [1.0, -math.log(2.0)])
    _close(y, [lam, -lam * alp / 2.0], 1e-15, 1e-16, "selu values")
    _close(dx, [lam, lam * alp / 2.0], 1e-15, 1e-16, "selu derivative")


def pin_relu6_hardtanh_values(o):
    # z = x as above; closed forms from the definitions: relu6 clamps to [0, 6]
    # and hardtanh to [-1, 1]; each derivative is 1 strictly inside the range and
    # 0 outside it and at both ends
    rm, rv = np.zeros(1), np.array([0.75])

    def run(act, zs):
        z = np.array(zs).reshape(1, 1, len(zs))
        y = o.batchnorm_fwd(z, eps=0.25, training=False, act=ACT[act], running_mean=rm,
                            running_var=rv)["y"].ravel()
        dx = o.batchnorm_bwd(np.ones_like(z), z, None, np.ones(1), np.zeros(1), rm, rv, eps=0.25,
                             training=False, act=ACT[act])[0].ravel()
        return y, dx
    y, dx = run("relu6", [-2.5, 0.0, 0.75, 6.0, 7.5])
    _close(y, [0.0, 0.0, 0.75, 6.0, 6.0], 0, 0, "relu6 values")
    _close(dx, [0.0, 0.0, 1.0, 0.0, 0.0], 0, 0, "relu6 derivative")
    y, dx = run("hardtanh", [-3.0, -1.0, -0.25, 0.5, 1.0, 2.0])
    _close(y, [-1.0, -1.0, -0.25, 0.5, 1.0, 1.0], 0, 0, "hardtanh values")
    _close(dx, [0.0, 0.0, 1.0, 1.0, 0.0, 0.0], 0, 0, "hardtanh derivative")
    # the two are one clamp shifted and scaled: hardtanh(z) = relu6(3z + 3)/3 - 1
    zs = np.linspace(-2.0, 2.0, 41)
    ya = o.act_dropout_fwd(zs, ACT["hardtanh"], 0.0, 1)
    yb = o.act_dropout_fwd(3.0 * zs + 3.0, ACT["relu6"], 0.0, 1) / 3.0 - 1.0
    _close(ya, yb, 0, 1e-15, "hardtanh(z) = relu6(3z + 3)/3 - 1")


def pin_batchnorm_mask_layout(o):
    # eval mode, z = x: mask bit (i, ch, j) must be x > 0 with the documented layout
    n, c, l = 2, 3, 70
    words = (l + 31) // 32
    r = _rng(13)
    x = r.choice([-1.0, 2.0], size=(n, c, l))
    out = o.batchnorm_fwd(x, eps=0.25, training=False, act=ACT["relu"],
                          running_mean=np.zeros(c), running_var=np.full(c, 0.75),
                          want_mask=True)
    want = np.zeros(n * c * words, dtype=np.uint32)
    for i in range(n):
        for ch in range(c):
            for j in range(l):
                if x[i, ch, j] > 0:
                    want[(i * c + ch) * words + j // 32] |= np.uint32(1 << (j % 32))
    assert (out["mask"] == want).all(), "ReLU mask layout"


def _bn_inputs_away_from_kinks(r, n, c, l, act, with_res):
    """Tiny BatchNorm inputs whose pre-activation stays 1e-3 away from every
    kink of the activation (0 for ReLU, 0 and 6 for ReLU6, -1 and 1 for
    hardtanh), so finite differences do not cross one."""
    for _ in range(1000):
        x = r.normal(size=(n, c, l)) * 1.3 + 0.2
        res = r.normal(size=(n, c, l)) if with_res else None
        w = 1 + 0.3 * r.normal(size=c)
        b = 0.3 * r.normal(size=c)
        if act not in KINKS:
            return x, res, w, b
        xc = x.transpose(1, 0, 2).reshape(c, -1)
        mu = xc.mean(1)[None, :, None]
        rs = (1 / np.sqrt(xc.var(1) + 1e-3))[None, :, None]
        z = (x - mu) * rs * w[None, :, None] + b[None, :, None] + (res if with_res else 0)
        if min(np.abs(z - k).min() for k in KINKS[act]) > 1e-3:
            return x, res, w, b
    raise RuntimeError("no input away from the ReLU kink")


def pin_batchnorm_bwd_fd(o):
    r = _rng(14)
    eps = 1e-3
    for (n, c, l) in ((2, 3, 4), (3, 2, 5)):
        for training in (True, False):
            for act in ALL_ACTS:
                for with_res in (False, True):
                    x, res, w, b = _bn_inputs_away_from_kinks(r, n, c, l, act, with_res)
                    dy = r.normal(size=(n, c, l))
                    rm = 0.1 * r.normal(size=c)
                    rv = 1 + 0.2 * r.uniform(size=c)

                    def loss():
                        y = o.batchnorm_fwd(x, res, w, b, eps=eps, momentum=0.1,
                                            training=training, act=ACT[act],
                                            running_mean=rm, running_var=rv,
                                            act_param=ACT_PARAM.get(act, 0.0))["y"]
                        return float((dy * y).sum())
                    dx, dres, dw, db = o.batchnorm_bwd(dy, x, res, w, b, rm, rv, eps=eps,
                                                       training=training, act=ACT[act],
                                                       act_param=ACT_PARAM.get(act, 0.0))
                    tag = f"batchnorm bwd training={training} act={act} res={with_res}"
                    h = 1e-6
                    _close(dx, _central_diff(loss, x, h), 1e-6, 1e-7, tag + " dx vs FD")
                    _close(dw, _central_diff(loss, w, h), 1e-6, 1e-7, tag + " dw vs FD")
                    _close(db, _central_diff(loss, b, h), 1e-6, 1e-7, tag + " db vs FD")
                    if with_res:
                        _close(dres, _central_diff(loss, res, h), 1e-6, 1e-7, tag + " dres vs FD")


def pin_batchnorm_bwd_invariants(o):
    # per channel: sum dx = 0 and sum dx*xhat = w*rstd*sum(dy*xhat)*eps/(var+eps)
    r = _rng(15)
    n, c, l = 5, 3, 9
    x = r.normal(size=(n, c, l)) * 2 + 1
    w = 1 + 0.3 * r.normal(size=c)
    dy = r.normal(size=(n, c, l))
    eps = 0.3
    dx, _, _, _ = o.batchnorm_bwd(dy, x, None, w, None, eps=eps, training=True)
    xc = x.transpose(1, 0, 2).reshape(c, -1)
    var = xc.var(1, keepdims=True)
    rstd = 1 / np.sqrt(var + eps)
    xhat = (xc - xc.mean(1, keepdims=True)) * rstd
    dyc = dy.transpose(1, 0, 2).reshape(c, -1)
    dxc = dx.transpose(1, 0, 2).reshape(c, -1)
    scale = np.abs(dxc).sum(1)
    _close(dxc.sum(1) / scale, np.zeros(c), 0, 1e-13, "channel sum of dx")
    want = (w[:, None] * rstd * (dyc * xhat).sum(1, keepdims=True) * eps / (var + eps)).ravel()
    _close((dxc * xhat).sum(1), want, 1e-10, 1e-13, "channel sum of dx*xhat")


def pin_batchnorm_bwd_vs_torch(o):
    import torch
    F = torch.nn.functional
    r = _rng(16)
    n, c, l = 3, 4, 6
    acts = {"none": lambda z: z, "gelu": lambda z: F.gelu(z, approximate="none"), "silu": F.silu,
            "mish": F.mish, "elu": lambda z: F.elu(z, ACT_PARAM["elu"]), "sigmoid": torch.sigmoid,
            "celu": lambda z: F.celu(z, ACT_PARAM["celu"]), "selu": F.selu, "relu6": F.relu6,
            "hardtanh": F.hardtanh}
    for training in (True, False):
        for act in acts:
            x = torch.tensor(r.normal(size=(n, c, l)) * 1.5, requires_grad=True)
            res = torch.tensor(r.normal(size=(n, c, l)), requires_grad=True)
            w = torch.tensor(1 + 0.3 * r.normal(size=c), requires_grad=True)
            b = torch.tensor(0.3 * r.normal(size=c), requires_grad=True)
            rm = 0.1 * r.normal(size=c)
            rv = 1 + 0.2 * r.uniform(size=c)
            z = F.batch_norm(x, torch.from_numpy(rm.copy()), torch.from_numpy(rv.copy()), w, b,
                             training=training, momentum=0.1, eps=1e-5) + res
            y = acts[act](z)
            dy = r.normal(size=(n, c, l))
            y.backward(torch.from_numpy(dy))
            dx, dres, dw, db = o.batchnorm_bwd(dy, x.detach().numpy(), res.detach().numpy(),
                                               w.detach().numpy(), b.detach().numpy(), rm, rv,
                                               eps=1e-5, training=training, act=ACT[act],
                                               act_param=ACT_PARAM.get(act, 0.0))
            tag = f"batchnorm bwd vs torch training={training} act={act}"
            rt = _torch_rtol(act, 1e-10)
            _close(dx, x.grad.numpy(), rt, 1e-12, tag + " dx")
            _close(dres, res.grad.numpy(), rt, 1e-12, tag + " dres")
            _close(dw, w.grad.numpy(), rt, 1e-12, tag + " dw")
            _close(db, b.grad.numpy(), rt, 1e-12, tag + " db")


def pin_batchnorm_bwd_mask_matches_recompute(o):
    r = _rng(17)
    n, c, l = 3, 2, 45
    x, res, w, b = _bn_inputs_away_from_kinks(r, n, c, l, "relu", True)
    dy = r.normal(size=(n, c, l))
    out = o.batchnorm_fwd(x, res, w, b, eps=1e-3, training=True, act=ACT["relu"], want_mask=True)
    a = o.batchnorm_bwd(dy, x, res, w, b, eps=1e-3, training=True, act=ACT["relu"],
                        mask=out["mask"])
    bb = o.batchnorm_bwd(dy, x, res, w, b, eps=1e-3, training=True, act=ACT["relu"])
    for u, v, name in zip(a, bb, ("dx", "dres", "dw", "db")):
        _close(u, v, 1e-14, 1e-15, "mask-driven vs recomputed ReLU' " + name)


def pin_layernorm_cf_is_row_layernorm_of_the_transpose(o):
    # channels-first LayerNorm of x[n, c, l] = row LayerNorm of the [n*l, c] matrix
    # whose row (i, p) is x[i, :, p]; both sum the channels in the same order, so
    # the results agree to the last bit
    r = _rng(30)
    n, c, l = 3, 7, 11
    x = r.normal(size=(n, c, l)) * 1.4 + 0.3
    w = 1 + 0.2 * r.normal(size=c)
    b = 0.2 * r.normal(size=c)
    y, mean, rstd = o.layernorm_cf_fwd(x, w, b, eps=1e-5)
    rows = x.transpose(0, 2, 1).reshape(n * l, c)
    yr, mr, rr = o.layernorm_fwd(rows, w, b, eps=1e-5)
    _close(y, yr.reshape(n, l, c).transpose(0, 2, 1), 0, 0, "cf y == row y of the transpose")
    _close(mean.ravel(), mr, 0, 0, "cf mean")
    _close(rstd.ravel(), rr, 0, 0, "cf rstd")
    dy = r.normal(size=(n, c, l))
    dx, dw, db = o.layernorm_cf_bwd(dy, x, w, eps=1e-5)
    dxr, dwr, dbr = o.layernorm_bwd(dy.transpose(0, 2, 1).reshape(n * l, c), rows, w, eps=1e-5)
    _close(dx, dxr.reshape(n, l, c).transpose(0, 2, 1), 0, 0, "cf dx")
    _close(dw, dwr, 1e-15, 1e-15, "cf dw")
    _close(db, dbr, 1e-15, 1e-15, "cf db")


def pin_layernorm_cf_vs_torch(o):
    import torch
    F = torch.nn.functional
    r = _rng(31)
    n, c, l = 2, 5, 9
    x = torch.tensor(r.normal(size=(n, c, l)) * 2 - 0.5, requires_grad=True)
    w = torch.tensor(1 + 0.3 * r.normal(size=c), requires_grad=True)
    b = torch.tensor(0.3 * r.normal(size=c), requires_grad=True)
    y = F.layer_norm(x.permute(0, 2, 1), [c], w, b, eps=1e-6).permute(0, 2, 1)
    dy = r.normal(size=(n, c, l))
    y.backward(torch.from_numpy(dy))
    yo, _, _ = o.layernorm_cf_fwd(x.detach().numpy(), w.detach().numpy(), b.detach().numpy(), eps=1e-6)
    dx, dw, db = o.layernorm_cf_bwd(dy, x.detach().numpy(), w.detach().numpy(), eps=1e-6)
    _close(yo, y.detach().numpy(), 1e-12, 1e-13, "cf y vs torch")
    _close(dx, x.grad.numpy(), 1e-10, 1e-12, "cf dx vs torch")
    _close(dw, w.grad.numpy(), 1e-10, 1e-12, "cf dw vs torch")
    _close(db, b.grad.numpy(), 1e-10, 1e-12, "cf db vs torch")


def pin_layernorm_cf_bwd_fd(o):
    r = _rng(32)
    n, c, l = 2, 4, 3
    x = r.normal(size=(n, c, l)) + 0.2
    w = 1 + 0.3 * r.normal(size=c)
    b = 0.3 * r.normal(size=c)
    dy = r.normal(size=(n, c, l))

    def loss():
        return float((dy * o.layernorm_cf_fwd(x, w, b, eps=1e-3)[0]).sum())
    dx, dw, db = o.layernorm_cf_bwd(dy, x, w, eps=1e-3)
    _close(dx, _central_diff(loss, x, 1e-6), 1e-6, 1e-7, "cf dx vs FD")
    _close(dw, _central_diff(loss, w, 1e-6), 1e-6, 1e-7, "cf dw vs FD")
    _close(db, _central_diff(loss, b, 1e-6), 1e-6, 1e-7, "cf db vs FD")


# ---------------------------------------------------------------------------
# activation with fused dropout
# ---------------------------------------------------------------------------

def pin_philox_known_answers(o):
    """The generator against the published Philox4x32-10 known-answer vectors."""
    with open(os.path.join(GOLDEN, "philox4x32_10_known_answers.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        ctr = [int(v, 16) for v in case["ctr"]]
        key = [int(v, 16) for v in case["key"]]
        want = [int(v, 16) for v in case["out"]]
        got = [int(v) for v in o.philox4x32_10(ctr, key)]
        assert got == want, f"philox4x32-10 {case['ctr']} {case['key']}: {[hex(v) for v in got]}"


def pin_dropout_keep_rate(o):
    """Each element is kept with probability 1 - p (binomial bound, 6 sigma);
    p = 0 keeps everything and p = 1 nothing."""
    n = 200_000
    for p in (0.1, 0.5, 0.9):
        for seed in (0, 12345, 65535):
            kept = o.dropout_mask(n, p, seed).mean()
            sigma = (p * (1 - p) / n) ** 0.5
            assert abs(kept - (1 - p)) < 6 * sigma, f"keep rate {kept} for p={p}, seed={seed}"
    assert o.dropout_mask(1000, 0.0, 3).all()
    assert not o.dropout_mask(1000, 1.0, 3).any()


def pin_dropout_window_is_slice(o):
    """A window of elements starting at `first` gets the flags and values of
    that slice of the whole tensor (the random value belongs to the element's
    offset in the tensor)."""
    x = _rng(45).normal(size=1000)
    full_mask = o.dropout_mask(1000, 0.3, 21)
    full_y = o.act_dropout_fwd(x, 2, 0.3, 21)
    full_dx = o.act_dropout_bwd(np.ones(1000), x, 2, 0.3, 21)
    for first in (0, 1, 3, 4, 517):
        assert (o.dropout_mask(1000 - first, 0.3, 21, first=first) == full_mask[first:]).all()
        assert (o.act_dropout_fwd(x[first:], 2, 0.3, 21, first=first) == full_y[first:]).all()
        assert (o.act_dropout_bwd(np.ones(1000 - first), x[first:], 2, 0.3, 21, first=first)
                == full_dx[first:]).all()


def pin_dropout_independence(o):
    """Neighbouring elements (the same generator call), elements four apart (the
    next counter) and two seeds agree as often as independent fair coins do."""
    n = 200_000
    a = o.dropout_mask(n + 4, 0.5, 77).astype(bool)
    b = o.dropout_mask(n, 0.5, 78).astype(bool)
    sigma = (0.25 / n) ** 0.5
    for what, u, v in (("adjacent", a[:n], a[1:n + 1]), ("four apart", a[:n], a[4:n + 4]),
                       ("seeds", a[:n], b)):
        agree = float((u == v).mean())
        assert abs(agree - 0.5) < 6 * sigma, f"dropout masks {what}: agreement {agree}"


# torch evaluates CELU with 1/alpha held in single precision (its elu kernel's
# input scale: a relative error of about 3e-8 * |z/alpha| in e^(z/alpha)), so
# CELU is compared with torch to 1e-6 relative; the finite differences and the
# closed forms pin it exactly
def _torch_rtol(act, rtol):
    return max(rtol, 1e-6) if act in (8, "celu") else rtol


def _act_torch():
    """act code -> (torch function, the parameter passed to the oracle)."""
    import torch
    import torch.nn.functional as F
    lk, al, ca = ACT_PARAM["leaky_relu"], ACT_PARAM["elu"], ACT_PARAM["celu"]
    return {0: (lambda t: t, 0.0), 1: (torch.relu, 0.0), 2: (F.gelu, 0.0), 3: (F.silu, 0.0),
            4: (F.mish, 0.0), 5: (lambda t: F.leaky_relu(t, lk), lk), 6: (lambda t: F.elu(t, al), al),
            7: (torch.sigmoid, 0.0), 8: (lambda t: F.celu(t, ca), ca), 9: (F.selu, 0.0),
            10: (F.relu6, 0.0), 11: (F.hardtanh, 0.0)}


def pin_act_dropout_no_drop_is_activation(o):
    """p = 0: the kernel is the plain activation (torch's reference functions)."""
    import torch
    x = _rng(40).normal(size=4096) * 3
    for act, (fn, prm) in _act_torch().items():
        y = o.act_dropout_fwd(x, act, 0.0, 9, act_param=prm)
        _close(y, fn(torch.from_numpy(x)).numpy(), _torch_rtol(act, 1e-15), 1e-14, f"act {act} without dropout")


def pin_act_dropout_inverted_scale(o):
    """Kept elements are act(x) / (1 - p); dropped ones are 0; the mask is the
    generator's."""
    import torch
    x = _rng(41).normal(size=20000) * 2
    p = 0.25
    keep = o.dropout_mask(x.size, p, 4321).astype(bool)
    for act, (fn, prm) in _act_torch().items():
        y = o.act_dropout_fwd(x, act, p, 4321, act_param=prm)
        a = fn(torch.from_numpy(x)).numpy()
        _close(y[keep], a[keep] / (1 - p), _torch_rtol(act, 1e-15), 1e-14, f"act {act} kept elements")
        assert not y[~keep].any(), f"act {act}: dropped elements must be 0"
    # the mean is preserved in expectation (inverted dropout)
    xs = np.abs(_rng(42).normal(size=200_000)) + 1.0
    y = o.act_dropout_fwd(xs, 0, p, 5)
    assert abs(y.mean() - xs.mean()) < 6 * xs.std() * (p / (1 - p) / xs.size) ** 0.5 + 6 * xs.std() / xs.size ** 0.5


def pin_act_dropout_bwd_fd(o):
    """Backward = derivative of sum(dy * forward) with the seed held fixed."""
    r = _rng(43)
    x = r.normal(size=64) * 2
    # keep the kinks (0, and ReLU6's 6 and hardtanh's -1, 1) out of the stencil
    near = np.min([np.abs(x - k) for k in (-1.0, 0.0, 1.0, 6.0)], axis=0) < 0.05
    x = np.where(near, x + 0.3, x)
    dy = r.normal(size=64)
    for act, (_, prm) in _act_torch().items():
        for p in (0.0, 0.3):
            def loss():
                return float((dy * o.act_dropout_fwd(x, act, p, 11, act_param=prm)).sum())
            dx = o.act_dropout_bwd(dy, x, act, p, 11, act_param=prm)
            _close(dx, _central_diff(loss, x, 1e-6), 1e-7, 1e-7, f"act {act} p {p} dx vs FD")


def pin_act_dropout_bwd_vs_torch(o):
    """Backward against torch autograd of act(x) * keep / (1 - p)."""
    import torch
    r = _rng(44)
    x = torch.tensor(r.normal(size=5000) * 2, requires_grad=True)
    dy = r.normal(size=5000)
    p = 0.4
    keep = torch.from_numpy(o.dropout_mask(5000, p, 999).astype(np.float64))
    for act, (fn, prm) in _act_torch().items():
        if x.grad is not None:
            x.grad = None
        (fn(x) * keep / (1 - p)).backward(torch.from_numpy(dy))
        dx = o.act_dropout_bwd(dy, x.detach().numpy(), act, p, 999, act_param=prm)
        _close(dx, x.grad.numpy(), _torch_rtol(act, 1e-14), 1e-13, f"act {act} dx vs torch")


def _two_point(x1, x2, eps):
    """Standardising two values by hand: with u = (x1 - x2)/2 their biased
    variance is u^2, so xhat1 = u/sqrt(u^2 + eps) = -xhat2, and
    d xhat1 / d x1 = -d xhat1 / d x2 = eps / (2 (u^2 + eps)^(3/2))."""
    u = (x1 - x2) / 2
    return u / np.sqrt(u * u + eps), eps / (2 * (u * u + eps) ** 1.5), u


def pin_row_norms_one_and_two_columns(o):
    """Rows of one and two columns, worked by hand.  One column: LayerNorm's
    xhat is 0, so y = b, dx = 0, dw = 0, db = sum(dy), rstd = 1/sqrt(eps);
    RMSNorm's rstd is 1/sqrt(x^2 + eps) and dy/dx = w eps/(x^2 + eps)^(3/2).
    Two columns: the two-point standardisation of _two_point, whose
    derivative gives dx1 = -dx2 = (g1 - g2) eps/(2 (u^2 + eps)^(3/2)).
    The gaps u are taken below, near and above sqrt(eps), so that an eps
    placed outside the root, or a variance divided by N - 1, fails."""
    r = _rng(45)
    eps = 1e-2
    rows = 5
    # one column
    x = r.normal(size=(rows, 1)) * 3
    w = 1 + 0.4 * r.normal(size=1)
    b = 0.7 * r.normal(size=1)
    dy = r.normal(size=(rows, 1))
    y, mean, rstd = o.layernorm_fwd(x, w, b, eps=eps)
    _close(y, np.broadcast_to(b, (rows, 1)), 0, 1e-15, "one-column LayerNorm y = b")
    _close(mean, x[:, 0], 0, 0, "one-column LayerNorm mean")
    _close(rstd, np.full(rows, 1 / math.sqrt(eps)), 1e-15, 0, "one-column LayerNorm rstd")
    dx, dw, db = o.layernorm_bwd(dy, x, w, eps=eps)
    _close(dx, np.zeros_like(x), 0, 1e-15, "one-column LayerNorm dx = 0")
    _close(dw, np.zeros(1), 0, 1e-15, "one-column LayerNorm dw = 0")
    _close(db, dy.sum(0), 1e-14, 1e-15, "one-column LayerNorm db = sum dy")
    y, rstd = o.rmsnorm_fwd(x, w, eps=eps)
    _close(rstd, 1 / np.sqrt(x[:, 0] ** 2 + eps), 1e-14, 0, "one-column RMSNorm rstd")
    _close(y, x * w / np.sqrt(x * x + eps), 1e-14, 0, "one-column RMSNorm y")
    dx, dw = o.rmsnorm_bwd(dy, x, w, eps=eps)
    _close(dx, dy * w * eps / (x * x + eps) ** 1.5, 1e-13, 1e-16, "one-column RMSNorm dx")
    _close(dw, (dy * x / np.sqrt(x * x + eps)).sum(0), 1e-13, 1e-15, "one-column RMSNorm dw")
    # two columns: rows of centre m and half-gap u, in both orders
    m = r.uniform(-4, 4, size=rows)
    u = np.array([0.03, -0.08, 0.1, 0.4, -2.5])
    x = np.stack([m + u, m - u], axis=1)
    w = 1 + 0.4 * r.normal(size=2)
    b = 0.7 * r.normal(size=2)
    dy = r.normal(size=(rows, 2))
    xh1, dxh, _ = _two_point(x[:, 0], x[:, 1], eps)
    xh = np.stack([xh1, -xh1], axis=1)
    y, mean, rstd = o.layernorm_fwd(x, w, b, eps=eps)
    _close(y, xh * w + b, 1e-13, 1e-15, "two-column LayerNorm y")
    _close(mean, x.mean(1), 1e-15, 1e-15, "two-column LayerNorm mean")
    dx, dw, db = o.layernorm_bwd(dy, x, w, eps=eps)
    g = dy * w
    d1 = (g[:, 0] - g[:, 1]) * dxh
    _close(dx, np.stack([d1, -d1], axis=1), 1e-12, 1e-15, "two-column LayerNorm dx")
    _close(dw, (dy * xh).sum(0), 1e-13, 1e-15, "two-column LayerNorm dw")
    _close(db, dy.sum(0), 1e-14, 1e-15, "two-column LayerNorm db")


def pin_batchnorm_two_element_channels(o):
    """Channels of two elements (n = 2, l = 1 and n = 1, l = 2), worked by
    hand.  Training: the mean is the midpoint, xhat = +-u/sqrt(u^2 + eps),
    the running variance takes the unbiased 2u^2, and with no activation
    dx1 = -dx2 = w (dy1 - dy2) eps/(2 (u^2 + eps)^(3/2)), dw = (dy1 - dy2) xhat1,
    db = dy1 + dy2, dres = dy.  Eval: the running statistics replace the
    batch ones and dx = dy w / sqrt(rv + eps)."""
    r = _rng(46)
    eps, mom = 1e-2, 0.2
    c = 4
    u = np.array([0.05, -0.1, 0.3, 1.7])
    m = r.uniform(-3, 3, size=c)
    w = 1 + 0.3 * r.normal(size=c)
    b = 0.5 * r.normal(size=c)
    rm = r.normal(size=c)
    rv = r.uniform(0.5, 2, size=c)
    for n, l in ((2, 1), (1, 2)):
        pair = np.stack([m + u, m - u], axis=0)  # [2, c]: element k of each channel
        x = pair[:, :, None] if l == 1 else pair.T[None, :, :]
        res = r.normal(size=x.shape)
        dy = r.normal(size=x.shape)
        def el(t, k):  # element k of every channel of t
            return t[k, :, 0] if l == 1 else t[0, :, k]
        xh1, dxh, uu = _two_point(el(x, 0), el(x, 1), eps)
        f = o.batchnorm_fwd(x, res=res, w=w, b=b, eps=eps, momentum=mom, training=True,
                            running_mean=rm, running_var=rv)
        xh = np.stack([xh1, -xh1], axis=0)
        want_y = (xh * w + b)
        want_y = want_y[:, :, None] if l == 1 else want_y.T[None, :, :]
        _close(f["y"], want_y + res, 1e-13, 1e-15, f"BatchNorm [{n},{c},{l}] y")
        _close(f["save_mean"], m, 1e-15, 1e-15, f"BatchNorm [{n},{c},{l}] mean")
        _close(f["save_rstd"], 1 / np.sqrt(uu * uu + eps), 1e-14, 0, f"BatchNorm [{n},{c},{l}] rstd")
        _close(f["running_mean"], (1 - mom) * rm + mom * m, 1e-15, 1e-15, "running mean")
        _close(f["running_var"], (1 - mom) * rv + mom * 2 * uu * uu, 1e-14, 1e-16, "running var")
        dx, dres, dw, db = o.batchnorm_bwd(dy, x, res=res, w=w, b=b, eps=eps, training=True)
        dy1, dy2 = el(dy, 0), el(dy, 1)
        d1 = w * (dy1 - dy2) * dxh
        want_dx = np.stack([d1, -d1], axis=0)
        want_dx = want_dx[:, :, None] if l == 1 else want_dx.T[None, :, :]
        _close(dx, want_dx, 1e-12, 1e-15, f"BatchNorm [{n},{c},{l}] dx")
        _close(dres, dy, 0, 0, f"BatchNorm [{n},{c},{l}] dres = dy")
        _close(dw, (dy1 - dy2) * xh1, 1e-13, 1e-15, f"BatchNorm [{n},{c},{l}] dw")
        _close(db, dy1 + dy2, 1e-14, 1e-15, f"BatchNorm [{n},{c},{l}] db")
        # eval: the running statistics, untouched
        f = o.batchnorm_fwd(x, w=w, b=b, eps=eps, momentum=mom, training=False,
                            running_mean=rm, running_var=rv)
        k = 1 / np.sqrt(rv + eps)
        _close(f["y"], (x - rm[None, :, None]) * (k * w)[None, :, None] + b[None, :, None], 1e-14, 1e-15,
               f"BatchNorm [{n},{c},{l}] eval y")
        _close(f["running_mean"], rm, 0, 0, "eval leaves running mean")
        _close(f["running_var"], rv, 0, 0, "eval leaves running var")
        dx, _, dw, db = o.batchnorm_bwd(dy, x, w=w, b=b, running_mean=rm, running_var=rv, eps=eps,
                                        training=False)
        _close(dx, dy * (k * w)[None, :, None], 1e-14, 1e-16, f"BatchNorm [{n},{c},{l}] eval dx")
        _close(dw, (dy * (x - rm[None, :, None]) * k[None, :, None]).sum(axis=(0, 2)), 1e-13, 1e-15,
               f"BatchNorm [{n},{c},{l}] eval dw")
        _close(db, dy.sum(axis=(0, 2)), 1e-14, 1e-15, f"BatchNorm [{n},{c},{l}] eval db")


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
