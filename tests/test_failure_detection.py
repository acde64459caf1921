"""Failure detection of the BatchNorm kernels whose channels span several CTAs,
without a GPU fault.

Those kernels wait, bounded, for every CTA of a channel to publish its partial
sums.  nrm_test_expire_peer_waits arms, for the next training call on this
thread, a wait for one CTA more than the launch has and a short limit: every
waiting CTA then gives up, records the timeout, finishes its own part of the
call and waits for its own copies before it exits.  The tests check that the
timeout is reported (NRM_ERR_TIMEOUT from nrm_sync_status, after a run that
took about the armed limit), that the device stays usable, and that the next
call, unarmed, matches the oracle.  The arming itself and its argument check
need no GPU."""
import time

import pytest
import torch

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import synth
from parity_util import compare_bn, oracle_bn, run_bn

LIMIT_NS = 20_000_000  # 20 ms

# (dtype, n, c, l): 16-byte aligned channels that several CTAs share (the
# training ring kernels), and a shape whose segments are not 16-byte
# multiples and too long for the channel-group path (the scalar kernels)
CASES = [("f32", 64, 3, 3136), ("bf16", 32, 6, 1568), ("f16", 64, 2, 3001)]


def _inputs(dtype, n, c, l, seed):
    cfg = synth.BnConfig("fd", n, c, l, dtype, 1e-5, 0.1, seed=seed, act="relu", residual=True,
                         x_kind="offset_scale", w_std=0.2, b_std=0.2)
    return cfg, synth.bn_inputs(cfg)


@pytest.mark.gpu
@pytest.mark.parametrize("phase", ["fwd", "bwd"])
@pytest.mark.parametrize("case", CASES, ids=[f"{d}-{n}x{c}x{l}" for d, n, c, l in CASES])
def test_peer_wait_runs_out_reports_timeout_then_next_call_is_exact(orc, case, phase):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nrm.load()
    dtype, n, c, l = case
    cfg, inp = _inputs(dtype, n, c, l, seed=1100 + n + c)
    x = inp["x"].torch("cuda")
    res = inp["res"].torch("cuda")
    w, b, dy = inp["w"].torch("cuda"), inp["b"].torch("cuda"), inp["dy"].torch("cuda")
    rm, rv = inp["running_mean"].torch("cuda").clone(), inp["running_var"].torch("cuda").clone()
    y, dx, dres = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    sm, sr = torch.empty(c, device="cuda"), torch.empty(c, device="cuda")
    dw, db = torch.empty(c, device="cuda"), torch.empty(c, device="cuda")
    ws = nrm.batchnorm_workspace(x)

    def fwd():
        nrm.nrm_batchnorm_fwd(x, res, w, b, y, rm, rv, sm, sr, None, cfg.eps, cfg.momentum, True, "relu", ws)

    def bwd():
        nrm.nrm_batchnorm_bwd(dy, x, res, w, b, sm, sr, None, dx, dres, dw, db, True, "relu", ws)

    fwd()
    nrm.nrm_sync_status()
    nrm.nrm_test_expire_peer_waits(LIMIT_NS)
    t0 = time.perf_counter()
    (fwd if phase == "fwd" else bwd)()
    with pytest.raises(nrm.NrmError) as e:
        nrm.nrm_sync_status()
    waited = time.perf_counter() - t0
    assert e.value.status == nrm.NRM_ERR_TIMEOUT, str(e.value)
    # every CTA waited about the armed limit once (its later waits return at once)
    assert LIMIT_NS * 1e-9 <= waited < 2.0, f"the failed call took {waited:.3f} s"
    # the report was cleared, the context is usable, and an unarmed call is exact
    nrm.nrm_sync_status()
    got = run_bn(inp, dtype, cfg.eps, cfg.momentum, True, "relu", True, False)
    want = oracle_bn(orc, inp, cfg.eps, cfg.momentum, True, "relu", True)
    compare_bn(got, want, dtype, True, "relu", f"after a timed-out {phase} {dtype} [{n},{c},{l}]")


def test_arming_checks_its_limit():
    pytest.importorskip("ctypes")
    try:
        lib = nrm.load()
    except ImportError:
        pytest.skip("libnorm is not built")
    assert lib.nrm_test_expire_peer_waits(0) == nrm.NRM_ERR_INVALID_ARG
    assert lib.nrm_test_expire_peer_waits(10**9 + 1) == nrm.NRM_ERR_INVALID_ARG
    # arming needs no device; disarm by taking it on a thread that makes no call
    import threading
    out = []
    t = threading.Thread(target=lambda: out.append(lib.nrm_test_expire_peer_waits(1000)))
    t.start()
    t.join()
    assert out == [nrm.NRM_OK]
