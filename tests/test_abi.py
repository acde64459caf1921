"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/libnorm.h declares, and rejects bad arguments on the host before any
CUDA call.  CPU only (no compute calls)."""
import ctypes
import os
import re
import subprocess

import pytest

import normalization_layernorm_rmsnorm_gb300 as nrm
from normalization_layernorm_rmsnorm_gb300 import build as nbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "libnorm.h")


@pytest.fixture(scope="module")
def lib():
    nbuild.build()
    return nrm.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"NRM_API\s+[\w\s\*]+?\b(nrm_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(nrm.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", nbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (nrm_\w+)", out))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, f"not exported: {missing}"
    for f in declared_functions():
        assert hasattr(lib, f)
    # nothing else leaks out of the library's own code
    assert exported == set(declared_functions())


def test_header_compiles_as_c():
    src = f'#include "{HEADER}"\nint main(void) {{ return NRM_OK; }}\n'
    r = subprocess.run(["gcc", "-x", "c", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_and_sizes(lib):
    assert nrm.nrm_status_str(nrm.NRM_ERR_WORKSPACE) == "NRM_ERR_WORKSPACE"
    assert nrm.nrm_status_str(nrm.NRM_OK) == "NRM_OK"
    assert nrm.nrm_act_mask_words(256, 64, 3136) == 256 * 64 * 98
    assert nrm.nrm_act_mask_words(128, 512, 49) == 128 * 512 * 2
    assert nrm.nrm_act_mask_words(2, 3, 0) == 0
    assert nrm.nrm_version() >= 100


P = 1 << 20  # a fake, aligned, non-null address: never dereferenced (validation fails first)


@pytest.mark.parametrize("call,expect", [
    # null x / y
    (lambda L: L.nrm_layernorm_fwd(None, None, None, None, None, None, 4, 8, 1e-5, 0, None), 1),
    # cols = 0
    (lambda L: L.nrm_layernorm_fwd(P, None, None, P * 2, None, None, 4, 0, 1e-5, 0, None), 1),
    # negative rows
    (lambda L: L.nrm_rmsnorm_fwd(P, None, None, P * 2, None, -1, 8, 1e-5, 0, None), 1),
    # eps <= 0
    (lambda L: L.nrm_rmsnorm_fwd(P, None, None, P * 2, None, 4, 8, 0.0, 0, None), 1),
    # unknown dtype
    (lambda L: L.nrm_rmsnorm_fwd(P, None, None, P * 2, None, 4, 8, 1e-5, 7, None), 1),
    # element-misaligned fp32 pointer
    (lambda L: L.nrm_layernorm_fwd(P + 2, None, None, P * 2, None, None, 4, 8, 1e-5, 0, None), 1),
    # in place
    (lambda L: L.nrm_layernorm_fwd(P, None, None, P, None, None, 4, 8, 1e-5, 0, None), 1),
    # cols too large
    (lambda L: L.nrm_layernorm_fwd(P, None, None, P * 2, None, None, 1, 1 << 31, 1e-5, 0, None), 2),
    # backward without saved statistics
    (lambda L: L.nrm_layernorm_bwd(P, P * 2, None, None, None, P * 3, None, None, 4, 8, 0, None, 0,
                                   None), 1),
    # training BatchNorm with one value per channel
    (lambda L: L.nrm_batchnorm_fwd(P, None, None, None, P * 2, None, None, None, None, None, 1, 3,
                                   1, 1e-5, 0.1, 1, 0, 0.0, 0, None, 0, None), 1),
    # running_mean without running_var
    (lambda L: L.nrm_batchnorm_fwd(P, None, None, None, P * 2, P * 3, None, None, None, None, 2, 3,
                                   4, 1e-5, 0.1, 1, 0, 0.0, 0, None, 0, None), 1),
    # eval without running statistics
    (lambda L: L.nrm_batchnorm_fwd(P, None, None, None, P * 2, None, None, None, None, None, 2, 3,
                                   4, 1e-5, 0.1, 0, 0, 0.0, 0, None, 0, None), 1),
    # momentum out of range
    (lambda L: L.nrm_batchnorm_fwd(P, None, None, None, P * 2, None, None, None, None, None, 2, 3,
                                   4, 1e-5, 1.5, 1, 0, 0.0, 0, None, 0, None), 1),
    # a mask for GELU
    (lambda L: L.nrm_batchnorm_fwd(P, None, None, None, P * 2, None, None, None, None, P * 3, 2, 3,
                                   4, 1e-5, 0.1, 1, 2, 0.0, 0, None, 0, None), 1),
    # unknown activation
    (lambda L: L.nrm_batchnorm_bwd(P, P * 2, None, None, None, P * 3, P * 4, None, P * 5, None, None,
                                   None, 2, 3, 4, 1, 12, 0.0, 0, None, 0, None), 1),
    # a channel with 2^31 elements
    (lambda L: L.nrm_batchnorm_fwd(P, None, None, None, P * 2, None, None, None, None, None,
                                   1 << 16, 1, 1 << 15, 1e-5, 0.1, 1, 0, 0.0, 0, None, 0, None), 2),
    # channels-first LayerNorm with no channels
    (lambda L: L.nrm_layernorm_cf_fwd(P, None, None, P * 2, None, None, 2, 0, 5, 1e-5, 0, None), 1),
    # dropout probability above 1, NaN, negative count, unknown activation, null y
    (lambda L: L.nrm_act_dropout_fwd(P, P * 2, 16, 2, 0.0, 1.5, 7, 1, None), 1),
    (lambda L: L.nrm_act_dropout_fwd(P, P * 2, 16, 2, 0.0, float("nan"), 7, 1, None), 1),
    (lambda L: L.nrm_act_dropout_bwd(P, P * 2, P * 3, -1, 2, 0.0, 0.5, 7, 1, None), 1),
    (lambda L: L.nrm_act_dropout_bwd(P, P * 2, P * 3, 16, 12, 0.0, 0.5, 7, 1, None), 1),
    (lambda L: L.nrm_act_dropout_fwd(P, None, 16, 2, 0.0, 0.5, 7, 1, None), 1),
    # a non-finite activation parameter (BatchNorm and dropout)
    (lambda L: L.nrm_batchnorm_fwd(P, None, None, None, P * 2, None, None, None, None, None, 2, 3,
                                   4, 1e-5, 0.1, 1, 5, float("inf"), 0, None, 0, None), 1),
    (lambda L: L.nrm_act_dropout_fwd(P, P * 2, 16, 6, float("nan"), 0.5, 7, 1, None), 1),
    # CELU with alpha 0, an activation past the last one
    (lambda L: L.nrm_act_dropout_fwd(P, P * 2, 16, 8, 0.0, 0.5, 7, 1, None), 1),
    (lambda L: L.nrm_act_dropout_fwd(P, P * 2, 16, 12, 0.0, 0.5, 7, 1, None), 1),
    # an fp32 input with a 16-bit output (only 16-bit inputs may widen), an unknown output dtype
    (lambda L: L.nrm_layernorm_fwd_ex(P, None, None, P * 2, None, None, 4, 8, 1e-5, 0, 1, None), 2),
    (lambda L: L.nrm_rmsnorm_fwd_ex(P, None, None, P * 2, None, 4, 8, 1e-5, 1, 5, None), 1),
    # element-misaligned fp16 pointer
    (lambda L: L.nrm_act_dropout_fwd(P + 1, P * 2, 16, 2, 0.0, 0.5, 7, 1, None), 1),
])
def test_bad_arguments_are_rejected_on_the_host(lib, call, expect):
    assert call(lib) == expect
    assert nrm.nrm_last_error_message() != ""


def test_workspace_query_without_a_device_returns_zero(lib):
    # no GPU in this process: the query reports 0 rather than failing
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert nrm.nrm_workspace_bytes(nrm.NRM_OP_LAYERNORM_BWD, 64, 256, nrm.NRM_F32) == 0
