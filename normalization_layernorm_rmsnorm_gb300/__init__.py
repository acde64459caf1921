"""libnorm for GB300: LayerNorm (rows and channels first), RMSNorm, BatchNorm
(with fused residual and activation) and an activation with fused dropout,
forward and backward, as hand-written sm_103a CUDA kernels behind a C ABI
(include/libnorm.h).

This package holds the CUDA sources (``csrc/``), their build (``build.py``),
the ctypes binding of the C ABI (``_binding``, re-exported here under the C
names) and the seeded synthetic input generator (``synth``).
"""
from ._binding import (  # noqa: F401
    ACTS, EXPORTS, LIB_PATH, NRM_ACT_ELU, NRM_ACT_GELU, NRM_ACT_LEAKY_RELU, NRM_ACT_MISH, NRM_ACT_NONE,
    NRM_ACT_RELU, NRM_ACT_SILU,
    NRM_BF16, NRM_ERR_CUDA,
    NRM_ERR_INVALID_ARG, NRM_ERR_TIMEOUT, NRM_ERR_UNSUPPORTED, NRM_ERR_WORKSPACE, NRM_F16,
    NRM_F32, NRM_OK, NRM_OP_LAYERNORM_BWD, NRM_OP_LAYERNORM_CF_BWD, NRM_OP_RMSNORM_BWD, NrmError, batchnorm_workspace, load,
    nrm_act_dropout_bwd, nrm_act_dropout_fwd, nrm_act_mask_words, nrm_batchnorm_bwd, nrm_batchnorm_fwd, nrm_batchnorm_workspace_bytes, nrm_last_error_message,
    nrm_layernorm_bwd, nrm_layernorm_bwd_ex, nrm_layernorm_bwd_noalloc, nrm_layernorm_fwd_ex, nrm_rmsnorm_bwd_ex, nrm_rmsnorm_fwd_ex, nrm_layernorm_cf_bwd, nrm_layernorm_cf_fwd, nrm_layernorm_fwd, nrm_rmsnorm_bwd, nrm_rmsnorm_fwd, nrm_status_str,
    nrm_sync_status, nrm_test_expire_peer_waits, nrm_version, nrm_workspace_bytes,
)
