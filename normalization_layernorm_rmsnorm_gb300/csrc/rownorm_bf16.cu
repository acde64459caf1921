// LayerNorm / RMSNorm kernels for __nv_bfloat16 storage.
#include "rownorm.cuh"
NRM_INSTANTIATE_ROWNORM(__nv_bfloat16)
