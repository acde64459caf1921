// BatchNorm kernels for __nv_bfloat16 storage.
#include "batchnorm.cuh"
NRM_INSTANTIATE_BATCHNORM(__nv_bfloat16)
