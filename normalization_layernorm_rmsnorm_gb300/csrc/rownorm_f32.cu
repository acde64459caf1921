// LayerNorm / RMSNorm kernels for float storage.
#include "rownorm.cuh"
NRM_INSTANTIATE_ROWNORM(float)
