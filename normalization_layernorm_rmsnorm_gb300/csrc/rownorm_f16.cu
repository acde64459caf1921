// LayerNorm / RMSNorm kernels for __half storage.
#include "rownorm.cuh"
NRM_INSTANTIATE_ROWNORM(__half)
