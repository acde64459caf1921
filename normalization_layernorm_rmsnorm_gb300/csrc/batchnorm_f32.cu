// BatchNorm kernels for float storage.
#include "batchnorm.cuh"
NRM_INSTANTIATE_BATCHNORM(float)
