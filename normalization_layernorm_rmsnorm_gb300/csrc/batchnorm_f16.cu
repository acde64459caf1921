// BatchNorm kernels for __half storage.
#include "batchnorm.cuh"
NRM_INSTANTIATE_BATCHNORM(__half)
