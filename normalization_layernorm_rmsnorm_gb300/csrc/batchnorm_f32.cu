// BatchNorm kernels for float storage.
#include "batchnorm.cuh"
NRM_INSTANTIATE_BATCHNORM(float)

size_t nrm::batchnorm_workspace_bytes(const nrm::DevInfo& d, int64_t c) { return nrm::bn_workspace_bytes(d, c); }
