// internal.h -- host-side declarations shared by the C ABI (api.cu) and the
// per-dtype kernel translation units.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; the driver is reached through the runtime)
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "libnorm.h"

namespace nrm {

// Properties of the current device, read once per device.
struct DevInfo {
    int device;
    int sms;
    int max_smem_optin;   // bytes of dynamic shared memory a CTA may opt into
    unsigned int* err;    // device address of the library's error word
};
const DevInfo* dev_info();  // nullptr if no usable device

// Clears this thread's last error message (at the start of an entry point).
void clear_error();
// Records a human-readable reason for the status returned to the caller.
nrm_status fail(nrm_status s, const char* fmt, ...);
// Maps a CUDA error to NRM_ERR_CUDA with its message (NRM_OK for cudaSuccess).
nrm_status cuda_status(cudaError_t e, const char* what);

// Failure-path test hook (nrm_test_expire_peer_waits): the wait limit armed on
// this thread for the next BatchNorm launch that waits for other CTAs, if any;
// taking it disarms it.
constexpr uint64_t kPeerTestMaxNs = 1000000000ull;  // 1 s
extern thread_local uint64_t t_peer_test_ns;
bool take_peer_wait_test(uint64_t* ns);

// Resident CTAs per SM of kernel `fn` (cached per device and kernel).
int cached_occupancy(const void* fn, int block, size_t smem);
// Opts `fn` into `dyn_smem` bytes of dynamic shared memory and, if asked, into
// non-portable cluster sizes (once per device and kernel).
nrm_status prepare_kernel(const void* fn, size_t dyn_smem, bool nonportable_cluster);
// Clusters of `cs` CTAs of `fn` (kBnThreads threads, `smem` bytes) that fit at once.
int max_active_clusters(const void* fn, int cs, int block, size_t smem);
// Launch with programmatic stream serialisation (the kernel waits on its
// predecessor with griddepcontrol.wait, so its launch overlaps the predecessor).
nrm_status launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t s);

// Host copy of the device-side FastDiv.
struct FastDivHost {
    uint32_t d;
    uint64_t m;
};
inline FastDivHost make_fast_div(uint32_t d) {
    FastDivHost f;
    f.d = d;
    f.m = d <= 1 ? 0 : (~uint64_t(0)) / d + 1;
    return f;
}

// ---------------------------------------------------------------------------
// row norms (LayerNorm, RMSNorm)
// ---------------------------------------------------------------------------
struct RowArgs {
    const void* x;
    const void* w;
    const void* b;
    const void* dy;
    void* y;
    void* dx;
    float* mean;          // forward outputs (nullable)
    float* rstd;
    const float* mean_in; // backward inputs
    const float* rstd_in;
    float* ws_dw;         // backward: per-CTA partial rows [P][cols] (nullable)
    float* ws_db;
    void* dw;             // backward outputs in the storage dtype (nullable)
    void* db;
    int64_t rows;
    int cols;
    float eps;
    int max_partials;     // backward: cap on the partial rows P (0 = no cap)
    unsigned int* err;    // device error word (set by the launcher; bounded waits that gave up)
};

// LayerNorm over the channels of x[n, c, l] (channels first, l = H*W).
// The backward keeps a CTA's dw/db partial row (2*c floats) in shared memory.
constexpr int64_t kCfMaxChannels = 16384;
struct CfArgs {
    const void* x;
    const void* w;        // [c] in the storage dtype (nullable)
    const void* b;
    const void* dy;
    void* y;
    void* dx;
    float* mean;          // forward outputs [n*l] (nullable)
    float* rstd;
    const float* mean_in; // backward inputs [n*l]
    const float* rstd_in;
    float* ws_dw;         // backward: per-CTA partial rows [P][c] (nullable)
    float* ws_db;
    void* dw;             // backward outputs [c] in the storage dtype (nullable)
    void* db;
    int64_t n, c, l;
    float eps;
    unsigned int* err;    // device error word (bounded waits that gave up)
};

// A 3-D tiled TMA map of a [n, c, l] tensor of es-byte elements (dims {l, c, n},
// box {box_l, box_c, 1}, out-of-range elements read as zero).  The base must be
// 16-byte aligned and l*es a multiple of 16.
nrm_status encode_ncl_map(CUtensorMap* map, const void* base, size_t es, int64_t n, int64_t c, int64_t l,
                          int box_l, int box_c);

// Activation with fused dropout (dropout.cu): out = y (forward) or dx (backward).
nrm_status act_dropout(const void* x, const void* dy, void* out, int64_t count, int act, float act_param, float p,
                       uint32_t seed, nrm_dtype dt, bool bwd, bool vec, cudaStream_t s);

template <typename T> nrm_status cf_fwd(const CfArgs& a, bool vec, cudaStream_t s);
template <typename T> nrm_status cf_bwd(CfArgs a, bool vec, cudaStream_t s);

// Upper bound of per-CTA partial rows of the row-norm backward (P).
int row_bwd_max_partials(const DevInfo& d);

// One entry per storage dtype (defined in rownorm_<dtype>.cu).
template <typename T> nrm_status row_fwd(const RowArgs& a, bool layernorm, bool vec,
                                         cudaStream_t s);
template <typename T> nrm_status row_bwd(RowArgs a, bool layernorm, bool vec, cudaStream_t s);
// The same with the forward's output, and so the backward's dy, held in fp32
// for a 16-bit input (the autocast_to_fp32-style option).
template <typename T> nrm_status row_fwd_f32out(const RowArgs& a, bool layernorm, bool vec, cudaStream_t s);
template <typename T> nrm_status row_bwd_f32dy(RowArgs a, bool layernorm, bool vec, cudaStream_t s);

// ---------------------------------------------------------------------------
// BatchNorm
// ---------------------------------------------------------------------------
struct BnArgs {
    const void* x;
    const void* res;
    const float* w;
    const float* b;
    void* y;
    float* rm;
    float* rv;
    float* save_mean;
    float* save_rstd;
    uint32_t* mask;
    const void* dy;
    void* dx;
    void* dres;
    float* dw;
    float* db;
    const float* mean_in;
    const float* rstd_in;
    const uint32_t* mask_in;
    int64_t n, c, l;
    float eps;
    float momentum;
    int act;
    float act_param;      // slope (leaky_relu) or alpha (elu)
    unsigned int* err;    // device error word (bounded waits that gave up)
};

template <typename T> nrm_status bn_fwd(const BnArgs& a, bool training, bool vec, void* ws, size_t ws_bytes,
                                        cudaStream_t s);
template <typename T> nrm_status bn_bwd(const BnArgs& a, bool training, bool vec, void* ws, size_t ws_bytes,
                                        cudaStream_t s);
// Workspace bytes that suffice for any BatchNorm call with c channels.
size_t batchnorm_workspace_bytes(const DevInfo& d, int64_t c);

}  // namespace nrm
