// api.cu -- the C ABI of libnorm (declared in include/libnorm.h): argument
// checks, dispatch by storage dtype and alignment, per-device caches and status
// reporting.  The kernels live in rownorm_<dtype>.cu and batchnorm_<dtype>.cu.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

// Set by a kernel whose bounded wait gave up; read and cleared by nrm_sync_status.
__device__ unsigned int g_nrm_error_word = 0;

namespace nrm {

namespace {

thread_local char t_msg[512] = "";
std::mutex g_mu;
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices] = {};
std::map<std::tuple<int, const void*, int, size_t>, int> g_occ;
std::map<std::tuple<int, const void*, int, int, size_t>, int> g_clusters;
std::map<std::tuple<int, const void*>, std::pair<size_t, bool>> g_prepared;

constexpr int64_t kMaxElems = int64_t(1) << 40;

}  // namespace

void clear_error() { t_msg[0] = 0; }

thread_local uint64_t t_peer_test_ns = 0;

bool take_peer_wait_test(uint64_t* ns) {
    if (t_peer_test_ns == 0) return false;
    *ns = t_peer_test_ns;
    t_peer_test_ns = 0;
    return true;
}

nrm_status fail(nrm_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
    va_end(ap);
    return s;
}

nrm_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return NRM_OK;
    (void)cudaGetLastError();  // clear the launch error this call reports
    return fail(NRM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

const DevInfo* dev_info() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_ok[dev]) {
        DevInfo d{};
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        void* err = nullptr;
        if (cudaGetSymbolAddress(&err, g_nrm_error_word) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        d.err = static_cast<unsigned int*>(err);
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    return &g_dev[dev];
}

int cached_occupancy(const void* fn, int block, size_t smem) {
    const DevInfo* d = dev_info();
    if (!d) return 0;
    const auto key = std::make_tuple(d->device, fn, block, smem);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, block, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[key] = n;
    return n;
}

nrm_status prepare_kernel(const void* fn, size_t dyn_smem, bool nonportable_cluster) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    const auto key = std::make_tuple(d->device, fn);
    std::lock_guard<std::mutex> lk(g_mu);
    auto& st = g_prepared[key];
    if (dyn_smem > st.first) {
        // dynamic + static shared memory of a CTA may not exceed the opt-in limit
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return cuda_status(e, "cudaFuncGetAttributes");
        const size_t cap = size_t(d->max_smem_optin) - fa.sharedSizeBytes;
        if (dyn_smem > cap)
            return fail(NRM_ERR_UNSUPPORTED, "kernel needs %zu bytes of shared memory, %zu available",
                        dyn_smem, cap);
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(cap));
        if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(max dynamic smem)");
        st.first = cap;
    }
    if (nonportable_cluster && !st.second) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(non-portable cluster)");
        st.second = true;
    }
    return NRM_OK;
}

int max_active_clusters(const void* fn, int cs, int block, size_t smem) {
    const DevInfo* d = dev_info();
    if (!d) return 0;
    const auto key = std::make_tuple(d->device, fn, cs, block, smem);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_clusters.find(key);
        if (it != g_clusters.end()) return it->second;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(cs));
    cfg.blockDim = dim3(unsigned(block));
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_clusters[key] = n;
    return n;
}

nrm_status launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelExC(&cfg, fn, args), "dependent launch");
}

int row_bwd_max_partials(const DevInfo& d) { return 4 * d.sms; }

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}
}  // namespace

nrm_status encode_ncl_map(CUtensorMap* map, const void* base, size_t es, int64_t n, int64_t c, int64_t l,
                          int box_l, int box_c) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return fail(NRM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[3] = {cuuint64_t(l), cuuint64_t(c), cuuint64_t(n)};
    const cuuint64_t strides[2] = {cuuint64_t(l) * es, cuuint64_t(c) * cuuint64_t(l) * es};
    const cuuint32_t box[3] = {cuuint32_t(box_l), cuuint32_t(box_c), 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapDataType dt = es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    const CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NRM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return NRM_OK;
}

}  // namespace nrm

using namespace nrm;

namespace {

bool dtype_ok(nrm_dtype dt) { return dt == NRM_F32 || dt == NRM_F16 || dt == NRM_BF16; }
size_t dsize(nrm_dtype dt) { return dt == NRM_F32 ? 4 : 2; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool all_aligned(std::initializer_list<const void*> ptrs, size_t a) {
    for (const void* p : ptrs)
        if (p && !aligned(p, a)) return false;
    return true;
}

// rows*cols and friends: non-negative and below 2^40 elements, without overflow.
bool size_ok(int64_t a, int64_t b, int64_t c = 1) {
    if (a < 0 || b < 0 || c < 0) return false;
    if (a == 0 || b == 0 || c == 0) return true;
    if (a > kMaxElems / b) return false;
    return a * b <= kMaxElems / c;
}

nrm_status check_eps(float eps) {
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(NRM_ERR_INVALID_ARG, "eps must be finite and > 0");
    return NRM_OK;
}

nrm_status check_rows(int64_t rows, int64_t cols, nrm_dtype dt) {
    if (!dtype_ok(dt)) return fail(NRM_ERR_INVALID_ARG, "unknown dtype %d", int(dt));
    if (rows < 0) return fail(NRM_ERR_INVALID_ARG, "rows must be >= 0");
    if (cols < 1) return fail(NRM_ERR_INVALID_ARG, "cols must be >= 1");
    if (cols >= (int64_t(1) << 31)) return fail(NRM_ERR_UNSUPPORTED, "cols must be < 2^31");
    if (!size_ok(rows, cols)) return fail(NRM_ERR_UNSUPPORTED, "rows*cols must be < 2^40");
    return NRM_OK;
}

template <typename F>
nrm_status by_dtype(nrm_dtype dt, F&& f) {
    switch (dt) {
    case NRM_F32: return f(float{});
    case NRM_F16: return f(__half{});
    case NRM_BF16: return f(__nv_bfloat16{});
    }
    return fail(NRM_ERR_INVALID_ARG, "unknown dtype");
}

size_t row_ws_bytes(bool layernorm, int64_t cols) {
    const DevInfo* d = dev_info();
    if (!d) return 0;
    return size_t(row_bwd_max_partials(*d)) * size_t(cols) * sizeof(float) * (layernorm ? 2 : 1);
}

// The output's storage type: the input's, or fp32 for a 16-bit input.
nrm_status check_out_dtype(nrm_dtype dt, nrm_dtype out_dt) {
    if (!dtype_ok(out_dt)) return fail(NRM_ERR_INVALID_ARG, "unknown output dtype %d", int(out_dt));
    if (out_dt != dt && out_dt != NRM_F32)
        return fail(NRM_ERR_UNSUPPORTED, "the output dtype is the input's or float32");
    return NRM_OK;
}

nrm_status row_fwd_common(bool ln, const void* x, const void* w, const void* b, void* y, float* mean,
                          float* rstd, int64_t rows, int64_t cols, float eps, nrm_dtype dt,
                          nrm_stream_t stream, nrm_dtype y_dt) {
    t_msg[0] = 0;
    nrm_status st = check_rows(rows, cols, dt);
    if (st != NRM_OK) return st;
    if ((st = check_out_dtype(dt, y_dt)) != NRM_OK) return st;
    if ((st = check_eps(eps)) != NRM_OK) return st;
    if (rows > 0 && (!x || !y)) return fail(NRM_ERR_INVALID_ARG, "x and y must not be NULL");
    const size_t es = dsize(dt);
    const bool f32out = y_dt != dt;
    if (!all_aligned({x, w, b}, es) || !all_aligned({y}, dsize(y_dt)) || !all_aligned({mean, rstd}, 4))
        return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    if (rows > 0 && x == y) return fail(NRM_ERR_INVALID_ARG, "in-place (y == x) is not supported");
    const bool vec = (size_t(cols) * es) % 16 == 0 && all_aligned({x, y, w, b}, 16);
    RowArgs a{};
    a.x = x;
    a.w = w;
    a.b = b;  // RMSNorm's is optional
    a.y = y;
    a.mean = ln ? mean : nullptr;
    a.rstd = rstd;
    a.rows = rows;
    a.cols = int(cols);
    a.eps = eps;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (f32out) return by_dtype(dt, [&](auto tag) { return row_fwd_f32out<decltype(tag)>(a, ln, vec, s); });
    return by_dtype(dt, [&](auto tag) { return row_fwd<decltype(tag)>(a, ln, vec, s); });
}

nrm_status row_bwd_common(bool ln, const void* dy, const void* x, const void* w, const float* mean,
                          const float* rstd, void* dx, void* dw, void* db, int64_t rows, int64_t cols,
                          nrm_dtype dt, void* ws, size_t ws_bytes, nrm_stream_t stream, nrm_dtype dy_dt) {
    t_msg[0] = 0;
    nrm_status st = check_rows(rows, cols, dt);
    if (st != NRM_OK) return st;
    if ((st = check_out_dtype(dt, dy_dt)) != NRM_OK) return st;
    if (rows > 0 && (!dy || !x || !dx || !rstd || (ln && !mean)))
        return fail(NRM_ERR_INVALID_ARG, "dy, x, dx and the saved statistics must not be NULL");
    const size_t es = dsize(dt);
    const bool f32dy = dy_dt != dt;
    if (!all_aligned({x, dx, w, dw, db}, es) || !all_aligned({dy}, dsize(dy_dt)) || !all_aligned({mean, rstd}, 4))
        return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    if (rows > 0 && (dx == dy || dx == x))
        return fail(NRM_ERR_INVALID_ARG, "in-place (dx == dy or x) is not supported");
    const bool want = dw || db;
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    RowArgs a{};
    if (want && rows > 0) {
        const size_t need = row_ws_bytes(ln || db, cols);
        if (!ws || !aligned(ws, 16)) return fail(NRM_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned");
        if (ws_bytes < need)
            return fail(NRM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
        a.ws_dw = reinterpret_cast<float*>(ws);
        a.ws_db = (ln || db) ? a.ws_dw + size_t(row_bwd_max_partials(*d)) * size_t(cols) : nullptr;
    }
    const bool vec = (size_t(cols) * es) % 16 == 0 && all_aligned({dy, x, dx, w}, 16);
    a.x = x;
    a.w = w;
    a.dy = dy;
    a.dx = dx;
    a.mean_in = mean;
    a.rstd_in = rstd;
    a.dw = dw;
    a.db = db;
    a.rows = rows;
    a.cols = int(cols);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (f32dy) return by_dtype(dt, [&](auto tag) { return row_bwd_f32dy<decltype(tag)>(a, ln, vec, s); });
    return by_dtype(dt, [&](auto tag) { return row_bwd<decltype(tag)>(a, ln, vec, s); });
}

nrm_status check_cf_shape(int64_t n, int64_t c, int64_t l, nrm_dtype dt) {
    if (!dtype_ok(dt)) return fail(NRM_ERR_INVALID_ARG, "unknown dtype %d", int(dt));
    if (n < 0 || l < 0) return fail(NRM_ERR_INVALID_ARG, "n and l must be >= 0");
    if (c < 1) return fail(NRM_ERR_INVALID_ARG, "c must be >= 1");
    if (c > kCfMaxChannels) return fail(NRM_ERR_UNSUPPORTED, "c must be <= %d", kCfMaxChannels);
    if (!size_ok(n, c, l)) return fail(NRM_ERR_UNSUPPORTED, "n*c*l must be < 2^40");
    return NRM_OK;
}

nrm_status check_act(nrm_act act, float act_param) {
    if (int(act) < int(NRM_ACT_NONE) || int(act) > int(NRM_ACT_HARDTANH))
        return fail(NRM_ERR_INVALID_ARG, "unknown activation %d", int(act));
    if (!std::isfinite(act_param)) return fail(NRM_ERR_INVALID_ARG, "act_param must be finite");
    if (act == NRM_ACT_CELU && act_param == 0.f) return fail(NRM_ERR_INVALID_ARG, "CELU needs act_param != 0");
    return NRM_OK;
}

nrm_status check_bn_shape(int64_t n, int64_t c, int64_t l, nrm_dtype dt, int training, nrm_act act,
                          float act_param) {
    if (!dtype_ok(dt)) return fail(NRM_ERR_INVALID_ARG, "unknown dtype %d", int(dt));
    if (n < 0 || c < 0 || l < 0) return fail(NRM_ERR_INVALID_ARG, "n, c, l must be >= 0");
    if (!size_ok(n, c, l)) return fail(NRM_ERR_UNSUPPORTED, "n*c*l must be < 2^40");
    if (!size_ok(n, l) || (n > 0 && l > 0 && n * l >= (int64_t(1) << 31)))
        return fail(NRM_ERR_UNSUPPORTED, "a channel must hold fewer than 2^31 elements");
    if (c * 16 >= (int64_t(1) << 31)) return fail(NRM_ERR_UNSUPPORTED, "c must be < 2^27");
    if (nrm_status st = check_act(act, act_param); st != NRM_OK) return st;
    if (training && c > 0 && n * l < 2)
        return fail(NRM_ERR_INVALID_ARG, "training needs more than one value per channel (n*l >= 2)");
    return NRM_OK;
}

}  // namespace

extern "C" {

nrm_status nrm_layernorm_fwd(const void* x, const void* w, const void* b, void* y, float* mean,
                             float* rstd, int64_t rows, int64_t cols, float eps, nrm_dtype dt,
                             nrm_stream_t stream) {
    return row_fwd_common(true, x, w, b, y, mean, rstd, rows, cols, eps, dt, stream, dt);
}

nrm_status nrm_layernorm_bwd(const void* dy, const void* x, const void* w, const float* mean,
                             const float* rstd, void* dx, void* dw, void* db, int64_t rows,
                             int64_t cols, nrm_dtype dt, void* workspace, size_t workspace_bytes,
                             nrm_stream_t stream) {
    return row_bwd_common(true, dy, x, w, mean, rstd, dx, dw, db, rows, cols, dt, workspace,
                          workspace_bytes, stream, dt);
}

nrm_status nrm_layernorm_fwd_ex(const void* x, const void* w, const void* b, void* y, float* mean,
                                float* rstd, int64_t rows, int64_t cols, float eps, nrm_dtype dt,
                                nrm_dtype y_dt, nrm_stream_t stream) {
    return row_fwd_common(true, x, w, b, y, mean, rstd, rows, cols, eps, dt, stream, y_dt);
}

nrm_status nrm_layernorm_bwd_ex(const void* dy, const void* x, const void* w, const float* mean,
                                const float* rstd, void* dx, void* dw, void* db, int64_t rows,
                                int64_t cols, nrm_dtype dt, nrm_dtype dy_dt, void* workspace,
                                size_t workspace_bytes, nrm_stream_t stream) {
    return row_bwd_common(true, dy, x, w, mean, rstd, dx, dw, db, rows, cols, dt, workspace,
                          workspace_bytes, stream, dy_dt);
}

nrm_status nrm_layernorm_cf_fwd(const void* x, const void* w, const void* b, void* y, float* mean,
                                float* rstd, int64_t n, int64_t c, int64_t l, float eps, nrm_dtype dt,
                                nrm_stream_t stream) {
    t_msg[0] = 0;
    nrm_status st = check_cf_shape(n, c, l, dt);
    if (st != NRM_OK) return st;
    if ((st = check_eps(eps)) != NRM_OK) return st;
    const bool has_data = n > 0 && l > 0;
    if (has_data && (!x || !y)) return fail(NRM_ERR_INVALID_ARG, "x and y must not be NULL");
    const size_t es = dsize(dt);
    if (!all_aligned({x, y, w, b}, es) || !all_aligned({mean, rstd}, 4))
        return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    if (has_data && x == y) return fail(NRM_ERR_INVALID_ARG, "in-place (y == x) is not supported");
    CfArgs a{};
    a.x = x;
    a.w = w;
    a.b = b;
    a.y = y;
    a.mean = mean;
    a.rstd = rstd;
    a.n = n;
    a.c = c;
    a.l = l;
    a.eps = eps;
    const bool vec = (size_t(l) * es) % 16 == 0 && all_aligned({x, y}, 16);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return by_dtype(dt, [&](auto tag) { return cf_fwd<decltype(tag)>(a, vec, s); });
}

nrm_status nrm_layernorm_cf_bwd(const void* dy, const void* x, const void* w, const float* mean,
                                const float* rstd, void* dx, void* dw, void* db, int64_t n, int64_t c,
                                int64_t l, nrm_dtype dt, void* workspace, size_t workspace_bytes,
                                nrm_stream_t stream) {
    t_msg[0] = 0;
    nrm_status st = check_cf_shape(n, c, l, dt);
    if (st != NRM_OK) return st;
    const bool has_data = n > 0 && l > 0;
    if (has_data && (!dy || !x || !dx || !mean || !rstd))
        return fail(NRM_ERR_INVALID_ARG, "dy, x, dx and the saved statistics must not be NULL");
    const size_t es = dsize(dt);
    if (!all_aligned({dy, x, dx, w, dw, db}, es) || !all_aligned({mean, rstd}, 4))
        return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    if (has_data && (dx == dy || dx == x))
        return fail(NRM_ERR_INVALID_ARG, "in-place (dx == dy or x) is not supported");
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    CfArgs a{};
    if ((dw || db) && has_data) {
        const size_t need = row_ws_bytes(true, c);
        if (!workspace || !aligned(workspace, 16))
            return fail(NRM_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned");
        if (workspace_bytes < need)
            return fail(NRM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                        workspace_bytes, need);
        a.ws_dw = reinterpret_cast<float*>(workspace);
        a.ws_db = a.ws_dw + size_t(row_bwd_max_partials(*d)) * size_t(c);
    }
    a.x = x;
    a.w = w;
    a.dy = dy;
    a.dx = dx;
    a.mean_in = mean;
    a.rstd_in = rstd;
    a.dw = dw;
    a.db = db;
    a.n = n;
    a.c = c;
    a.l = l;
    const bool vec = (size_t(l) * es) % 16 == 0 && all_aligned({dy, x, dx}, 16);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return by_dtype(dt, [&](auto tag) { return cf_bwd<decltype(tag)>(a, vec, s); });
}

nrm_status nrm_rmsnorm_fwd(const void* x, const void* w, const void* b, void* y, float* rstd, int64_t rows,
                           int64_t cols, float eps, nrm_dtype dt, nrm_stream_t stream) {
    return row_fwd_common(false, x, w, b, y, nullptr, rstd, rows, cols, eps, dt, stream, dt);
}

nrm_status nrm_rmsnorm_bwd(const void* dy, const void* x, const void* w, const float* rstd, void* dx,
                           void* dw, void* db, int64_t rows, int64_t cols, nrm_dtype dt, void* workspace,
                           size_t workspace_bytes, nrm_stream_t stream) {
    return row_bwd_common(false, dy, x, w, nullptr, rstd, dx, dw, db, rows, cols, dt, workspace,
                          workspace_bytes, stream, dt);
}

nrm_status nrm_rmsnorm_fwd_ex(const void* x, const void* w, const void* b, void* y, float* rstd,
                              int64_t rows, int64_t cols, float eps, nrm_dtype dt, nrm_dtype y_dt,
                              nrm_stream_t stream) {
    return row_fwd_common(false, x, w, b, y, nullptr, rstd, rows, cols, eps, dt, stream, y_dt);
}

nrm_status nrm_rmsnorm_bwd_ex(const void* dy, const void* x, const void* w, const float* rstd, void* dx,
                              void* dw, void* db, int64_t rows, int64_t cols, nrm_dtype dt, nrm_dtype dy_dt,
                              void* workspace, size_t workspace_bytes, nrm_stream_t stream) {
    return row_bwd_common(false, dy, x, w, nullptr, rstd, dx, dw, db, rows, cols, dt, workspace,
                          workspace_bytes, stream, dy_dt);
}

nrm_status nrm_batchnorm_fwd(const void* x, const void* residual, const float* w, const float* b,
                             void* y, float* running_mean, float* running_var, float* save_mean,
                             float* save_rstd, uint32_t* act_mask, int64_t n, int64_t c, int64_t l,
                             float eps, float momentum, int training, nrm_act act, float act_param,
                             nrm_dtype dt, void* workspace, size_t workspace_bytes, nrm_stream_t stream) {
    t_msg[0] = 0;
    nrm_status st = check_bn_shape(n, c, l, dt, training, act, act_param);
    if (st != NRM_OK) return st;
    if ((st = check_eps(eps)) != NRM_OK) return st;
    if (!(momentum >= 0.f && momentum <= 1.f)) return fail(NRM_ERR_INVALID_ARG, "momentum must be in [0, 1]");
    const bool has_data = n > 0 && c > 0 && l > 0;
    if (has_data && (!x || !y)) return fail(NRM_ERR_INVALID_ARG, "x and y must not be NULL");
    if ((running_mean == nullptr) != (running_var == nullptr))
        return fail(NRM_ERR_INVALID_ARG, "running_mean and running_var must be both NULL or both set");
    if (!training && c > 0 && !running_mean)
        return fail(NRM_ERR_INVALID_ARG, "eval mode needs running_mean and running_var");
    if (act_mask && act != NRM_ACT_RELU) return fail(NRM_ERR_INVALID_ARG, "act_mask is only written for ReLU");
    const size_t es = dsize(dt);
    if (!all_aligned({x, residual, y}, es) ||
        !all_aligned({w, b, running_mean, running_var, save_mean, save_rstd, act_mask}, 4))
        return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    if (has_data && (x == y || (residual && residual == y)))
        return fail(NRM_ERR_INVALID_ARG, "in-place is not supported");
    if (c == 0) return NRM_OK;
    const bool vec = (size_t(l) * es) % 16 == 0 && all_aligned({x, residual, y}, 16);
    BnArgs a{};
    a.x = x;
    a.res = residual;
    a.w = w;
    a.b = b;
    a.y = y;
    a.rm = running_mean;
    a.rv = running_var;
    a.save_mean = save_mean;
    a.save_rstd = save_rstd;
    a.mask = act_mask;
    a.n = n;
    a.c = c;
    a.l = l;
    a.eps = eps;
    a.momentum = momentum;
    a.act = int(act);
    a.act_param = act_param;
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    a.err = d->err;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (workspace && !aligned(workspace, 16)) return fail(NRM_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    return by_dtype(dt, [&](auto tag) {
        return bn_fwd<decltype(tag)>(a, training != 0, vec, workspace, workspace_bytes, s);
    });
}

nrm_status nrm_batchnorm_bwd(const void* dy, const void* x, const void* residual, const float* w,
                             const float* b, const float* save_mean, const float* save_rstd,
                             const uint32_t* act_mask, void* dx, void* dres, float* dw, float* db,
                             int64_t n, int64_t c, int64_t l, int training, nrm_act act, float act_param,
                             nrm_dtype dt, void* workspace, size_t workspace_bytes, nrm_stream_t stream) {
    t_msg[0] = 0;
    nrm_status st = check_bn_shape(n, c, l, dt, training, act, act_param);
    if (st != NRM_OK) return st;
    const bool has_data = n > 0 && c > 0 && l > 0;
    if ((has_data && (!dy || !x || !dx)) || (c > 0 && (!save_mean || !save_rstd)))
        return fail(NRM_ERR_INVALID_ARG, "dy, x, dx, save_mean and save_rstd must not be NULL");
    if (act_mask && act != NRM_ACT_RELU) return fail(NRM_ERR_INVALID_ARG, "act_mask is only read for ReLU");
    const size_t es = dsize(dt);
    if (!all_aligned({dy, x, residual, dx, dres}, es) ||
        !all_aligned({w, b, save_mean, save_rstd, act_mask, dw, db}, 4))
        return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    if (has_data && (dx == dy || dx == x || (dres && (dres == dy || dres == x || dres == dx))))
        return fail(NRM_ERR_INVALID_ARG, "in-place is not supported");
    if (c == 0) return NRM_OK;
    const bool vec = (size_t(l) * es) % 16 == 0 && all_aligned({dy, x, residual, dx, dres}, 16);
    BnArgs a{};
    a.x = x;
    a.res = residual;
    a.w = w;
    a.b = b;
    a.dy = dy;
    a.dx = dx;
    a.dres = dres;
    a.dw = dw;
    a.db = db;
    a.mean_in = save_mean;
    a.rstd_in = save_rstd;
    a.mask_in = act_mask;
    a.n = n;
    a.c = c;
    a.l = l;
    a.act = int(act);
    a.act_param = act_param;
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    a.err = d->err;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (workspace && !aligned(workspace, 16)) return fail(NRM_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    return by_dtype(dt, [&](auto tag) {
        return bn_bwd<decltype(tag)>(a, training != 0, vec, workspace, workspace_bytes, s);
    });
}

size_t nrm_workspace_bytes(nrm_op op, int64_t rows, int64_t cols, nrm_dtype dt) {
    if (op != NRM_OP_LAYERNORM_BWD && op != NRM_OP_RMSNORM_BWD && op != NRM_OP_LAYERNORM_CF_BWD) return 0;
    if (check_rows(rows, cols, dt) != NRM_OK) return 0;
    if (op == NRM_OP_LAYERNORM_CF_BWD && cols > kCfMaxChannels) return 0;
    return row_ws_bytes(true, cols);  // dw and db partial rows (RMSNorm's db: the optional bias)
}

size_t nrm_batchnorm_workspace_bytes(int64_t n, int64_t c, int64_t l, nrm_dtype dt) {
    if (!dtype_ok(dt) || n < 0 || c < 0 || l < 0 || !size_ok(n, c, l)) return 0;
    const DevInfo* d = dev_info();
    if (!d) return 0;
    return batchnorm_workspace_bytes(*d, c);
}

namespace {
nrm_status check_act_dropout(int64_t count, nrm_act act, float act_param, float p, nrm_dtype dt) {
    if (!dtype_ok(dt)) return fail(NRM_ERR_INVALID_ARG, "unknown dtype %d", int(dt));
    if (count < 0) return fail(NRM_ERR_INVALID_ARG, "count must be >= 0");
    if (count >= (int64_t(1) << 40)) return fail(NRM_ERR_UNSUPPORTED, "count must be < 2^40");
    if (nrm_status st = check_act(act, act_param); st != NRM_OK) return st;
    if (!(p >= 0.f && p <= 1.f)) return fail(NRM_ERR_INVALID_ARG, "drop_p must be in [0, 1]");
    return NRM_OK;
}
}  // namespace

nrm_status nrm_act_dropout_fwd(const void* x, void* y, int64_t count, nrm_act act, float act_param, float drop_p,
                               uint32_t seed, nrm_dtype dt, nrm_stream_t stream) {
    t_msg[0] = 0;
    nrm_status st = check_act_dropout(count, act, act_param, drop_p, dt);
    if (st != NRM_OK) return st;
    if (count > 0 && (!x || !y)) return fail(NRM_ERR_INVALID_ARG, "x and y must not be NULL");
    const size_t es = dsize(dt);
    if (!all_aligned({x, y}, es)) return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    const bool vec = all_aligned({x, y}, 16);
    return act_dropout(x, nullptr, y, count, int(act), act_param, drop_p, seed, dt, false, vec,
                       reinterpret_cast<cudaStream_t>(stream));
}

nrm_status nrm_act_dropout_bwd(const void* dy, const void* x, void* dx, int64_t count, nrm_act act,
                               float act_param, float drop_p, uint32_t seed, nrm_dtype dt, nrm_stream_t stream) {
    t_msg[0] = 0;
    nrm_status st = check_act_dropout(count, act, act_param, drop_p, dt);
    if (st != NRM_OK) return st;
    if (count > 0 && (!dy || !x || !dx)) return fail(NRM_ERR_INVALID_ARG, "dy, x and dx must not be NULL");
    const size_t es = dsize(dt);
    if (!all_aligned({dy, x, dx}, es))
        return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    const bool vec = all_aligned({dy, x, dx}, 16);
    return act_dropout(x, dy, dx, count, int(act), act_param, drop_p, seed, dt, true, vec,
                       reinterpret_cast<cudaStream_t>(stream));
}

int64_t nrm_act_mask_words(int64_t n, int64_t c, int64_t l) {
    if (n < 0 || c < 0 || l < 0) return 0;
    return n * c * ((l + 31) / 32);
}

nrm_status nrm_sync_status(nrm_stream_t stream) {
    t_msg[0] = 0;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e, "stream synchronize");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_nrm_error_word, sizeof(word));
    if (e != cudaSuccess) return cuda_status(e, "reading the device error word");
    if (word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_nrm_error_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_status(e, "clearing the device error word");
        return fail(NRM_ERR_TIMEOUT, "a kernel's bounded wait gave up (code %u)", word);
    }
    return NRM_OK;
}

const char* nrm_status_str(nrm_status status) {
    switch (status) {
    case NRM_OK: return "NRM_OK";
    case NRM_ERR_INVALID_ARG: return "NRM_ERR_INVALID_ARG";
    case NRM_ERR_UNSUPPORTED: return "NRM_ERR_UNSUPPORTED";
    case NRM_ERR_WORKSPACE: return "NRM_ERR_WORKSPACE";
    case NRM_ERR_CUDA: return "NRM_ERR_CUDA";
    case NRM_ERR_TIMEOUT: return "NRM_ERR_TIMEOUT";
    }
    return "NRM_ERR_UNKNOWN";
}

const char* nrm_last_error_message(void) { return t_msg; }

nrm_status nrm_test_expire_peer_waits(uint64_t limit_ns) {
    t_msg[0] = 0;
    if (limit_ns == 0 || limit_ns > nrm::kPeerTestMaxNs)
        return fail(NRM_ERR_INVALID_ARG, "limit_ns must be in [1, %llu]", (unsigned long long)nrm::kPeerTestMaxNs);
    nrm::t_peer_test_ns = limit_ns;
    return NRM_OK;
}

int nrm_version(void) { return 100; }

}  // extern "C"
