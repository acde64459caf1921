// noalloc.cu -- nrm_layernorm_bwd_noalloc: the LayerNorm backward for callers
// that cannot hand the library a workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: code that executes while another framework owns every allocation
// (a plugin or custom op inside a host runtime whose allocator may not be
// bypassed, or whose memory accounting a stray cudaMalloc would break), code
// that must not enter the allocator at all after start-up (hard real-time
// loops, where cudaMalloc can synchronise the device and stall for
// milliseconds), and code without any allocator API of its own (a C caller
// that was handed device pointers and nothing else).  This entry point gives
// them the LayerNorm backward with no workspace argument: the per-CTA dw/db
// partial rows live in a file-scope device array that the library owns.
//
// The scratch array is fixed at kNoAllocScratchFloats floats (8 MiB) and is
// held by every GPU that loads the library until the process exits.  The
// caller still passes all inputs and outputs.  Every call shares the one array:
// two calls that overlap on the GPU (on different streams without ordering
// between them) race on it and give wrong dw/db.  Calls in the same stream, or
// otherwise ordered, are safe.  Nothing in the array needs to start at zero:
// each call writes every partial-row element it later reads.
#include <initializer_list>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace {

// dw partial rows in the first half, db partial rows in the second.
constexpr size_t kNoAllocScratchFloats = size_t(1) << 21;  // 8 MiB
constexpr size_t kNoAllocHalf = kNoAllocScratchFloats / 2;
// Widest row accepted: leaves at least 16 partial rows per gradient.
constexpr int64_t kNoAllocMaxCols = int64_t(kNoAllocHalf / 16);

static __device__ __align__(256) float g_ln_bwd_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is a host-side stand-in, not a device address, so it is looked
// up once per device with that device current.
nrm_status scratch_address(int dev, float** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_ln_bwd_scratch);
        if (e != cudaSuccess) return nrm::cuda_status(e, "cudaGetSymbolAddress(scratch)");
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return NRM_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" nrm_status nrm_layernorm_bwd_noalloc(const void* dy, const void* x, const void* w,
                                                const float* mean, const float* rstd, void* dx,
                                                void* dw, void* db, int64_t rows, int64_t cols,
                                                nrm_dtype dt, nrm_stream_t stream) {
    using namespace nrm;
    clear_error();
    if (dt != NRM_F32 && dt != NRM_F16 && dt != NRM_BF16)
        return fail(NRM_ERR_INVALID_ARG, "unknown dtype %d", int(dt));
    if (rows < 0 || cols < 1) return fail(NRM_ERR_INVALID_ARG, "rows must be >= 0 and cols >= 1");
    if (cols > kNoAllocMaxCols)
        return fail(NRM_ERR_UNSUPPORTED,
                    "nrm_layernorm_bwd_noalloc supports at most %lld columns (its static scratch "
                    "is %zu floats); use nrm_layernorm_bwd with a workspace",
                    (long long)kNoAllocMaxCols, kNoAllocScratchFloats);
    if (rows > (int64_t(1) << 40) / cols) return fail(NRM_ERR_UNSUPPORTED, "rows*cols must be < 2^40");
    if (rows > 0 && (!dy || !x || !dx || !mean || !rstd))
        return fail(NRM_ERR_INVALID_ARG, "dy, x, dx, mean and rstd must not be NULL");
    const size_t es = dt == NRM_F32 ? 4 : 2;
    for (const void* p : std::initializer_list<const void*>{dy, x, dx, w, dw, db})
        if (p && !aligned(p, es)) return fail(NRM_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    if (!aligned(mean, 4) || !aligned(rstd, 4))
        return fail(NRM_ERR_INVALID_ARG, "mean and rstd must be 4-byte aligned");
    if (rows > 0 && (dx == dy || dx == x))
        return fail(NRM_ERR_INVALID_ARG, "in-place (dx == dy or x) is not supported");

    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    float* scratch = nullptr;
    nrm_status st = scratch_address(d->device, &scratch);
    if (st != NRM_OK) return st;

    RowArgs a{};
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
    a.ws_dw = scratch;
    a.ws_db = scratch + kNoAllocHalf;
    a.max_partials = int(kNoAllocHalf / size_t(cols));
    bool vec = (size_t(cols) * es) % 16 == 0;
    for (const void* p : std::initializer_list<const void*>{dy, x, dx, w})
        if (p && !aligned(p, 16)) vec = false;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (dt) {
    case NRM_F32: return row_bwd<float>(a, true, vec, s);
    case NRM_F16: return row_bwd<__half>(a, true, vec, s);
    case NRM_BF16: return row_bwd<__nv_bfloat16>(a, true, vec, s);
    }
    return fail(NRM_ERR_INVALID_ARG, "unknown dtype");
}
