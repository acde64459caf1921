// dropout.cu -- an activation with fused dropout, forward and backward, for
// every storage dtype (the activation-dropout article, "算子融合实战：attorch激活
// 函数与Dropout融合核的完整实现原理"):
//   y  = act(x) / (1 - p)         where element e is kept, else 0   (sections 三, 四)
//   dx = dy / (1 - p) * act'(x)   where element e is kept, else 0   (section 五)
// The mask is never stored: both passes rebuild it from the seed and the
// element's offset with a counter-based generator, Philox4x32-10 (Salmon,
// Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC 2011), keyed by (seed, 0) with counter (e / 4, 0, 0); element e takes
// output word e % 4 and is dropped when (word >> 8) * 2^-24 < p, tested here as
// the integer comparison word < ceil(p * 2^24) * 2^8, which decides the same
// (p = 1 drops everything and is a zero fill).
//
// GB300 design: an elementwise kernel over 16-byte vectors; a persistent grid
// of 256-thread CTAs walks the tensor, one vector per thread per iteration.
// One generator call covers four elements (its four output words).  With
// GELU, SiLU or Mish the kernel is bound by instruction issue (ten Philox
// rounds per four elements plus the activation), not by HBM.  Tensors that are
// not 16-byte aligned take a scalar kernel over groups of four elements.
#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "activation.cuh"
#include "common.cuh"
#include "internal.h"

namespace nrm {

constexpr int kDropThreads = 512;  // 128 / 256 / 512 measured 99.5 / 98.3 / 96.3 us (GELU forward, fp16 [25216,3072])

constexpr int kPhiloxRounds = 10;

struct DropArgs {
    const void* x;
    const void* dy;
    void* y;
    void* dx;
    int64_t count;
    // the key of each round: (seed, 0) advanced by the Weyl increments, computed
    // on the host (the key depends on the seed alone), read from the constant bank
    uint32_t rk0[kPhiloxRounds];
    uint32_t rk1[kPhiloxRounds];
    uint32_t thresh_w;  // ceil(p * 2^24) << 8: element kept when its word >= thresh_w (p < 1)
    int drop_all;       // p == 1: every element dropped
    float scale;        // 1 / (1 - p)
    float act_param;    // slope (leaky_relu) or alpha (elu, celu)
    int act;            // the activation (read by the run-time dispatched instantiation)
};

// Philox4x32 with 10 rounds on counter c, with the round keys of `a`.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const DropArgs& a) {
#pragma unroll
    for (int r = 0; r < kPhiloxRounds; ++r) {
        const uint64_t p0 = uint64_t(0xD2511F53u) * c.x;
        const uint64_t p1 = uint64_t(0xCD9E8D57u) * c.z;
        c = make_uint4(uint32_t(p1 >> 32) ^ c.y ^ a.rk0[r], uint32_t(p1), uint32_t(p0 >> 32) ^ c.w ^ a.rk1[r],
                       uint32_t(p0));
    }
    return c;
}

// The four random words of elements 4g .. 4g+3.
__device__ __forceinline__ uint4 drop_words(uint64_t g, const DropArgs& a) {
    return philox4x32_10(make_uint4(uint32_t(g), uint32_t(g >> 32), 0u, 0u), a);
}

__device__ __forceinline__ uint32_t word_of(const uint4& r, int k) {
    return k == 0 ? r.x : (k == 1 ? r.y : (k == 2 ? r.z : r.w));
}

// (word >> 8) < ceil(p * 2^24)  <=>  word < ceil(p * 2^24) * 2^8, for p < 1
template <int ACT, bool BWD>
__device__ __forceinline__ float drop_elem(float xv, float dyv, uint32_t word, const DropArgs& a) {
    if (word < a.thresh_w) return 0.f;
    if constexpr (BWD) return dyv * a.scale * act_derivative_c<ACT>(xv, a.act_param, a.act);
    else return act_forward_c<ACT>(xv, a.act_param, a.act) * a.scale;
}

// drop_elem for GELU on two elements at once: the same products in the same
// order (GELU(x)*scale, dy*scale*GELU'(x)), each lane bitwise drop_elem's.
template <bool BWD>
__device__ __forceinline__ float2 drop_pair_gelu(float2 xv, float2 dyv, uint32_t w0, uint32_t w1, const DropArgs& a) {
    float2 o;
    if constexpr (BWD) o = __fmul2_rn(__fmul2_rn(dyv, act_pair(a.scale)), gelu_grad2_f(xv));
    else o = __fmul2_rn(gelu2_f(xv), act_pair(a.scale));
    return make_float2(w0 < a.thresh_w ? 0.f : o.x, w1 < a.thresh_w ? 0.f : o.y);
}

// One element by scalar accesses (tails and unaligned tensors).
template <typename T, int ACT, bool BWD>
__device__ __forceinline__ void drop_scalar(const DropArgs& a, int64_t e, uint32_t word) {
    using bits = typename Io<T>::bits_t;
    const float xv = Io<T>::load(reinterpret_cast<const bits*>(a.x)[e]);
    const float dyv = BWD ? Io<T>::load(reinterpret_cast<const bits*>(a.dy)[e]) : 0.f;
    const float o = drop_elem<ACT, BWD>(xv, dyv, word, a);
    reinterpret_cast<bits*>(BWD ? a.dx : a.y)[e] = Io<T>::store(o);
}

// 16-byte vectors (every pointer 16-byte aligned); the count % V tail elements
// by scalar accesses.  The element arithmetic runs on fp32 pairs, converted
// from and to T two elements per instruction.  (Loading a thread's next
// vector before computing the current one was measured slower: the kernel is
// bound by instruction issue, not by load latency.)
template <typename T, int ACT, bool BWD>
__global__ void __launch_bounds__(kDropThreads)
act_dropout_vec_kernel(const DropArgs a) {
    constexpr int V = kVec<T>;  // elements per vector: 4 (fp32) or 8 (16-bit)
    constexpr int H = V / 2;
    const int64_t nvec = a.count / V;
    const int64_t stride = int64_t(gridDim.x) * kDropThreads;
    const int64_t t0 = int64_t(blockIdx.x) * kDropThreads + threadIdx.x;
    const T* x = reinterpret_cast<const T*>(a.x);
    const T* dy = reinterpret_cast<const T*>(a.dy);
    T* out = reinterpret_cast<T*>(BWD ? a.dx : a.y);
    for (int64_t v = t0; v < nvec; v += stride) {
        float2 xv[H], dv[H], o[H];
        unpack2<T>(ld_stream_v4(x + v * V), xv);
        if (BWD) unpack2<T>(ld_stream_v4(dy + v * V), dv);
#pragma unroll
        for (int q = 0; q < V / 4; ++q) {
            const uint4 r = drop_words(uint64_t(v) * (V / 4) + q, a);
#pragma unroll
            for (int k = 0; k < 4; k += 2) {
                const int h = 2 * q + k / 2;
                const float2 d = BWD ? dv[h] : make_float2(0.f, 0.f);
                if constexpr (ACT == NRM_ACT_GELU) {  // both elements on packed fp32
                    o[h] = drop_pair_gelu<BWD>(xv[h], d, word_of(r, k), word_of(r, k + 1), a);
                } else {
                    o[h] = make_float2(drop_elem<ACT, BWD>(xv[h].x, d.x, word_of(r, k), a),
                                       drop_elem<ACT, BWD>(xv[h].y, d.y, word_of(r, k + 1), a));
                }
            }
        }
        st_v4(out + v * V, pack2x<T>(o));
    }
    // the tail: fewer than V elements after the last whole vector
    const int64_t e = nvec * V + t0;
    if (e < a.count) drop_scalar<T, ACT, BWD>(a, e, word_of(drop_words(uint64_t(e) >> 2, a), int(e & 3)));
}

// Any alignment: groups of four elements (one generator call), scalar accesses.
template <typename T, int ACT, bool BWD>
__global__ void __launch_bounds__(kDropThreads)
act_dropout_scalar_kernel(const DropArgs a) {
    const int64_t groups = (a.count + 3) / 4;
    const int64_t stride = int64_t(gridDim.x) * kDropThreads;
    for (int64_t g = int64_t(blockIdx.x) * kDropThreads + threadIdx.x; g < groups; g += stride) {
        const uint4 r = drop_words(uint64_t(g), a);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t e = 4 * g + k;
            if (e < a.count) drop_scalar<T, ACT, BWD>(a, e, word_of(r, k));
        }
    }
}

template <typename T, bool BWD>
nrm_status act_dropout_launch(const DropArgs& a, int act, bool vec, cudaStream_t s) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    if (a.count == 0) return NRM_OK;
    if (a.drop_all)  // p = 1: every output is 0 (the oracle's y = 0, dx = 0)
        return cuda_status(cudaMemsetAsync(BWD ? a.dx : a.y, 0, size_t(a.count) * sizeof(T), s),
                           "activation-dropout zero fill");
    const void* fn = with_act(act, [&](auto tag) {
        constexpr int A = decltype(tag)::value;
        return vec ? (const void*)&act_dropout_vec_kernel<T, A, BWD>
                   : (const void*)&act_dropout_scalar_kernel<T, A, BWD>;
    });
    const int64_t items = vec ? a.count / kVec<T> : (a.count + 3) / 4;
    int64_t blocks = (items + kDropThreads - 1) / kDropThreads;
    const int occ = cached_occupancy(fn, kDropThreads, 0);
    if (occ <= 0) return fail(NRM_ERR_CUDA, "activation-dropout kernel cannot be resident");
    const int64_t cap = int64_t(occ) * d->sms;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;  // the vector kernel's tail needs a thread even with no whole vector
    DropArgs args = a;
    void* kargs[] = {&args};
    return cuda_status(cudaLaunchKernel(fn, dim3(unsigned(blocks)), dim3(kDropThreads), kargs, 0, s),
                       "activation-dropout launch");
}

nrm_status act_dropout(const void* x, const void* dy, void* out, int64_t count, int act, float act_param, float p,
                       uint32_t seed, nrm_dtype dt, bool bwd, bool vec, cudaStream_t s) {
    DropArgs a{};
    a.act_param = act_param;
    a.act = act;
    a.x = x;
    a.dy = dy;
    a.y = bwd ? nullptr : out;
    a.dx = bwd ? out : nullptr;
    a.count = count;
    uint32_t k0 = seed, k1 = 0u;
    for (int r = 0; r < kPhiloxRounds; ++r) {
        a.rk0[r] = k0;
        a.rk1[r] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    // p * 2^24 is exact in double; its ceiling is the smallest 24-bit value kept
    const uint32_t thresh = uint32_t(std::ceil(double(p) * 16777216.0));
    a.drop_all = thresh >= (1u << 24);
    a.thresh_w = a.drop_all ? 0u : thresh << 8;
    a.scale = a.drop_all ? 0.f : float(1.0 / (1.0 - double(p)));
    switch (dt) {
    case NRM_F32:
        return bwd ? act_dropout_launch<float, true>(a, act, vec, s) : act_dropout_launch<float, false>(a, act, vec, s);
    case NRM_F16:
        return bwd ? act_dropout_launch<__half, true>(a, act, vec, s) : act_dropout_launch<__half, false>(a, act, vec, s);
    default:
        return bwd ? act_dropout_launch<__nv_bfloat16, true>(a, act, vec, s)
                   : act_dropout_launch<__nv_bfloat16, false>(a, act, vec, s);
    }
}

}  // namespace nrm
