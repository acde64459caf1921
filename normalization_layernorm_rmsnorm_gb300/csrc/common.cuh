// common.cuh -- device helpers shared by the libnorm kernels: storage-type
// traits, 128-bit global loads/stores, warp reductions, Chan's merge of
// (count, mean, M2) triples, Kahan accumulation and division by a runtime
// constant.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace nrm {

// ---------------------------------------------------------------------------
// storage types: raw bits in memory, float32 in registers
// ---------------------------------------------------------------------------

template <typename T> struct Io;

template <> struct Io<float> {
    using bits_t = uint32_t;
    static __device__ __forceinline__ float load(bits_t b) { return __uint_as_float(b); }
    static __device__ __forceinline__ bits_t store(float v) { return __float_as_uint(v); }
};

template <> struct Io<__half> {
    using bits_t = uint16_t;
    static __device__ __forceinline__ float load(bits_t b) { return __half2float(__ushort_as_half(b)); }
    static __device__ __forceinline__ bits_t store(float v) { return __half_as_ushort(__float2half_rn(v)); }
};

template <> struct Io<__nv_bfloat16> {
    using bits_t = uint16_t;
    static __device__ __forceinline__ float load(bits_t b) { return __uint_as_float(uint32_t(b) << 16); }
    static __device__ __forceinline__ bits_t store(float v) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
};

// Elements per 128-bit access.
template <typename T> constexpr int kVec = 16 / int(sizeof(T));

// A vector of VE elements: one 128-bit access when VE == kVec<T>, else VE
// scalar accesses (the path for unaligned tensors uses VE == 1).
template <typename T, int VE>
union Pack {
    static_assert(VE == 1 || VE == kVec<T>, "VE is 1 or a full 16-byte vector");
    uint4 u;
    typename Io<T>::bits_t b[VE];
};

// Streaming read-only load: the data is read once, so keep it out of L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Read-only load that may hit L1 (small tensors re-read by every row: w, b).
__device__ __forceinline__ uint4 ld_cached_v4(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

template <typename T, int VE, bool STREAM = true>
__device__ __forceinline__ void load_vec(const T* p, float (&out)[VE]) {
    Pack<T, VE> pk;
    if constexpr (VE == kVec<T> && VE > 1) {
        pk.u = STREAM ? ld_stream_v4(p) : ld_cached_v4(p);
    } else {
        const typename Io<T>::bits_t* q = reinterpret_cast<const typename Io<T>::bits_t*>(p);
#pragma unroll
        for (int k = 0; k < VE; ++k) pk.b[k] = STREAM ? q[k] : __ldg(q + k);
    }
#pragma unroll
    for (int k = 0; k < VE; ++k) out[k] = Io<T>::load(pk.b[k]);
}

template <typename T, int VE>
__device__ __forceinline__ void store_vec(T* p, const float (&in)[VE]) {
    Pack<T, VE> pk;
#pragma unroll
    for (int k = 0; k < VE; ++k) pk.b[k] = Io<T>::store(in[k]);
    if constexpr (VE == kVec<T> && VE > 1) {
        st_v4(p, pk.u);
    } else {
        typename Io<T>::bits_t* q = reinterpret_cast<typename Io<T>::bits_t*>(p);
#pragma unroll
        for (int k = 0; k < VE; ++k) q[k] = pk.b[k];
    }
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------

// Butterfly sum over a full warp.  Every lane ends with the same bits (IEEE
// addition is commutative, and each level adds the same two partial sums).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Named barrier over `nthreads` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Running (count, mean, M2) of a set of values; merged with Chan et al.'s
// pairwise formula, the blockwise Welford update the articles describe.
struct Moments {
    float n;
    float mean;
    float m2;
};

__device__ __forceinline__ void chan_merge(Moments& a, float nb, float meanb, float m2b) {
    const float nt = a.n + nb;
    if (nb == 0.f) return;
    const float f = nb / nt;
    const float d = meanb - a.mean;
    a.mean = fmaf(d, f, a.mean);
    a.m2 = a.m2 + m2b + d * d * a.n * f;
    a.n = nt;
}

// Warp-level merge; lane 0 holds the result.
__device__ __forceinline__ void warp_merge(Moments& m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float nb = __shfl_down_sync(0xffffffffu, m.n, o);
        const float mb = __shfl_down_sync(0xffffffffu, m.mean, o);
        const float qb = __shfl_down_sync(0xffffffffu, m.m2, o);
        chan_merge(m, nb, mb, qb);
    }
}

// Compensated (Kahan) float accumulation.
struct Kahan {
    float s = 0.f;
    float c = 0.f;
    __device__ __forceinline__ void add(float v) {
        const float y = v - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
};

// ---------------------------------------------------------------------------
// division of 32-bit unsigned integers by a runtime constant d < 2^32:
// q = floor(n * m / 2^64) with m = floor((2^64 - 1) / d) + 1 (exact for n < 2^32)
// ---------------------------------------------------------------------------
struct FastDiv {
    uint32_t d;
    uint64_t m;
};

__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
    return f.d == 1u ? n : uint32_t(__umul64hi(uint64_t(n), f.m));
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace nrm
