// common.cuh -- device helpers shared by the libnorm kernels: storage-type
// traits, 128-bit global loads/stores, warp reductions, Chan's merge of
// (count, mean, M2) triples, float-float sums, mbarrier and bulk-copy
// wrappers, and division by a runtime constant.
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

// The element loops of the 16-byte vector paths work on pairs of fp32 values
// with Blackwell's packed FP32 instructions (add/mul/fma.rn.f32x2): two
// elements per instruction, each rounded as the scalar instruction would.
template <typename T> constexpr int kPairs = kVec<T> / 2;

template <typename T> __device__ __forceinline__ float2 cvt2(uint32_t w);
template <> __device__ __forceinline__ float2 cvt2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <> __device__ __forceinline__ float2 cvt2<__nv_bfloat16>(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}
template <typename T> __device__ __forceinline__ uint32_t pack2(float2 v);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float2 v) {
    const __half2 h = __float22half2_rn(v);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float2 v) {
    const __nv_bfloat162 h = __float22bfloat162_rn(v);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// 16 raw bytes as fp32 pairs.
template <typename T>
__device__ __forceinline__ void unpack2(const uint4 u, float2 (&v)[kPairs<T>]) {
    if constexpr (sizeof(T) == 4) {
        v[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        v[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    } else {
        v[0] = cvt2<T>(u.x);
        v[1] = cvt2<T>(u.y);
        v[2] = cvt2<T>(u.z);
        v[3] = cvt2<T>(u.w);
    }
}

// fp32 pairs rounded to T, as 16 raw bytes.
template <typename T>
__device__ __forceinline__ uint4 pack2x(const float2 (&o)[kPairs<T>]) {
    if constexpr (sizeof(T) == 4)
        return make_uint4(__float_as_uint(o[0].x), __float_as_uint(o[0].y), __float_as_uint(o[1].x),
                          __float_as_uint(o[1].y));
    else
        return make_uint4(pack2<T>(o[0]), pack2<T>(o[1]), pack2<T>(o[2]), pack2<T>(o[3]));
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 f2neg(float2 v) { return make_float2(-v.x, -v.y); }

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

// An unevaluated sum hi + lo of two floats (about 48 significant bits), added
// with Knuth's TwoSum and renormalised: sums that need more than fp32 stay on
// the fp32 pipe (double-precision throughput on this part is a small fraction
// of fp32).
struct FF {
    float hi, lo;
};
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (b.hi - bb);
    const float t = e + (a.lo + b.lo);
    const float hi = s + t;
    return FF{hi, t - (hi - s)};
}
// Sum over the warp (every lane gets it; the tree is fixed, so it is bitwise reproducible).
__device__ __forceinline__ FF ff_warp_sum(FF v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const FF w{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
        v = ff_add(v, w);
    }
    return v;
}
__device__ __forceinline__ double ff_to_double(FF v) { return double(v.hi) + double(v.lo); }

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
// L2 eviction priority (cache policies) for loads and stores
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_v4_policy(const void* p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint32_t ld_u32_policy(const void* p, uint64_t pol) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint16_t ld_u16_policy(const void* p, uint64_t pol) {
    uint16_t r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(r) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ void st_v4_policy(void* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol) : "memory");
}

__device__ __forceinline__ void st_v2_policy(void* p, uint2 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "l"(pol) : "memory");
}

// ---------------------------------------------------------------------------
// mbarriers and 1-D bulk copies (TMA) into shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}
// Makes initialised mbarriers visible to the async proxy (the TMA unit).
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}
// Non-blocking test: has the phase with parity `parity` completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}
// try_wait that may suspend the thread for up to `hint_ns` (it wakes when the
// phase completes): waiting threads issue no instructions meanwhile.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns) : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for phase `parity` of `bar` for at most `limit_ns`; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}
// As mbar_wait_bounded, suspending between polls instead of spinning.
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}
// Copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to this CTA's shared memory; completion is signalled on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses issued after a CTA barrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Cross-CTA signalling through global memory (all CTAs are co-resident).
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
// Loads that bypass L1 (data written by other CTAs during this kernel).
// Atomic add with acquire-release ordering at GPU scope; returns the old value.
__device__ __forceinline__ uint32_t atom_acq_rel_add_u32(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// One 4-byte asynchronous copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_addr(dst)), "l"(src) : "memory");
}
// Arrives on `bar` once this thread's earlier cp.async copies have landed; the
// barrier's expected count includes this arrival.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_addr(bar)) : "memory");
}
// ---------------------------------------------------------------------------
// thread-block clusters: rank, barrier, distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Barrier over every thread of the cluster (all threads must call it); orders
// shared-memory writes before it with reads by other CTAs after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of this CTA's shared variable `p` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
    return a;
}
// Split cluster barrier: arrive (relaxed: orders nothing) now, wait later.
// A CTA may write a peer's shared memory only once every CTA of the cluster
// has started, which the arrive at kernel start / wait before the first remote
// write establishes.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_dsmem_f4(uint32_t a, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" :: "r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_dsmem_d2(uint32_t a, double2 v) {
    asm volatile("st.shared::cluster.v2.f64 [%0], {%1,%2};" :: "r"(a), "d"(v.x), "d"(v.y) : "memory");
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ double2 ld_dsmem_d2(uint32_t a) {
    double2 v;
    asm volatile("ld.shared::cluster.v2.f64 {%0,%1}, [%2];" : "=d"(v.x), "=d"(v.y) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cg_f4(const float4* p) {
    float4 r;
    asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p) : "memory");
    return r;
}
__device__ __forceinline__ double2 ld_cg_d2(const double2* p) {
    double2 r;
    asm volatile("ld.global.cg.v2.f64 {%0,%1}, [%2];" : "=d"(r.x), "=d"(r.y) : "l"(p) : "memory");
    return r;
}


// Copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from this
// CTA's shared memory to global memory; completion is tracked by bulk groups.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 :: "l"(dst), "r"(smem_addr(src)), "r"(bytes), "l"(pol) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Device-side error codes reported through the library's error word.
constexpr unsigned int kErrTimeoutStage = 1u;
constexpr unsigned int kErrTimeoutPeers = 2u;

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace nrm
