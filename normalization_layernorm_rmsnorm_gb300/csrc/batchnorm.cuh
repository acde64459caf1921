// batchnorm.cuh -- BatchNorm over (batch, spatial) per channel of an NCHW
// tensor viewed as [n, c, l], with fused residual add and activation, forward
// and backward, for one storage dtype T (included by batchnorm_<dtype>.cu).
//
// What is computed follows the attorch normalization article
// ("attorch如何实现LayerNorm、BatchNorm与RMSNorm？3种归一化Triton核代码全解析"),
// section "BatchNorm：按特征并行 + 激活融合": one program per channel; the
// batch x spatial elements are visited block by block with an online
// mean/variance update (no second pass over the input for the statistics);
// running statistics follow an EMA with momentum in training and are read
// directly in eval; the residual (pre_act_add) and the activation are applied
// in the same kernel; the backward first undoes the activation.  The Welford
// update and the EMA form are those of the math-helper article
// ("如何用attorch.math快速开发自定义GPU算子：面向进阶开发者的算子融合实战指南",
// section "实战二 Welford EMA 组合手写 BatchNorm 融合统计").
//
// GB300 design:
//   * A channel (M = n*l elements, up to a few MB) is split over a thread-block
//     cluster of `cs` CTAs (up to 16, co-scheduled on one GPC).  The channel's
//     elements are numbered in blocks of 32 vectors (one vector per lane) within
//     each (sample, channel) segment; CTA rank r owns a contiguous range of
//     those blocks, and its warps take the blocks round-robin, kBnUnroll at a
//     time so several 16-byte loads per lane are in flight.
//   * Forward: the CTA keeps its slice of x in shared memory (up to ~220 KB) as
//     it streams it in, and folds every vector into per-thread (count, mean, M2)
//     with Chan's merge.  Warp, CTA and cluster partials are merged in a fixed
//     order, the cluster step over distributed shared memory, so every CTA gets
//     bit-identical statistics.  The normalise/affine/residual/activation pass
//     then reads x from shared memory: x crosses HBM once.
//   * Backward: dz = dy * act'(z) is formed once, written as dres, kept in
//     shared memory (fp32), and summed (sum dz, sum dz*(x-mean)) with Kahan
//     compensation; the cluster merges the sums in rank order; the dx pass reads
//     dz from shared memory and x again (an L2 hit: the cluster's slice was
//     read microseconds before).
//   * A slice larger than the shared-memory budget keeps what fits and reads
//     the rest from global memory twice.  Eval-mode forward needs no statistics
//     and runs without a cluster.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace nrm {

namespace cg = cooperative_groups;

constexpr int kBnThreads = 512;
constexpr int kBnWarps = kBnThreads / 32;
constexpr int kBnUnroll = 4;

// Geometry of one launch (device copy).
struct BnGeom {
    int64_t c;            // channels
    int lv;               // vectors per (sample, channel) segment = l / VE
    int nbs;              // blocks of 32 vectors per segment
    int words;            // ReLU-mask words per segment = ceil(l / 32)
    FastDiv div_nbs;      // division by nbs
    uint32_t nb_chan;     // blocks per channel = n * nbs
    int cs;               // CTAs per channel
    uint32_t stage_blocks;// blocks a CTA keeps in shared memory
    float inv_m;          // 1 / (n*l)
    float inv_m1;         // 1 / (n*l - 1)
};

__device__ __forceinline__ float act_forward(int act, float z) {
    if (act == NRM_ACT_RELU) return z > 0.f ? z : 0.f;
    if (act == NRM_ACT_GELU) return 0.5f * z * (1.f + erff(z * 0.70710678118654752f));
    return z;
}

// Derivative at the pre-activation value z (ReLU'(0) = 0).
__device__ __forceinline__ float act_derivative(int act, float z) {
    if (act == NRM_ACT_RELU) return z > 0.f ? 1.f : 0.f;
    if (act == NRM_ACT_GELU) {
        const float cdf = 0.5f * (1.f + erff(z * 0.70710678118654752f));
        const float pdf = expf(-0.5f * z * z) * 0.39894228040143268f;
        return fmaf(z, pdf, cdf);
    }
    return 1.f;
}

// Location of lane `lane` of block `bi` of channel `ch`.
struct BlockPos {
    uint32_t ni;      // sample
    uint32_t bs;      // block within the segment
    int v;            // vector within the segment
    int64_t seg;      // segment index ni*c + ch
};

__device__ __forceinline__ BlockPos block_pos(const BnGeom& g, uint32_t bi, int lane, int64_t ch) {
    BlockPos p;
    p.ni = fast_div(bi, g.div_nbs);
    p.bs = bi - p.ni * uint32_t(g.nbs);
    p.v = int(p.bs) * 32 + lane;
    p.seg = int64_t(p.ni) * g.c + ch;
    return p;
}

template <typename T, int VE>
__device__ __forceinline__ void raw_load(const T* base, int64_t vec_index, Pack<T, VE>& pk) {
    const T* p = base + vec_index * VE;
    if constexpr (VE > 1) {
        pk.u = ld_stream_v4(p);
    } else {
        pk.b[0] = *reinterpret_cast<const typename Io<T>::bits_t*>(p);
    }
}

template <typename T, int VE>
__device__ __forceinline__ void unpack(const Pack<T, VE>& pk, float (&v)[VE]) {
#pragma unroll
    for (int k = 0; k < VE; ++k) v[k] = Io<T>::load(pk.b[k]);
}

template <typename T, int VE>
__device__ __forceinline__ void stage_put(unsigned char* stage, uint32_t slot, const Pack<T, VE>& pk) {
    if constexpr (VE > 1) {
        reinterpret_cast<uint4*>(stage)[slot] = pk.u;
    } else {
        reinterpret_cast<typename Io<T>::bits_t*>(stage)[slot] = pk.b[0];
    }
}

template <typename T, int VE>
__device__ __forceinline__ void stage_get(const unsigned char* stage, uint32_t slot, Pack<T, VE>& pk) {
    if constexpr (VE > 1) {
        pk.u = reinterpret_cast<const uint4*>(stage)[slot];
    } else {
        pk.b[0] = reinterpret_cast<const typename Io<T>::bits_t*>(stage)[slot];
    }
}

// Packs bit k of `nib` (element lane*VE + k of the block) into the segment's
// mask words and stores them.  Called by the whole warp.
template <int VE>
__device__ __forceinline__ void store_mask_bits(uint32_t* mask, const BnGeom& g, const BlockPos& p,
                                                int lane, uint32_t nib) {
    uint32_t* seg_words = mask + p.seg * g.words;
    if constexpr (VE == 1) {
        const uint32_t word = __ballot_sync(0xffffffffu, nib != 0);
        if (lane == 0) seg_words[p.bs] = word;
    } else {
        const int q_mine = (lane * VE) >> 5;
        const uint32_t shifted = nib << ((lane * VE) & 31);
#pragma unroll
        for (int q = 0; q < VE; ++q) {
            const uint32_t word = __reduce_or_sync(0xffffffffu, q == q_mine ? shifted : 0u);
            const int wi = int(p.bs) * VE + q;
            if (lane == q && wi < g.words) seg_words[wi] = word;
        }
    }
}

// The VE mask bits of this lane's vector.
template <int VE>
__device__ __forceinline__ uint32_t load_mask_bits(const uint32_t* mask, const BnGeom& g,
                                                   const BlockPos& p, int lane) {
    const int e = lane * VE;  // element offset within the block's 32*VE elements
    const uint32_t word = mask[p.seg * g.words + int64_t(p.bs) * VE + (e >> 5)];
    return (word >> (e & 31)) & ((1u << VE) - 1u);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <typename T, int VE, bool TRAIN>
__global__ void __launch_bounds__(kBnThreads, 1)
bn_fwd_kernel(const BnArgs a, const BnGeom g) {
    extern __shared__ __align__(16) unsigned char stage[];
    __shared__ Moments warp_m[kBnWarps];
    __shared__ Moments cta_m;
    __shared__ float s_scale, s_shift;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = blockIdx.x % uint32_t(g.cs);
    const int64_t ch = blockIdx.x / uint32_t(g.cs);
    const uint32_t b0 = uint32_t(uint64_t(rank) * g.nb_chan / uint32_t(g.cs));
    const uint32_t b1 = uint32_t(uint64_t(rank + 1) * g.nb_chan / uint32_t(g.cs));
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);
    const float wc = a.w ? a.w[ch] : 1.f;
    const float bc = a.b ? a.b[ch] : 0.f;

    if constexpr (TRAIN) {
        // ---- pass over x: stage in shared memory, Welford/Chan per thread ----
        Moments m{0.f, 0.f, 0.f};
        for (uint32_t base = b0 + warp; base < b1; base += kBnWarps * kBnUnroll) {
            Pack<T, VE> pk[kBnUnroll];
            bool ok[kBnUnroll];
#pragma unroll
            for (int u = 0; u < kBnUnroll; ++u) {
                const uint32_t bi = base + u * kBnWarps;
                ok[u] = false;
                if (bi < b1) {
                    const BlockPos p = block_pos(g, bi, lane, ch);
                    if (p.v < g.lv) {
                        ok[u] = true;
                        raw_load<T, VE>(x, p.seg * g.lv + p.v, pk[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kBnUnroll; ++u) {
                if (!ok[u]) continue;
                const uint32_t bi = base + u * kBnWarps;
                if (bi - b0 < g.stage_blocks) stage_put<T, VE>(stage, (bi - b0) * 32 + lane, pk[u]);
                float v[VE];
                unpack<T, VE>(pk[u], v);
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < VE; ++k) s += v[k];
                const float vm = s * (1.f / VE);
                float q = 0.f;
#pragma unroll
                for (int k = 0; k < VE; ++k) q = fmaf(v[k] - vm, v[k] - vm, q);
                chan_merge(m, float(VE), vm, q);
            }
        }
        // ---- warp -> CTA -> cluster, fixed order ----
        warp_merge(m);
        if (lane == 0) warp_m[warp] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            Moments t = warp_m[0];
            for (int w = 1; w < kBnWarps; ++w) chan_merge(t, warp_m[w].n, warp_m[w].mean, warp_m[w].m2);
            cta_m = t;
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (threadIdx.x == 0) {
            Moments tot{0.f, 0.f, 0.f};
            for (int r = 0; r < g.cs; ++r) {
                const Moments* pm = cluster.map_shared_rank(&cta_m, r);
                chan_merge(tot, pm->n, pm->mean, pm->m2);
            }
            const float var = tot.m2 * g.inv_m;
            const float rs = rsqrtf(var + a.eps);
            s_scale = wc * rs;
            s_shift = bc - tot.mean * wc * rs;
            if (rank == 0) {
                if (a.save_mean) a.save_mean[ch] = tot.mean;
                if (a.save_rstd) a.save_rstd[ch] = rs;
                if (a.rm) a.rm[ch] = fmaf(a.momentum, tot.mean, (1.f - a.momentum) * a.rm[ch]);
                if (a.rv) a.rv[ch] = fmaf(a.momentum, tot.m2 * g.inv_m1, (1.f - a.momentum) * a.rv[ch]);
            }
        }
        // peers have read cta_m; s_scale/s_shift are visible to the CTA
        cluster.sync();
    } else {
        if (threadIdx.x == 0) {
            const float rs = rsqrtf(a.rv[ch] + a.eps);
            const float mu = a.rm[ch];
            s_scale = wc * rs;
            s_shift = bc - mu * wc * rs;
            if (rank == 0) {
                if (a.save_mean) a.save_mean[ch] = mu;
                if (a.save_rstd) a.save_rstd[ch] = rs;
            }
        }
        __syncthreads();
    }
    const float scale = s_scale;
    const float shift = s_shift;

    // ---- normalise, affine, residual, activation, store (+ ReLU mask) ----
    for (uint32_t base = b0 + warp; base < b1; base += kBnWarps * kBnUnroll) {
        Pack<T, VE> px[kBnUnroll], pr[kBnUnroll];
#pragma unroll
        for (int u = 0; u < kBnUnroll; ++u) {
            const uint32_t bi = base + u * kBnWarps;
            if (bi < b1) {
                const BlockPos p = block_pos(g, bi, lane, ch);
                if (p.v < g.lv) {
                    if (TRAIN && bi - b0 < g.stage_blocks)
                        stage_get<T, VE>(stage, (bi - b0) * 32 + lane, px[u]);
                    else
                        raw_load<T, VE>(x, p.seg * g.lv + p.v, px[u]);
                    if (res) raw_load<T, VE>(res, p.seg * g.lv + p.v, pr[u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBnUnroll; ++u) {
            const uint32_t bi = base + u * kBnWarps;
            if (bi >= b1) break;  // uniform across the warp
            const BlockPos p = block_pos(g, bi, lane, ch);
            uint32_t nib = 0;
            if (p.v < g.lv) {
                float v[VE], r[VE], o[VE];
                unpack<T, VE>(px[u], v);
                if (res) unpack<T, VE>(pr[u], r);
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    float z = fmaf(v[k], scale, shift);
                    if (res) z += r[k];
                    o[k] = act_forward(a.act, z);
                    nib |= uint32_t(z > 0.f) << k;
                }
                store_vec<T, VE>(y + (p.seg * g.lv + p.v) * VE, o);
            }
            if (a.mask) store_mask_bits<VE>(a.mask, g, p, lane, nib);
        }
    }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------

// dz for one lane's vector of block position p.
template <typename T, int VE>
__device__ __forceinline__ void form_dz(const BnArgs& a, const BnGeom& g, const BlockPos& p, int lane,
                                        bool need_z, float scale, float shift, const float (&dyv)[VE],
                                        const float (&xv)[VE], float (&dz)[VE]) {
    if (a.act == NRM_ACT_NONE) {
#pragma unroll
        for (int k = 0; k < VE; ++k) dz[k] = dyv[k];
        return;
    }
    if (a.act == NRM_ACT_RELU && !need_z) {
        const uint32_t bits = load_mask_bits<VE>(a.mask_in, g, p, lane);
#pragma unroll
        for (int k = 0; k < VE; ++k) dz[k] = ((bits >> k) & 1u) ? dyv[k] : 0.f;
        return;
    }
    float r[VE];
    if (a.res) {
        Pack<T, VE> pk;
        raw_load<T, VE>(reinterpret_cast<const T*>(a.res), p.seg * g.lv + p.v, pk);
        unpack<T, VE>(pk, r);
    } else {
#pragma unroll
        for (int k = 0; k < VE; ++k) r[k] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < VE; ++k) {
        const float z = fmaf(xv[k], scale, shift) + r[k];
        dz[k] = dyv[k] * act_derivative(a.act, z);
    }
}

template <typename T, int VE, bool TRAIN>
__global__ void __launch_bounds__(kBnThreads, 1)
bn_bwd_kernel(const BnArgs a, const BnGeom g) {
    extern __shared__ __align__(16) unsigned char stage_raw[];
    float* dz_stage = reinterpret_cast<float*>(stage_raw);
    __shared__ double warp_s[kBnWarps][2];
    __shared__ double cta_s[2];
    __shared__ float s_c1, s_c2;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = blockIdx.x % uint32_t(g.cs);
    const int64_t ch = blockIdx.x / uint32_t(g.cs);
    const uint32_t b0 = uint32_t(uint64_t(rank) * g.nb_chan / uint32_t(g.cs));
    const uint32_t b1 = uint32_t(uint64_t(rank + 1) * g.nb_chan / uint32_t(g.cs));
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ dy = reinterpret_cast<const T*>(a.dy);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    T* __restrict__ dres = reinterpret_cast<T*>(a.dres);

    const float mu = a.mean_in[ch];
    const float rs = a.rstd_in[ch];
    const float wc = a.w ? a.w[ch] : 1.f;
    const float bc = a.b ? a.b[ch] : 0.f;
    const float scale = wc * rs;
    const float shift = bc - mu * scale;
    const bool need_z = a.act == NRM_ACT_GELU || (a.act == NRM_ACT_RELU && a.mask_in == nullptr);

    // ---- undo the activation; dres; stage dz; channel sums ----
    Kahan s1, s2;
    for (uint32_t base = b0 + warp; base < b1; base += kBnWarps * kBnUnroll) {
        Pack<T, VE> pdy[kBnUnroll], px[kBnUnroll];
#pragma unroll
        for (int u = 0; u < kBnUnroll; ++u) {
            const uint32_t bi = base + u * kBnWarps;
            if (bi < b1) {
                const BlockPos p = block_pos(g, bi, lane, ch);
                if (p.v < g.lv) {
                    raw_load<T, VE>(dy, p.seg * g.lv + p.v, pdy[u]);
                    raw_load<T, VE>(x, p.seg * g.lv + p.v, px[u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBnUnroll; ++u) {
            const uint32_t bi = base + u * kBnWarps;
            if (bi >= b1) break;
            const BlockPos p = block_pos(g, bi, lane, ch);
            if (p.v >= g.lv) continue;
            float dyv[VE], xv[VE], dz[VE];
            unpack<T, VE>(pdy[u], dyv);
            unpack<T, VE>(px[u], xv);
            form_dz<T, VE>(a, g, p, lane, need_z, scale, shift, dyv, xv, dz);
            const int64_t e = (p.seg * g.lv + p.v) * VE;
            if (dres) store_vec<T, VE>(dres + e, dz);
            float t1 = 0.f, t2 = 0.f;
#pragma unroll
            for (int k = 0; k < VE; ++k) {
                t1 += dz[k];
                t2 = fmaf(dz[k], xv[k] - mu, t2);
            }
            s1.add(t1);
            s2.add(t2);
            if constexpr (TRAIN) {
                if (bi - b0 < g.stage_blocks) {
                    float* d = dz_stage + (size_t((bi - b0) * 32 + lane)) * VE;
#pragma unroll
                    for (int k = 0; k < VE; ++k) d[k] = dz[k];
                }
            } else {
                float o[VE];
#pragma unroll
                for (int k = 0; k < VE; ++k) o[k] = dz[k] * scale;
                store_vec<T, VE>(dx + e, o);
            }
        }
    }

    // ---- sums: thread -> warp -> CTA (double, fixed order) -> cluster ----
    double d1 = double(s1.s), d2 = double(s2.s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        d1 += __shfl_xor_sync(0xffffffffu, d1, o);
        d2 += __shfl_xor_sync(0xffffffffu, d2, o);
    }
    if (lane == 0) {
        warp_s[warp][0] = d1;
        warp_s[warp][1] = d2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t1 = 0.0, t2 = 0.0;
        for (int w = 0; w < kBnWarps; ++w) {
            t1 += warp_s[w][0];
            t2 += warp_s[w][1];
        }
        cta_s[0] = t1;
        cta_s[1] = t2;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (threadIdx.x == 0) {
        double t1 = 0.0, t2 = 0.0;
        for (int r = 0; r < g.cs; ++r) {
            const double* ps = cluster.map_shared_rank(&cta_s[0], r);
            t1 += ps[0];
            t2 += ps[1];
        }
        const float sum_dz = float(t1);
        const float sum_dz_xhat = float(t2 * double(rs));
        if (rank == 0) {
            if (a.db) a.db[ch] = sum_dz;
            if (a.dw) a.dw[ch] = sum_dz_xhat;
        }
        s_c1 = float(t1 * double(g.inv_m));
        s_c2 = float(t2 * double(rs) * double(g.inv_m));
    }
    cluster.sync();

    if constexpr (TRAIN) {
        // ---- dx = w*rstd*(dz - sum(dz)/M - xhat*sum(dz*xhat)/M) ----
        const float c1 = s_c1;
        const float c2 = s_c2;
        for (uint32_t base = b0 + warp; base < b1; base += kBnWarps * kBnUnroll) {
            Pack<T, VE> px[kBnUnroll], pdy[kBnUnroll];
#pragma unroll
            for (int u = 0; u < kBnUnroll; ++u) {
                const uint32_t bi = base + u * kBnWarps;
                if (bi < b1) {
                    const BlockPos p = block_pos(g, bi, lane, ch);
                    if (p.v < g.lv) {
                        raw_load<T, VE>(x, p.seg * g.lv + p.v, px[u]);
                        if (bi - b0 >= g.stage_blocks) raw_load<T, VE>(dy, p.seg * g.lv + p.v, pdy[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kBnUnroll; ++u) {
                const uint32_t bi = base + u * kBnWarps;
                if (bi >= b1) break;
                const BlockPos p = block_pos(g, bi, lane, ch);
                if (p.v >= g.lv) continue;
                float xv[VE], dz[VE], o[VE];
                unpack<T, VE>(px[u], xv);
                if (bi - b0 < g.stage_blocks) {
                    const float* d = dz_stage + (size_t((bi - b0) * 32 + lane)) * VE;
#pragma unroll
                    for (int k = 0; k < VE; ++k) dz[k] = d[k];
                } else {
                    float dyv[VE];
                    unpack<T, VE>(pdy[u], dyv);
                    form_dz<T, VE>(a, g, p, lane, need_z, scale, shift, dyv, xv, dz);
                }
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    const float xh = (xv[k] - mu) * rs;
                    o[k] = scale * (dz[k] - c1 - xh * c2);
                }
                store_vec<T, VE>(dx + (p.seg * g.lv + p.v) * VE, o);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Shared-memory budget for staging, leaving room for the static arrays.
inline size_t bn_stage_budget(const DevInfo& d) {
    const size_t cap = size_t(d.max_smem_optin);
    const size_t reserve = 2048;
    return cap > reserve ? cap - reserve : 0;
}

struct BnPlan {
    BnGeom g;
    size_t smem;
    int cluster;   // cluster size of the launch (1 = no cluster)
};

inline void bn_geometry(BnGeom& g, const BnArgs& a, int ve) {
    g.c = a.c;
    g.lv = int(a.l / ve);
    g.nbs = (g.lv + 31) / 32;
    g.words = int((a.l + 31) / 32);
    const FastDivHost f = make_fast_div(uint32_t(g.nbs > 0 ? g.nbs : 1));
    g.div_nbs.d = f.d;
    g.div_nbs.m = f.m;
    g.nb_chan = uint32_t(a.n * g.nbs);
    const double m = double(a.n) * double(a.l);
    g.inv_m = m > 0 ? float(1.0 / m) : 0.f;
    g.inv_m1 = m > 1 ? float(1.0 / (m - 1.0)) : 0.f;
}

// Picks the cluster size and the staged blocks.  `slot_bytes` is the shared
// memory one block occupies when staged (0: nothing is staged).
inline nrm_status bn_plan(BnPlan& pl, const BnArgs& a, int ve, size_t slot_bytes, bool use_cluster,
                          const void* fn) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    bn_geometry(pl.g, a, ve);
    BnGeom& g = pl.g;
    const uint32_t nb = g.nb_chan;
    const int64_t target_ctas = 2 * int64_t(d->sms);
    const size_t budget = bn_stage_budget(*d);
    const int max_cs = use_cluster ? 16 : 64;

    auto per_cta = [&](int cs) -> uint64_t { return (uint64_t(nb) + cs - 1) / cs; };
    int cs = 1;
    if (slot_bytes > 0) {
        while (cs < max_cs && per_cta(cs) * slot_bytes > budget) cs *= 2;
    }
    // more CTAs per channel while the GPU is not filled and each CTA keeps
    // at least one block per warp
    const int grow_limit = use_cluster ? 8 : 64;
    while (cs < grow_limit && a.c * cs < target_ctas && per_cta(cs * 2) >= uint64_t(kBnWarps)) cs *= 2;
    // every CTA owns at least one block when possible
    while (cs > 1 && uint64_t(cs) > nb) cs /= 2;

    for (;;) {
        const uint64_t fit = slot_bytes ? budget / slot_bytes : 0;
        const uint64_t want = per_cta(cs);
        g.cs = cs;
        g.stage_blocks = uint32_t(slot_bytes ? (want < fit ? want : fit) : 0);
        pl.smem = size_t(g.stage_blocks) * slot_bytes;
        pl.cluster = use_cluster ? cs : 1;
        nrm_status st = prepare_kernel(fn, pl.smem, pl.cluster > 8);
        if (st != NRM_OK) return st;
        if (!use_cluster || cs == 1) break;
        if (max_active_clusters(fn, cs, kBnThreads, pl.smem) > 0) break;
        cs /= 2;  // this cluster shape cannot be scheduled here: smaller cluster
    }
    return NRM_OK;
}

inline nrm_status launch_bn(const void* fn, const BnArgs& a, const BnPlan& pl, cudaStream_t s) {
    if (a.c == 0) return NRM_OK;
    BnArgs args = a;
    BnGeom geom = pl.g;
    void* kargs[] = {&args, &geom};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.c * pl.g.cs));
    cfg.blockDim = dim3(kBnThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(pl.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelExC(&cfg, fn, kargs), "batchnorm launch");
}

template <typename T>
nrm_status bn_fwd(const BnArgs& a, bool training, bool vec, cudaStream_t s) {
    const int ve = vec ? kVec<T> : 1;
    const void* fn;
    if (training)
        fn = vec ? (const void*)&bn_fwd_kernel<T, kVec<T>, true> : (const void*)&bn_fwd_kernel<T, 1, true>;
    else
        fn = vec ? (const void*)&bn_fwd_kernel<T, kVec<T>, false> : (const void*)&bn_fwd_kernel<T, 1, false>;
    BnPlan pl;
    const size_t slot = training ? size_t(32) * ve * sizeof(T) : 0;
    nrm_status st = bn_plan(pl, a, ve, slot, training, fn);
    if (st != NRM_OK) return st;
    return launch_bn(fn, a, pl, s);
}

template <typename T>
nrm_status bn_bwd(const BnArgs& a, bool training, bool vec, cudaStream_t s) {
    const int ve = vec ? kVec<T> : 1;
    const void* fn;
    if (training)
        fn = vec ? (const void*)&bn_bwd_kernel<T, kVec<T>, true> : (const void*)&bn_bwd_kernel<T, 1, true>;
    else
        fn = vec ? (const void*)&bn_bwd_kernel<T, kVec<T>, false> : (const void*)&bn_bwd_kernel<T, 1, false>;
    BnPlan pl;
    const size_t slot = training ? size_t(32) * ve * sizeof(float) : 0;
    nrm_status st = bn_plan(pl, a, ve, slot, true, fn);
    if (st != NRM_OK) return st;
    return launch_bn(fn, a, pl, s);
}

}  // namespace nrm

#define NRM_INSTANTIATE_BATCHNORM(T)                                                    \
    template nrm_status nrm::bn_fwd<T>(const nrm::BnArgs&, bool, bool, cudaStream_t);   \
    template nrm_status nrm::bn_bwd<T>(const nrm::BnArgs&, bool, bool, cudaStream_t);
