// batchnorm.cuh -- BatchNorm over (batch, spatial) per channel of an NCHW
// tensor viewed as [n, c, l], with fused residual add and activation, forward
// and backward, for one storage dtype T (included by batchnorm_<dtype>.cu).
//
// What is computed follows the attorch normalization article
// ("attorch如何实现LayerNorm、BatchNorm与RMSNorm？3种归一化Triton核代码全解析"),
// section "BatchNorm：按特征并行 + 激活融合": statistics per channel over the
// batch x spatial elements, gathered block by block with an online update (one
// pass over the input for the statistics); running statistics follow an EMA
// with momentum in training and are read directly in eval; the residual
// (pre_act_add) and the activation are applied in the same kernel; the backward
// first undoes the activation.  The Welford update and the EMA form are those
// of the math-helper article ("如何用attorch.math快速开发自定义GPU算子：面向进阶
// 开发者的算子融合实战指南", section "实战二 Welford EMA 组合手写 BatchNorm 融合统计").
//
// GB300 design (kernel families, chosen per call):
//   * Training, 16-byte vectors (batchnorm_train.cuh): a persistent
//     cooperative grid, one CTA per SM.  A channel is cut into S slices, one
//     per CTA; the grid holds a whole number k of channels, so the S slices of
//     a channel run in the same round on different CTAs.  Inside a CTA one
//     team of warps makes the first pass of round q (statistics, or the
//     gradient sums; data from HBM, kept in L2) while another makes the
//     second pass of an earlier round (apply, or dx; data re-read from L2),
//     each team fed by its own producer warp and ring of shared-memory slots;
//     a bookkeeper warp publishes the CTA's partial sums (release counter per
//     channel), merges a channel's S partials in one fixed order once they
//     have all arrived and hands the second team the coefficients.
//   * Eval forward, 16-byte vectors (bn_fwd_eval_stream_kernel below): the
//     output is elementwise once the running statistics fix the coefficients,
//     so warps stream blocks of vectors through registers with a per-CTA table
//     of (scale, shift) in dynamic shared memory; more than kEsMaxChannels
//     channels take the ring kernel below.
//   * Eval backward, 16-byte vectors (bn_bwd_eval_kernel below), and the eval
//     forward for very many channels (bn_fwd_eval_kernel): the same rings with
//     one pass per round, coefficients from the running statistics.
//   * Channel-group kernels (batchnorm_group.cuh): short segments, staged
//     whole in shared memory by a thread-block cluster per channel group.
//   * Scalar kernels (bn_fwd_kernel / bn_bwd_kernel with VE = 1): tensors not
//     aligned to 16 bytes, with the same cooperative schedule and L2 staging.
//   * Statistics: per-thread sums of (x - K) and (x - K)^2 about the thread's
//     first value K, turned into (n, mean, M2) and merged with Chan's formula.
//     Backward sums: sum(dz) and sum(dz*(x - mean)), centred on the saved
//     mean (no cancellation), in fp32 per thread and float-float / double
//     across threads, CTAs and slices.
#pragma once

#include "activation.cuh"
#include "common.cuh"
#include "internal.h"

namespace nrm {

constexpr int kBnThreads = 512;
constexpr int kBnWarps = kBnThreads / 32;
constexpr int kBnUnroll = 8;        // blocks per warp in flight when streaming one tensor from HBM
constexpr int kBnUnroll2 = 6;       // ... two tensors
constexpr int kBnUnrollL2 = 4;      // ... when re-reading data that sits in L2
constexpr uint64_t kBnWaitLimitNs = 2000000000ull;  // 2 s

// Geometry and schedule of one launch (device copy).
struct BnGeom {
    int64_t c;             // channels
    int lv;                // vectors per (sample, channel) segment = l / VE
    int nbs;               // blocks of 32 vectors per segment
    int words;             // ReLU-mask words per segment = ceil(l / 32)
    FastDiv div_nbs;       // division by nbs
    uint32_t nb_chan;      // blocks per channel = n * nbs
    int S;                 // slices (CTAs) per channel
    int rounds;            // items per CTA: item = blockIdx.x + r * gridDim.x
    float inv_m;           // 1 / (n*l)
    float inv_m1;          // 1 / (n*l - 1)
    uint32_t* counters;    // [c] arrivals per channel, zero at launch (S > 1)
    void* partials;        // [c][S]: float4 (n, mean, m2, 0) forward; double2 backward
    uint32_t peer_extra;   // arrivals awaited beyond S (0; 1 under the failure-path test hook)
    uint64_t peer_wait_ns; // how long a CTA waits for a channel's other slices before giving up
};

// Whether the backward recomputes z = x*scale + shift (+ residual) to take the
// activation's derivative (every activation but none, and ReLU with a mask).
__host__ __device__ __forceinline__ bool bn_need_z(int act, const void* mask_in) {
    return act != NRM_ACT_NONE && !(act == NRM_ACT_RELU && mask_in != nullptr);
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
__device__ __forceinline__ void raw_load_pol(const T* base, int64_t vec_index, Pack<T, VE>& pk,
                                             uint64_t pol) {
    const T* p = base + vec_index * VE;
    if constexpr (VE > 1) {
        pk.u = ld_v4_policy(p, pol);
    } else if constexpr (sizeof(T) == 4) {
        pk.b[0] = ld_u32_policy(p, pol);
    } else {
        pk.b[0] = ld_u16_policy(p, pol);
    }
}

template <typename T, int VE>
__device__ __forceinline__ void unpack(const Pack<T, VE>& pk, float (&v)[VE]) {
#pragma unroll
    for (int k = 0; k < VE; ++k) v[k] = Io<T>::load(pk.b[k]);
}

template <typename T, int VE>
__device__ __forceinline__ void store_vec_pol(T* p, const float (&in)[VE], uint64_t pol) {
    Pack<T, VE> pk;
#pragma unroll
    for (int k = 0; k < VE; ++k) pk.b[k] = Io<T>::store(in[k]);
    if constexpr (VE > 1) {
        st_v4_policy(p, pk.u, pol);
    } else {
        *reinterpret_cast<typename Io<T>::bits_t*>(p) = pk.b[0];
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
                                                   const BlockPos& p, int lane, uint64_t pol) {
    const int e = lane * VE;  // element offset within the block's 32*VE elements
    const uint32_t word = ld_u32_policy(mask + p.seg * g.words + int64_t(p.bs) * VE + (e >> 5), pol);
    return (word >> (e & 31)) & ((1u << VE) - 1u);
}

__device__ __forceinline__ void slice_range(const BnGeom& g, int s, uint32_t& b0, uint32_t& b1) {
    b0 = uint32_t(uint64_t(s) * g.nb_chan / uint32_t(g.S));
    b1 = uint32_t(uint64_t(s + 1) * g.nb_chan / uint32_t(g.S));
}



// One value per lane of each of this thread's vectors, accumulated as sums of
// (x - K) and (x - K)^2 about the thread's first value K.
struct ShiftedSums {
    float k = 0.f, s = 0.f, q = 0.f;
    int n = 0;
    template <int VE>
    __device__ __forceinline__ void add(const float (&v)[VE]) {
        if (n == 0) k = v[0];
#pragma unroll
        for (int i = 0; i < VE; ++i) {
            const float d = v[i] - k;
            s += d;
            q = fmaf(d, d, q);
        }
        n += VE;
    }
    __device__ __forceinline__ Moments moments() const {
        Moments m;
        m.n = float(n);
        m.mean = n ? k + s / float(n) : 0.f;
        m.m2 = n ? fmaxf(q - s * (s / float(n)), 0.f) : 0.f;
        return m;
    }
};

// Bounded wait until a channel's S slices (plus g.peer_extra) have signalled
// `counter`.  Gives up after g.peer_wait_ns and sets `lost`; once `lost` is
// set, later waits of the thread return at once (the peers' partial sums are
// then unusable, and the CTA only finishes its own work).
__device__ __forceinline__ void wait_peers(const BnGeom& g, const uint32_t* counter, bool& lost) {
    const uint32_t count = uint32_t(g.S) + g.peer_extra;
    if (lost || ld_acquire_u32(counter) >= count) return;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire_u32(counter) >= count) return;
        if (global_timer_ns() - t0 > g.peer_wait_ns) {
            lost = true;
            return;
        }
    }
}

// Rounds of one CTA: item = blockIdx.x + r * gridDim.x, channel item / S,
// slice item % S.
struct Rounds {
    const BnGeom& g;
    int64_t items;
    __device__ explicit Rounds(const BnGeom& g_) : g(g_), items(g_.c * g_.S) {}
    __device__ bool valid(int r) const {
        return r < g.rounds && int64_t(blockIdx.x) + int64_t(r) * gridDim.x < items;
    }
    // number of valid rounds of this CTA
    __device__ int count() const {
        if (int64_t(blockIdx.x) >= items) return 0;
        const int64_t n = (items - int64_t(blockIdx.x) + gridDim.x - 1) / gridDim.x;
        return n < g.rounds ? int(n) : g.rounds;
    }
    __device__ void range(int r, int64_t& ch, int& s, uint32_t& b0, uint32_t& b1) const {
        const int64_t it = int64_t(blockIdx.x) + int64_t(r) * gridDim.x;
        ch = it / g.S;
        s = int(it % g.S);
        slice_range(g, s, b0, b1);
    }
};


// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

// Statistics of round r's slice, streamed from HBM (kept in L2 for the apply
// pass) and published to the workspace when the channel has S > 1 slices, or
// kept in `keep` (by round parity) when S == 1.
template <typename T, int VE>
__device__ void fwd_stats(const T* x, const Rounds& rd, int r, Moments* warp_m, Moments* keep, int warp,
                          int lane, uint64_t pol) {
    const BnGeom& g = rd.g;
    int64_t ch;
    int s;
    uint32_t b0, b1;
    rd.range(r, ch, s, b0, b1);
    ShiftedSums acc;
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
                    raw_load_pol<T, VE>(x, p.seg * g.lv + p.v, pk[u], pol);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBnUnroll; ++u) {
            if (!ok[u]) continue;
            float v[VE];
            unpack<T, VE>(pk[u], v);
            acc.add(v);
        }
    }
    Moments m = acc.moments();
    warp_merge(m);
    if (lane == 0) warp_m[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        Moments cta = warp_m[0];
        for (int w = 1; w < kBnWarps; ++w) chan_merge(cta, warp_m[w].n, warp_m[w].mean, warp_m[w].m2);
        if (g.S > 1) {
            float4* part = reinterpret_cast<float4*>(g.partials) + ch * g.S;
            part[s] = make_float4(cta.n, cta.mean, cta.m2, 0.f);
            red_release_add_u32(g.counters + ch, 1u);
        } else {
            keep[r & 1] = cta;
        }
    }
    __syncthreads();  // warp_m is reused
}

template <typename T, int VE, bool TRAIN>
__global__ void __launch_bounds__(kBnThreads, 1)
bn_fwd_kernel(const BnArgs a, const BnGeom g) {
    __shared__ Moments warp_m[kBnWarps];
    __shared__ Moments keep[2];
    __shared__ float s_scale, s_shift;
    __shared__ int s_bad;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);
    const uint64_t pol_stream = l2_evict_first();
    const uint64_t pol_keep = TRAIN ? l2_evict_last() : pol_stream;
    const Rounds rd(g);
    bool bad = false;

    if (threadIdx.x == 0) s_bad = 0;
    if (TRAIN && rd.valid(0)) fwd_stats<T, VE>(x, rd, 0, warp_m, keep, warp, lane, pol_keep);

    for (int r = 0; rd.valid(r); ++r) {
        int64_t ch;
        int s;
        uint32_t b0, b1;
        rd.range(r, ch, s, b0, b1);
        // the next round's statistics go out before this round's wait
        if (TRAIN && rd.valid(r + 1)) fwd_stats<T, VE>(x, rd, r + 1, warp_m, keep, warp, lane, pol_keep);

        const float wc = a.w ? a.w[ch] : 1.f;
        const float bc = a.b ? a.b[ch] : 0.f;
        if constexpr (TRAIN) {
            if (warp == 0) {
                Moments tot = keep[r & 1];
                if (g.S > 1) {
                    const float4* part = reinterpret_cast<const float4*>(g.partials) + ch * g.S;
                    wait_peers(g, g.counters + ch, bad);
                    Moments lm{0.f, 0.f, 0.f};
                    for (int i = lane; i < g.S; i += 32) {
                        const float4 pv = ld_cg_f4(part + i);
                        chan_merge(lm, pv.x, pv.y, pv.z);
                    }
                    warp_merge(lm);
                    tot = lm;
                }
                if (lane == 0) {
                    const float var = tot.m2 * g.inv_m;
                    const float rs = rsqrtf(var + a.eps);
                    s_scale = wc * rs;
                    s_shift = bc - tot.mean * wc * rs;
                    if (s == 0) {
                        if (a.save_mean) a.save_mean[ch] = tot.mean;
                        if (a.save_rstd) a.save_rstd[ch] = rs;
                        if (a.rm) a.rm[ch] = fmaf(a.momentum, tot.mean, (1.f - a.momentum) * a.rm[ch]);
                        if (a.rv) a.rv[ch] = fmaf(a.momentum, tot.m2 * g.inv_m1, (1.f - a.momentum) * a.rv[ch]);
                    }
                }
            }
        } else {
            if (threadIdx.x == 0) {
                const float rs = rsqrtf(a.rv[ch] + a.eps);
                const float mu = a.rm[ch];
                s_scale = wc * rs;
                s_shift = bc - mu * wc * rs;
                if (s == 0) {
                    if (a.save_mean) a.save_mean[ch] = mu;
                    if (a.save_rstd) a.save_rstd[ch] = rs;
                }
            }
        }
        __syncthreads();
        const float scale = s_scale;
        const float shift = s_shift;

        // ---- normalise, affine, residual, activation, store (+ ReLU mask) ----
        for (uint32_t base = b0 + warp; base < b1; base += kBnWarps * kBnUnroll2) {
            Pack<T, VE> px[kBnUnroll2], pr[kBnUnroll2];
#pragma unroll
            for (int u = 0; u < kBnUnroll2; ++u) {
                const uint32_t bi = base + u * kBnWarps;
                if (bi < b1) {
                    const BlockPos p = block_pos(g, bi, lane, ch);
                    if (p.v < g.lv) {
                        raw_load_pol<T, VE>(x, p.seg * g.lv + p.v, px[u], pol_stream);
                        if (res) raw_load_pol<T, VE>(res, p.seg * g.lv + p.v, pr[u], pol_stream);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kBnUnroll2; ++u) {
                const uint32_t bi = base + u * kBnWarps;
                if (bi >= b1) break;  // uniform across the warp
                const BlockPos p = block_pos(g, bi, lane, ch);
                uint32_t nib = 0;
                if (p.v < g.lv) {
                    float v[VE], rr[VE], o[VE];
                    unpack<T, VE>(px[u], v);
                    if (res) unpack<T, VE>(pr[u], rr);
#pragma unroll
                    for (int k = 0; k < VE; ++k) {
                        float z = fmaf(v[k], scale, shift);
                        if (res) z += rr[k];
                        o[k] = act_forward(a.act, z, a.act_param);
                        nib |= uint32_t(z > 0.f) << k;
                    }
                    store_vec_pol<T, VE>(y + (p.seg * g.lv + p.v) * VE, o, pol_stream);
                }
                if (a.mask) store_mask_bits<VE>(a.mask, g, p, lane, nib);
            }
        }
        __syncthreads();  // s_scale / s_shift are rewritten next round
    }

    if (bad) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0 && s_bad) atomicOr(a.err, kErrTimeoutPeers);
}

// ---------------------------------------------------------------------------
// 16-byte vectors: rings of shared-memory slots fed by bulk copies
// ---------------------------------------------------------------------------
// A producer warp streams a CTA's passes in chunks through a ring of 32 KB
// shared-memory slots (the bulk copy engine moves the tensors, the warp's
// lanes move ReLU-mask words with 4-byte async copies); a chunk of a pass over
// nt tensors holds 64/nt blocks of each.  Consumer warps compute from the
// slots and release them.  Every wait is bounded: a wait that runs out sets
// the CTA's abort word, which ends every other wait of the CTA at once; the
// producers then stop issuing copies and wait, bounded, until each copy they
// issued has landed, so none is in flight when the CTA exits.
constexpr int kSlotBlocks = 64;                    // 512-byte blocks per slot
constexpr int kSlotBytes = kSlotBlocks * 512;
constexpr int kSlotMaskWords = 32 * 8;             // mask words of a chunk of >= 2 tensors

__host__ __device__ constexpr uint32_t chunk_span(int nt) { return uint32_t(kSlotBlocks / nt); }

// Calls f(sample n, first block lo, end block hi) for each (sample, channel)
// segment that blocks [b0, b1) of a channel touch.
template <typename F>
__device__ __forceinline__ void for_segments(const BnGeom& g, uint32_t b0, uint32_t b1, F&& f) {
    const uint32_t nbs = uint32_t(g.nbs);
    const uint32_t n_first = fast_div(b0, g.div_nbs);
    const uint32_t n_last = fast_div(b1 - 1, g.div_nbs);
    for (uint32_t n = n_first; n <= n_last; ++n) {
        const uint32_t lo = b0 > n * nbs ? b0 : n * nbs;
        const uint32_t hi = b1 < (n + 1) * nbs ? b1 : (n + 1) * nbs;
        f(n, lo, hi);
    }
}

// One pass over a slice as the producer sees it: up to three tensors (each
// with its L2 policy) and, optionally, the ReLU mask words.
template <typename T>
struct RingPass {
    const T* t[3];
    uint64_t pol[3];
    int nt;
    const uint32_t* mask;
};

template <int SLOTS>
struct Ring {
    unsigned char* data;   // SLOTS x kSlotBytes
    uint32_t* mask;        // SLOTS x kSlotMaskWords, or null
    uint64_t* full;
    uint64_t* empty;
    int seq = 0;
    __device__ int slot() const { return seq % SLOTS; }
    __device__ uint32_t use() const { return uint32_t(seq / SLOTS); }
};

// Waits for phase `parity` of `bar` for at most `limit_ns`; gives up at once
// when another thread of the CTA has given up (*abort != 0), and sets *abort
// when this wait runs out.  Called by every lane of a warp; the result is
// warp-uniform.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, volatile int* abort) {
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const uint64_t t0 = global_timer_ns();
        for (;;) {
            if (mbar_try_wait(bar, parity)) {
                ok = true;
                break;
            }
            if (*abort) break;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Producer (whole warp): one chunk of pass `ps`, blocks [cb, ce) of round r's
// slice, into the next slot of `rg` once its consumers have released it.
// False (nothing issued) when the wait for the slot gave up.
template <typename T, int VE, int SLOTS>
__device__ bool ring_produce_chunk(Ring<SLOTS>& rg, const Rounds& rd, int r, const RingPass<T>& ps, uint32_t cb,
                                   uint32_t ce, int lane, volatile int* abort) {
    const BnGeom& g = rd.g;
    int64_t ch;
    int s;
    uint32_t b0, b1;
    rd.range(r, ch, s, b0, b1);
    const uint32_t span = chunk_span(ps.nt);
    const int slot = rg.slot();
    const uint32_t use = rg.use();
    if (use > 0 && !ring_wait(&rg.empty[slot], (use - 1) & 1u, kBnWaitLimitNs, abort)) return false;
    unsigned char* base = rg.data + size_t(slot) * kSlotBytes;
    if (lane == 0) {
        uint32_t bytes = 0;
        for_segments(g, cb, ce, [&](uint32_t n, uint32_t lo, uint32_t hi) {
            const uint32_t v_lo = (lo - n * g.nbs) * 32;
            const uint32_t v_hi = min((hi - n * g.nbs) * 32, uint32_t(g.lv));
            bytes += (v_hi - v_lo) * 16;
        });
        mbar_arrive_expect_tx(&rg.full[slot], bytes * uint32_t(ps.nt));
        for_segments(g, cb, ce, [&](uint32_t n, uint32_t lo, uint32_t hi) {
            const uint32_t v_lo = (lo - n * g.nbs) * 32;
            const uint32_t v_hi = min((hi - n * g.nbs) * 32, uint32_t(g.lv));
            const int64_t e = ((int64_t(n) * g.c + ch) * g.lv + v_lo) * VE;
            const size_t off = size_t(lo - cb) * 512;
            for (int t = 0; t < ps.nt; ++t)
                bulk_g2s(base + size_t(t) * span * 512 + off, ps.t[t] + e, (v_hi - v_lo) * 16, &rg.full[slot],
                         ps.pol[t]);
        });
    }
    if (ps.mask) {
        uint32_t* mw = rg.mask + size_t(slot) * kSlotMaskWords;
        for_segments(g, cb, ce, [&](uint32_t n, uint32_t lo, uint32_t hi) {
            const uint32_t w_lo = (lo - n * g.nbs) * VE;
            const uint32_t w_hi = min((hi - n * g.nbs) * VE, uint32_t(g.words));
            const uint32_t* src = ps.mask + (int64_t(n) * g.c + ch) * g.words;
            uint32_t* dst = mw + (lo - cb) * VE;
            for (uint32_t w = w_lo + lane; w < w_hi; w += 32) cp_async_4(dst + (w - w_lo), src + w);
        });
        cp_async_mbar_arrive_noinc(&rg.full[slot]);
    }
    ++rg.seq;
    return true;
}

// Producer (whole warp): every chunk of round r's slice for pass `ps`.
template <typename T, int VE, int SLOTS>
__device__ bool ring_produce(Ring<SLOTS>& rg, const Rounds& rd, int r, const RingPass<T>& ps, int lane,
                             volatile int* abort) {
    int64_t ch;
    int s;
    uint32_t b0, b1;
    rd.range(r, ch, s, b0, b1);
    const uint32_t span = chunk_span(ps.nt);
    for (uint32_t cb = b0; cb < b1; cb += span)
        if (!ring_produce_chunk<T, VE>(rg, rd, r, ps, cb, b1 - cb < span ? b1 : cb + span, lane, abort)) return false;
    return true;
}

// Producer, at the end: waits (bounded, whatever *abort says) until the last
// copies issued into every slot have landed.  A slot's copies are issued only
// after its previous phase completed, so its last phase completing covers all
// of them.
template <int SLOTS>
__device__ void ring_drain(Ring<SLOTS>& rg, bool& bad) {
    for (int s = 0; s < SLOTS && s < rg.seq; ++s) {
        const int last = s + ((rg.seq - 1 - s) / SLOTS) * SLOTS;  // last sequence number that used slot s
        if (!mbar_wait_bounded(&rg.full[s], uint32_t(last / SLOTS) & 1u, kBnWaitLimitNs)) bad = true;
    }
}

// Consumer (whole warp): the slot of the next chunk once it has landed, or -1
// when the wait gave up.
template <int SLOTS>
__device__ __forceinline__ int ring_take(Ring<SLOTS>& rg, volatile int* abort) {
    const int slot = rg.slot();
    return ring_wait(&rg.full[slot], rg.use() & 1u, kBnWaitLimitNs, abort) ? slot : -1;
}
template <int SLOTS>
__device__ __forceinline__ void ring_give(Ring<SLOTS>& rg, int slot, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&rg.empty[slot]);
    ++rg.seq;
}

template <int SLOTS>
__device__ __forceinline__ void ring_init(Ring<SLOTS>& rg, uint32_t full_count, uint32_t empty_count) {
    for (int i = 0; i < SLOTS; ++i) {
        mbar_init(&rg.full[i], full_count);
        mbar_init(&rg.empty[i], empty_count);
    }
}

// The VE mask bits of `lane`'s vector of chunk block i, from the slot's words.
template <int VE>
__device__ __forceinline__ uint32_t slot_mask_bits(const uint32_t* mw, uint32_t i, int lane) {
    const int e = lane * VE;
    return (mw[i * VE + (e >> 5)] >> (e & 31)) & ((1u << VE) - 1u);
}

// Warp-uniform %globaltimer.
__device__ __forceinline__ uint64_t warp_now() {
    return __shfl_sync(0xffffffffu, (unsigned long long)global_timer_ns(), 0);
}

// ---------------------------------------------------------------------------
// eval mode on the ring: one pass per round, coefficients from the running
// statistics (no channel depends on another CTA)
// ---------------------------------------------------------------------------
// Roles: 12 consumer warps, a producer warp, and a bookkeeper warp that stages
// each round's channel parameters ahead of the consumers (and, backward,
// publishes the CTA's sums; the last slice of a channel to publish merges
// dw, db).
constexpr int kEvConsumerWarps = 12;
constexpr int kEvThreads = (kEvConsumerWarps + 2) * 32;
constexpr int kEvSlotsFwd = 7;
constexpr int kEvSlotsBwd = 6;

struct EvFwdShared {
    uint64_t coef_ready[2], coef_free[2];   // bookkeeper -> consumers, by round parity
    float2 coef[2];                         // (scale, shift)
    int abort;
};

// y = act(x*scale + shift (+ residual)) with scale, shift from the running
// statistics; saved statistics mean = running_mean, rstd = (running_var +
// eps)^-1/2 from slice 0.
template <typename T, int ACT>
__global__ void __launch_bounds__(kEvThreads, 1)
bn_fwd_eval_kernel(const BnArgs a, const BnGeom g) {
    constexpr int VE = kVec<T>;
    constexpr int SLOTS = kEvSlotsFwd;
    extern __shared__ __align__(128) unsigned char ring_data[];
    __shared__ __align__(8) uint64_t full[SLOTS];
    __shared__ __align__(8) uint64_t empty[SLOTS];
    __shared__ EvFwdShared sh;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);
    const Rounds rd(g);
    const int nr = rd.count();
    Ring<SLOTS> rg{ring_data, nullptr, full, empty};
    volatile int* abort = &sh.abort;
    bool bad = false;

    if (threadIdx.x == 0) {
        ring_init(rg, 1, kEvConsumerWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.coef_ready[i], 1);
            mbar_init(&sh.coef_free[i], kEvConsumerWarps);
        }
        sh.abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kEvConsumerWarps) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first();
        const RingPass<T> apply{{x, res, nullptr}, {pol, pol, 0}, res ? 2 : 1, nullptr};
        for (int r = 0; r < nr; ++r)
            if (!ring_produce<T, VE>(rg, rd, r, apply, lane, abort)) break;
        ring_drain(rg, bad);
    } else if (warp == kEvConsumerWarps + 1) {
        // ---------------- bookkeeper: (scale, shift) of round r ----------------
        for (int r = 0; r < nr; ++r) {
            if (r >= 2 && !ring_wait(&sh.coef_free[r & 1], uint32_t((r >> 1) - 1) & 1u, kBnWaitLimitNs, abort)) break;
            if (lane == 0) {
                int64_t ch;
                int s;
                uint32_t b0, b1;
                rd.range(r, ch, s, b0, b1);
                const float wc = a.w ? a.w[ch] : 1.f;
                const float bc = a.b ? a.b[ch] : 0.f;
                const float rs = rsqrtf(a.rv[ch] + a.eps);
                const float mu = a.rm[ch];
                sh.coef[r & 1] = make_float2(wc * rs, bc - mu * wc * rs);
                mbar_arrive(&sh.coef_ready[r & 1]);
                if (s == 0) {
                    if (a.save_mean) a.save_mean[ch] = mu;
                    if (a.save_rstd) a.save_rstd[ch] = rs;
                }
            }
        }
    } else {
        // ---------------- consumers ----------------
        const uint64_t pol_stream = l2_evict_first();
        const uint32_t span = chunk_span(res ? 2 : 1);
        for (int r = 0; r < nr; ++r) {
            if (!ring_wait(&sh.coef_ready[r & 1], uint32_t(r >> 1) & 1u, kBnWaitLimitNs, abort)) break;
            const float2 sc = sh.coef[r & 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.coef_free[r & 1]);
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(r, ch, s, b0, b1);
            bool ok = true;
            for (uint32_t cb = b0; cb < b1; cb += span) {
                const uint32_t n = b1 - cb < span ? b1 - cb : span;
                const int slot = ring_take(rg, abort);
                if (slot < 0) {
                    ok = false;
                    break;
                }
                const uint4* sx = reinterpret_cast<const uint4*>(ring_data + size_t(slot) * kSlotBytes);
                const uint4* sr = sx + span * 32;
                for (uint32_t i = warp; i < n; i += kEvConsumerWarps) {
                    const BlockPos p = block_pos(g, cb + i, lane, ch);
                    uint32_t nib = 0;
                    if (p.v < g.lv) {
                        Pack<T, VE> px, pr;
                        px.u = sx[i * 32 + lane];
                        float v[VE], rr[VE], o[VE];
                        unpack<T, VE>(px, v);
                        if (res) {
                            pr.u = sr[i * 32 + lane];
                            unpack<T, VE>(pr, rr);
                        }
#pragma unroll
                        for (int k = 0; k < VE; ++k) {
                            float z = fmaf(v[k], sc.x, sc.y);
                            if (res) z += rr[k];
                            nib |= uint32_t(z > 0.f) << k;
                            o[k] = act_forward_c<ACT>(z, a.act_param, a.act);
                        }
                        store_vec_pol<T, VE>(y + (p.seg * g.lv + p.v) * VE, o, pol_stream);
                    }
                    if (a.mask) store_mask_bits<VE>(a.mask, g, p, lane, nib);
                }
                ring_give(rg, slot, lane);
            }
            if (!ok) break;
        }
    }

    __syncthreads();
    if (threadIdx.x == 0 && sh.abort) atomicOr(a.err, kErrTimeoutStage);
    if (bad && lane == 0) atomicOr(a.err, kErrTimeoutStage);
}

// ---------------------------------------------------------------------------
// eval forward, streamed through registers
// ---------------------------------------------------------------------------
// y = act(x*scale[c] + shift[c] (+ residual)) is elementwise once the running
// statistics fix the coefficients, so the eval forward needs no rounds: every
// warp takes kEsUnroll consecutive blocks of 32 vectors (loads first, then the
// arithmetic), and a per-CTA table in dynamic shared memory holds (scale,
// shift) of every channel (8 bytes each: 128 KB at kEsMaxChannels; 64 KB for
// 8192 channels still leaves three CTAs per SM).
constexpr int kEsThreads = 256;
constexpr int kEsWarps = kEsThreads / 32;
constexpr int kEsUnroll = 4;
constexpr int kEsMaxChannels = 16384;

template <typename T, int ACT>
__global__ void __launch_bounds__(kEsThreads)
bn_fwd_eval_stream_kernel(const BnArgs a, const BnGeom g, const FastDiv div_c, const uint32_t nblocks) {
    constexpr int VE = kVec<T>;
    constexpr int U = kEsUnroll;
    extern __shared__ float2 coef[];  // [c]
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    for (int ch = threadIdx.x; ch < int(g.c); ch += kEsThreads) {
        const float wc = a.w ? a.w[ch] : 1.f;
        const float bc = a.b ? a.b[ch] : 0.f;
        const float rs = rsqrtf(a.rv[ch] + a.eps);
        const float mu = a.rm[ch];
        coef[ch] = make_float2(wc * rs, bc - mu * wc * rs);
        if (blockIdx.x == 0) {
            if (a.save_mean) a.save_mean[ch] = mu;
            if (a.save_rstd) a.save_rstd[ch] = rs;
        }
    }
    __syncthreads();
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);
    const uint64_t pol = l2_evict_first();
    const uint32_t step = gridDim.x * kEsWarps * U;
    for (uint32_t b0 = (blockIdx.x * kEsWarps + warp) * U; b0 < nblocks; b0 += step) {
        Pack<T, VE> px[U], pr[U];
        BlockPos p[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t b = b0 + u;
            const uint32_t seg = fast_div(b < nblocks ? b : 0u, g.div_nbs);
            p[u].ni = 0;
            p[u].bs = b - seg * uint32_t(g.nbs);
            p[u].v = int(p[u].bs) * 32 + lane;
            p[u].seg = int64_t(seg);
            if (b < nblocks && p[u].v < g.lv) {
                raw_load_pol<T, VE>(x, p[u].seg * g.lv + p[u].v, px[u], pol);
                if (res) raw_load_pol<T, VE>(res, p[u].seg * g.lv + p[u].v, pr[u], pol);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (b0 + u >= nblocks) break;  // the same for the whole warp
            const uint32_t seg = uint32_t(p[u].seg);
            const uint32_t ch = seg - fast_div(seg, div_c) * uint32_t(g.c);
            const float2 sc = coef[ch];
            uint32_t nib = 0;
            if (p[u].v < g.lv) {
                float v[VE], rr[VE], o[VE];
                unpack<T, VE>(px[u], v);
                if (res) unpack<T, VE>(pr[u], rr);
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    float z = fmaf(v[k], sc.x, sc.y);
                    if (res) z += rr[k];
                    nib |= uint32_t(z > 0.f) << k;
                    o[k] = act_forward_c<ACT>(z, a.act_param, a.act);
                }
                store_vec_pol<T, VE>(y + (p[u].seg * g.lv + p[u].v) * VE, o, pol);
            }
            if (a.mask) store_mask_bits<VE>(a.mask, g, p[u], lane, nib);
        }
    }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------

// dz for one lane's vector at block position p.
template <typename T, int VE>
__device__ __forceinline__ void form_dz(const BnArgs& a, const BnGeom& g, const BlockPos& p, int lane,
                                        bool need_z, float scale, float shift, const float (&dyv)[VE],
                                        const float (&xv)[VE], float (&dz)[VE], uint64_t pol) {
    if (a.act == NRM_ACT_NONE) {
#pragma unroll
        for (int k = 0; k < VE; ++k) dz[k] = dyv[k];
        return;
    }
    if (a.act == NRM_ACT_RELU && !need_z) {
        const uint32_t bits = load_mask_bits<VE>(a.mask_in, g, p, lane, pol);
#pragma unroll
        for (int k = 0; k < VE; ++k) dz[k] = ((bits >> k) & 1u) ? dyv[k] : 0.f;
        return;
    }
    float r[VE];
    if (a.res) {
        Pack<T, VE> pk;
        raw_load_pol<T, VE>(reinterpret_cast<const T*>(a.res), p.seg * g.lv + p.v, pk, pol);
        unpack<T, VE>(pk, r);
    } else {
#pragma unroll
        for (int k = 0; k < VE; ++k) r[k] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < VE; ++k) {
        const float z = fmaf(xv[k], scale, shift) + r[k];
        dz[k] = dyv[k] * act_derivative(a.act, z, a.act_param);
    }
}

// A thread's sums of dz and of dz*(x - mean), centred on the channel's saved
// mean so that the mean does not cancel against the sum of dz (the mean is
// known before the pass: it is part of z).  The thread's share of a slice is
// short, so plain fp32 sums keep about fp32 precision; they are combined
// across threads, CTAs and slices in float-float or double.
struct GradSums {
    float dz = 0.f, dzc = 0.f;
    float mu;
    __device__ __forceinline__ explicit GradSums(float mean) : mu(mean) {}
    template <int VE>
    __device__ __forceinline__ void add(const float (&dzv)[VE], const float (&xv)[VE]) {
#pragma unroll
        for (int k = 0; k < VE; ++k) {
            dz += dzv[k];
            dzc = fmaf(dzv[k], xv[k] - mu, dzc);
        }
    }
    __device__ __forceinline__ double sum_dz() const { return double(dz); }
    __device__ __forceinline__ double sum_dzc() const { return double(dzc); }
    __device__ __forceinline__ FF ff_dz() const { return FF{dz, 0.f}; }
    __device__ __forceinline__ FF ff_dzc() const { return FF{dzc, 0.f}; }
};

// First pass of round r: dz from dy and x (both streamed from HBM and kept in
// L2 for the dx pass in training), dres, the two channel sums (published when
// S > 1, kept when S == 1); in eval mode dx as well.
template <typename T, int VE, bool TRAIN>
__device__ void bwd_pass1(const BnArgs& a, const Rounds& rd, int r, double (*warp_s)[2], double2* keep,
                          int warp, int lane, uint64_t pol_stream, uint64_t pol_keep, bool need_z) {
    const BnGeom& g = rd.g;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ dy = reinterpret_cast<const T*>(a.dy);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    T* __restrict__ dres = reinterpret_cast<T*>(a.dres);
    int64_t ch;
    int s;
    uint32_t b0, b1;
    rd.range(r, ch, s, b0, b1);
    const float mu = a.mean_in[ch];
    const float rs = a.rstd_in[ch];
    const float wc = a.w ? a.w[ch] : 1.f;
    const float bc = a.b ? a.b[ch] : 0.f;
    const float scale = wc * rs;
    const float shift = bc - mu * scale;

    const bool use_mask = a.act == NRM_ACT_RELU && !need_z;
    GradSums acc(mu);
    for (uint32_t base = b0 + warp; base < b1; base += kBnWarps * kBnUnroll2) {
        Pack<T, VE> pdy[kBnUnroll2], px[kBnUnroll2];
        uint32_t mbits[kBnUnroll2];
#pragma unroll
        for (int u = 0; u < kBnUnroll2; ++u) {
            const uint32_t bi = base + u * kBnWarps;
            if (bi < b1) {
                const BlockPos p = block_pos(g, bi, lane, ch);
                if (p.v < g.lv) {
                    raw_load_pol<T, VE>(dy, p.seg * g.lv + p.v, pdy[u], pol_keep);
                    raw_load_pol<T, VE>(x, p.seg * g.lv + p.v, px[u], pol_keep);
                    if (use_mask) mbits[u] = load_mask_bits<VE>(a.mask_in, g, p, lane, pol_keep);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBnUnroll2; ++u) {
            const uint32_t bi = base + u * kBnWarps;
            if (bi >= b1) break;
            const BlockPos p = block_pos(g, bi, lane, ch);
            if (p.v >= g.lv) continue;
            float dyv[VE], xv[VE], dz[VE];
            unpack<T, VE>(pdy[u], dyv);
            unpack<T, VE>(px[u], xv);
            if (use_mask) {
#pragma unroll
                for (int k = 0; k < VE; ++k) dz[k] = ((mbits[u] >> k) & 1u) ? dyv[k] : 0.f;
            } else {
                form_dz<T, VE>(a, g, p, lane, need_z, scale, shift, dyv, xv, dz, pol_keep);
            }
            const int64_t e = (p.seg * g.lv + p.v) * VE;
            if (dres) store_vec_pol<T, VE>(dres + e, dz, pol_stream);
            acc.add(dz, xv);
            if constexpr (!TRAIN) {
                float o[VE];
#pragma unroll
                for (int k = 0; k < VE; ++k) o[k] = dz[k] * scale;
                store_vec_pol<T, VE>(dx + e, o, pol_stream);
            }
        }
    }
    double d1 = acc.sum_dz(), d2 = acc.sum_dzc();
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
        if (g.S > 1) {
            double2* part = reinterpret_cast<double2*>(g.partials) + ch * g.S;
            part[s] = make_double2(t1, t2);
            red_release_add_u32(g.counters + ch, 1u);
        } else {
            keep[r & 1] = make_double2(t1, t2);
        }
    }
    __syncthreads();
}

template <typename T, int VE, bool TRAIN>
__global__ void __launch_bounds__(kBnThreads, 1)
bn_bwd_kernel(const BnArgs a, const BnGeom g) {
    __shared__ double warp_s[kBnWarps][2];
    __shared__ double2 keep[2];
    __shared__ float s_c1, s_c2;
    __shared__ int s_bad;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ dy = reinterpret_cast<const T*>(a.dy);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    // training reads dy, x (and the mask / residual) twice: keep them in L2
    // until the dx pass; everything else streams through once
    const uint64_t pol_stream = l2_evict_first();
    const uint64_t pol_keep = TRAIN ? l2_evict_last() : pol_stream;
    const bool need_z = bn_need_z(a.act, a.mask_in);
    const Rounds rd(g);
    bool bad = false;

    if (threadIdx.x == 0) s_bad = 0;
    if (rd.valid(0)) bwd_pass1<T, VE, TRAIN>(a, rd, 0, warp_s, keep, warp, lane, pol_stream, pol_keep, need_z);

    for (int r = 0; rd.valid(r); ++r) {
        int64_t ch;
        int s;
        uint32_t b0, b1;
        rd.range(r, ch, s, b0, b1);
        if (rd.valid(r + 1))
            bwd_pass1<T, VE, TRAIN>(a, rd, r + 1, warp_s, keep, warp, lane, pol_stream, pol_keep, need_z);
        const float mu = a.mean_in[ch];
        const float rs = a.rstd_in[ch];
        const float wc = a.w ? a.w[ch] : 1.f;
        const float bc = a.b ? a.b[ch] : 0.f;
        const float scale = wc * rs;
        const float shift = bc - mu * scale;

        // ---- this round's channel sums ----
        if (warp == 0) {
            double t1 = keep[r & 1].x, t2 = keep[r & 1].y;
            if (g.S > 1) {
                const double2* part = reinterpret_cast<const double2*>(g.partials) + ch * g.S;
                wait_peers(g, g.counters + ch, bad);
                double l1 = 0.0, l2 = 0.0;
                for (int i = lane; i < g.S; i += 32) {
                    const double2 pv = ld_cg_d2(part + i);
                    l1 += pv.x;
                    l2 += pv.y;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
                    l2 += __shfl_xor_sync(0xffffffffu, l2, o);
                }
                t1 = l1;
                t2 = l2;
            }
            if (lane == 0) {
                const double t2c = t2;  // sum dz*(x - mean): centred on the saved mean as summed
                if (s == 0) {
                    if (a.db) a.db[ch] = float(t1);
                    if (a.dw) a.dw[ch] = float(t2c * double(rs));
                }
                s_c1 = float(t1 * double(g.inv_m));
                s_c2 = float(t2c * double(rs) * double(g.inv_m));
            }
        }
        __syncthreads();

        if constexpr (TRAIN) {
            // ---- dx = w*rstd*(dz - sum(dz)/M - xhat*sum(dz*xhat)/M) ----
            const float c1 = s_c1;
            const float c2 = s_c2;
            const bool use_mask = a.act == NRM_ACT_RELU && !need_z;
            for (uint32_t base = b0 + warp; base < b1; base += kBnWarps * kBnUnrollL2) {
                Pack<T, VE> pdy[kBnUnrollL2], px[kBnUnrollL2];
                uint32_t mbits[kBnUnrollL2];
#pragma unroll
                for (int u = 0; u < kBnUnrollL2; ++u) {
                    const uint32_t bi = base + u * kBnWarps;
                    if (bi < b1) {
                        const BlockPos p = block_pos(g, bi, lane, ch);
                        if (p.v < g.lv) {
                            raw_load_pol<T, VE>(dy, p.seg * g.lv + p.v, pdy[u], pol_stream);
                            raw_load_pol<T, VE>(x, p.seg * g.lv + p.v, px[u], pol_stream);
                            if (use_mask) mbits[u] = load_mask_bits<VE>(a.mask_in, g, p, lane, pol_stream);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kBnUnrollL2; ++u) {
                    const uint32_t bi = base + u * kBnWarps;
                    if (bi >= b1) break;
                    const BlockPos p = block_pos(g, bi, lane, ch);
                    if (p.v >= g.lv) continue;
                    float dyv[VE], xv[VE], dz[VE], o[VE];
                    unpack<T, VE>(pdy[u], dyv);
                    unpack<T, VE>(px[u], xv);
                    if (use_mask) {
#pragma unroll
                        for (int k = 0; k < VE; ++k) dz[k] = ((mbits[u] >> k) & 1u) ? dyv[k] : 0.f;
                    } else {
                        form_dz<T, VE>(a, g, p, lane, need_z, scale, shift, dyv, xv, dz, pol_stream);
                    }
#pragma unroll
                    for (int k = 0; k < VE; ++k) {
                        const float xh = (xv[k] - mu) * rs;
                        o[k] = scale * (dz[k] - c1 - xh * c2);
                    }
                    store_vec_pol<T, VE>(dx + (p.seg * g.lv + p.v) * VE, o, pol_stream);
                }
            }
        }
        __syncthreads();  // s_c1 / s_c2 are rewritten next round
    }

    if (bad) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0 && s_bad) atomicOr(a.err, kErrTimeoutPeers);
}

// ---------------------------------------------------------------------------
// backward on the ring: helpers shared by the eval and training kernels
// ---------------------------------------------------------------------------

// dz of one lane's vector from the slot: dy passed through the activation's
// derivative at z (mask bits, or z recomputed from x and the residual).
template <typename T, int VE, int ACT>
__device__ __forceinline__ void ring_dz(const BnArgs& a, bool use_mask, bool need_z, const uint32_t* mw,
                                        const uint4* sr, uint32_t i, int lane, float scale, float shift,
                                        const float (&dyv)[VE], const float (&xv)[VE], float (&dz)[VE]) {
    if (use_mask) {
        const uint32_t bits = slot_mask_bits<VE>(mw, i, lane);
#pragma unroll
        for (int k = 0; k < VE; ++k) dz[k] = ((bits >> k) & 1u) ? dyv[k] : 0.f;
    } else if (need_z) {
        float r[VE];
        if (a.res) {
            Pack<T, VE> pk;
            pk.u = sr[i * 32 + lane];
            unpack<T, VE>(pk, r);
        } else {
#pragma unroll
            for (int k = 0; k < VE; ++k) r[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < VE; ++k) {
            const float z = fmaf(xv[k], scale, shift) + r[k];
            dz[k] = dyv[k] * act_derivative_c<ACT>(z, a.act_param, a.act);
        }
    } else {
#pragma unroll
        for (int k = 0; k < VE; ++k) dz[k] = dyv[k];
    }
}

// Sum by one warp of the S published (sum dz, sum dz*x) of channel ch, in a
// fixed order.  Every lane must have acquired the complete counter first.
__device__ __forceinline__ void merge_grad_partials(const BnGeom& g, int64_t ch, int lane, double& t1, double& t2) {
    const double2* part = reinterpret_cast<const double2*>(g.partials) + ch * g.S;
    double l1 = 0.0, l2 = 0.0;
    for (int i = lane; i < g.S; i += 32) {
        const double2 pv = ld_cg_d2(part + i);
        l1 += pv.x;
        l2 += pv.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        l2 += __shfl_xor_sync(0xffffffffu, l2, o);
    }
    t1 = l1;
    t2 = l2;
}

// dw, db of channel ch from its two sums, sum dz (t1) and sum dz*(x - mean)
// (t2, centred on the saved mean as it was summed).  Returns sum dz*xhat.
__device__ __forceinline__ double grad_center(const BnArgs& a, int64_t ch, float mu, float rs, double t1, double t2,
                                              bool write_grads) {
    (void)mu;
    const double t2c = t2;
    if (write_grads) {
        if (a.db) a.db[ch] = float(t1);
        if (a.dw) a.dw[ch] = float(t2c * double(rs));
    }
    return t2c * double(rs);
}

struct EvBwdShared {
    uint64_t sums_ready[2], sums_free[2];   // consumers -> bookkeeper, by round parity
    uint64_t par_ready[4], par_free[4];     // a round's channel parameters, by round mod 4
    float4 warp_s[2][kEvConsumerWarps];     // per-warp (sum dz, sum dz*(x - mean)) as float-float pairs
    float4 par[4];                          // (mean, rstd, scale, shift)
    int abort;
};

// Eval backward: dz = dy*act'(z), dres = dz, dx = dz*w*rstd in one pass per
// round; the CTA's two channel sums are published to the workspace and the
// last slice of a channel to publish (acquire-release arrival count) merges
// them in slice order into dw = sum dz*xhat and db = sum dz.
template <typename T, int ACT>
__global__ void __launch_bounds__(kEvThreads, 1)
bn_bwd_eval_kernel(const BnArgs a, const BnGeom g) {
    constexpr int VE = kVec<T>;
    constexpr int SLOTS = kEvSlotsBwd;
    extern __shared__ __align__(128) unsigned char ring_data[];
    __shared__ __align__(8) uint64_t full[SLOTS];
    __shared__ __align__(8) uint64_t empty[SLOTS];
    __shared__ EvBwdShared sh;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ dy = reinterpret_cast<const T*>(a.dy);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    T* __restrict__ dres = reinterpret_cast<T*>(a.dres);
    const bool need_z = bn_need_z(ACT, a.mask_in);
    const bool use_mask = ACT == NRM_ACT_RELU && a.mask_in != nullptr;
    const int nt = (need_z && res) ? 3 : 2;
    const Rounds rd(g);
    const int nr = rd.count();
    Ring<SLOTS> rg{ring_data, reinterpret_cast<uint32_t*>(ring_data + size_t(SLOTS) * kSlotBytes), full, empty};
    volatile int* abort = &sh.abort;
    bool bad = false;

    if (threadIdx.x == 0) {
        ring_init(rg, use_mask ? 33u : 1u, kEvConsumerWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.sums_ready[i], kEvConsumerWarps);
            mbar_init(&sh.sums_free[i], 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&sh.par_ready[i], 1);
            mbar_init(&sh.par_free[i], kEvConsumerWarps);
        }
        sh.abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kEvConsumerWarps) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first();
        const RingPass<T> pass{{dy, x, res}, {pol, pol, pol}, nt, use_mask ? a.mask_in : nullptr};
        for (int q = 0; q < nr; ++q)
            if (!ring_produce<T, VE>(rg, rd, q, pass, lane, abort)) break;
        ring_drain(rg, bad);
    } else if (warp == kEvConsumerWarps + 1) {
        // ---------------- bookkeeper: parameters ahead, sums published, dw/db merged ----------------
        int q_par = 0, q_pub = 0;
        uint64_t t_last = warp_now();
        while ((q_par < nr || q_pub < nr) && !*abort) {
            bool moved = false;
            if (q_par < nr && (q_par < 4 || __all_sync(0xffffffffu, mbar_test_wait(&sh.par_free[q_par & 3],
                                                                                   ((q_par >> 2) - 1) & 1)))) {
                if (lane == 0) {
                    int64_t ch;
                    int s;
                    uint32_t b0, b1;
                    rd.range(q_par, ch, s, b0, b1);
                    const float mu = a.mean_in[ch];
                    const float rs = a.rstd_in[ch];
                    const float wc = a.w ? a.w[ch] : 1.f;
                    const float bc = a.b ? a.b[ch] : 0.f;
                    const float scale = wc * rs;
                    sh.par[q_par & 3] = make_float4(mu, rs, scale, bc - mu * scale);
                    mbar_arrive(&sh.par_ready[q_par & 3]);
                }
                ++q_par;
                moved = true;
            }
            if (q_pub < nr && __all_sync(0xffffffffu, mbar_test_wait(&sh.sums_ready[q_pub & 1], (q_pub >> 1) & 1))) {
                double2 v = make_double2(0.0, 0.0);
                if (lane < kEvConsumerWarps) {
                    const float4 f = sh.warp_s[q_pub & 1][lane];
                    v = make_double2(ff_to_double(FF{f.x, f.y}), ff_to_double(FF{f.z, f.w}));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.sums_free[q_pub & 1]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
                    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
                }
                int64_t ch;
                int s;
                uint32_t b0, b1;
                rd.range(q_pub, ch, s, b0, b1);
                if (g.S == 1) {
                    if (lane == 0) grad_center(a, ch, a.mean_in[ch], a.rstd_in[ch], v.x, v.y, true);
                } else {
                    uint32_t last = 0;
                    if (lane == 0) {
                        double2* part = reinterpret_cast<double2*>(g.partials) + ch * g.S;
                        part[s] = v;
                        last = atom_acq_rel_add_u32(g.counters + ch, 1u) == uint32_t(g.S - 1);
                    }
                    if (__shfl_sync(0xffffffffu, last, 0)) {
                        // every other slice has published: merge into dw, db
                        double t1, t2;
                        merge_grad_partials(g, ch, lane, t1, t2);
                        if (lane == 0) grad_center(a, ch, a.mean_in[ch], a.rstd_in[ch], t1, t2, true);
                    }
                }
                ++q_pub;
                moved = true;
            }
            const uint64_t now = warp_now();
            if (moved) {
                t_last = now;
            } else if (now - t_last > kBnWaitLimitNs) {
                if (lane == 0) *abort = 1;
                break;
            }
        }
    } else {
        // ---------------- consumers ----------------
        const uint64_t pol_stream = l2_evict_first();
        const uint32_t span = chunk_span(nt);
        for (int q = 0; q < nr; ++q) {
            if (!ring_wait(&sh.par_ready[q & 3], uint32_t(q >> 2) & 1u, kBnWaitLimitNs, abort)) break;
            const float4 pr = sh.par[q & 3];
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(q, ch, s, b0, b1);
            GradSums acc(pr.x);
            bool ok = true;
            for (uint32_t cb = b0; cb < b1; cb += span) {
                const uint32_t n = min(span, b1 - cb);
                const int slot = ring_take(rg, abort);
                if (slot < 0) {
                    ok = false;
                    break;
                }
                const uint4* sd = reinterpret_cast<const uint4*>(ring_data + size_t(slot) * kSlotBytes);
                const uint4* sx = sd + span * 32;
                const uint4* sr = sx + span * 32;
                const uint32_t* mw = rg.mask + size_t(slot) * kSlotMaskWords;
                for (uint32_t i = warp; i < n; i += kEvConsumerWarps) {
                    const BlockPos p = block_pos(g, cb + i, lane, ch);
                    if (p.v >= g.lv) continue;
                    Pack<T, VE> pdy, px;
                    pdy.u = sd[i * 32 + lane];
                    px.u = sx[i * 32 + lane];
                    float dyv[VE], xv[VE], dz[VE], o[VE];
                    unpack<T, VE>(pdy, dyv);
                    unpack<T, VE>(px, xv);
                    ring_dz<T, VE, ACT>(a, use_mask, need_z, mw, sr, i, lane, pr.z, pr.w, dyv, xv, dz);
                    const int64_t e = (p.seg * g.lv + p.v) * VE;
                    if (dres) store_vec_pol<T, VE>(dres + e, dz, pol_stream);
                    acc.add(dz, xv);
#pragma unroll
                    for (int k = 0; k < VE; ++k) o[k] = dz[k] * pr.z;
                    store_vec_pol<T, VE>(dx + e, o, pol_stream);
                }
                ring_give(rg, slot, lane);
            }
            if (!ok) break;
            // float-float warp sums: no double-precision arithmetic on the consumers' path
            const FF d1 = ff_warp_sum(acc.ff_dz());
            const FF d2 = ff_warp_sum(acc.ff_dzc());
            if (q >= 2 && !ring_wait(&sh.sums_free[q & 1], uint32_t((q >> 1) - 1) & 1u, kBnWaitLimitNs, abort)) break;
            if (lane == 0) {
                sh.warp_s[q & 1][warp] = make_float4(d1.hi, d1.lo, d2.hi, d2.lo);
                mbar_arrive(&sh.sums_ready[q & 1]);
                mbar_arrive(&sh.par_free[q & 3]);
            }
        }
    }

    __syncthreads();
    if (threadIdx.x == 0 && sh.abort) atomicOr(a.err, kErrTimeoutStage);
    if (bad && lane == 0) atomicOr(a.err, kErrTimeoutStage);
}

}  // namespace nrm

#include "batchnorm_train.cuh"
#include "batchnorm_group.cuh"

namespace nrm {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Upper bound of slices per channel (sizes the workspace).
inline int bn_max_slices(const DevInfo& d) { return 4 * d.sms; }
// Bytes of one (channel, slice) partial in the workspace: float4 (n, mean,
// M2, -) forward, double2 (sum dz, sum dz*(x - mean)) backward.
constexpr size_t kBnPartialBytes = 16;

// Workspace bytes: per-channel counters, then per-(channel, slice) partials.
inline size_t bn_workspace_bytes(const DevInfo& d, int64_t c) {
    const size_t counters = (size_t(c) * 4 + 255) / 256 * 256;
    return counters + size_t(c) * size_t(bn_max_slices(d)) * kBnPartialBytes;
}

struct BnPlan {
    BnGeom g;
    size_t smem;
    int grid;
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
    g.counters = nullptr;
    g.partials = nullptr;
    g.peer_extra = 0;
    g.peer_wait_ns = kBnWaitLimitNs;
}

// L2 held by the kept data of the rounds in flight (the first pass of round
// r+1 overlaps the second pass of round r).  The ring forward keeps one tensor
// and prefers fewer, longer rounds (measured on the ResNet shape), so it gets
// a larger share.
// L2 held between the two passes of the scalar kernels' rounds.
constexpr double kBnL2Budget = 48.0 * 1024 * 1024;
// The training kernels keep up to lag + 1 rounds of first-pass data in L2.
#ifndef NRM_BN_TRAIN_L2_MB_FWD
#define NRM_BN_TRAIN_L2_MB_FWD 128
#endif
#ifndef NRM_BN_TRAIN_L2_MB_BWD
#define NRM_BN_TRAIN_L2_MB_BWD 96
#endif
constexpr double kBnL2BudgetTrainFwd = double(NRM_BN_TRAIN_L2_MB_FWD) * 1024 * 1024;
constexpr double kBnL2BudgetTrainBwd = double(NRM_BN_TRAIN_L2_MB_BWD) * 1024 * 1024;
#ifndef NRM_BN_ROUND_OVERHEAD
#define NRM_BN_ROUND_OVERHEAD 32
#endif
// Fixed cost of a round (channel barrier, reductions), in blocks of work.
constexpr double kBnRoundOverheadBlocks = double(NRM_BN_ROUND_OVERHEAD);

// Chooses k channels per round and S = G/k slices per channel (the grid is a
// whole number of channels, every CTA resident).  `stage_bytes` is the bytes
// per element the passes keep in L2 between the two passes of a round.
inline nrm_status bn_plan(BnPlan& pl, const BnArgs& a, int ve, size_t stage_bytes, const void* fn) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    bn_geometry(pl.g, a, ve);
    BnGeom& g = pl.g;
    const int occ = cached_occupancy(fn, kBnThreads, 0);
    if (occ < 1) return fail(NRM_ERR_CUDA, "batchnorm kernel cannot be resident");
    const int64_t G = int64_t(occ) * d->sms;
    const uint64_t nb = g.nb_chan;
    const double chan_bytes = double(a.n) * double(a.l) * double(stage_bytes);
    int64_t k_max = int64_t(kBnL2Budget / (2.0 * (chan_bytes > 1.0 ? chan_bytes : 1.0)));
    if (k_max < 1) k_max = 1;
    if (k_max > G) k_max = G;
    if (k_max > a.c) k_max = a.c > 0 ? a.c : 1;
    // a channel with few blocks gets few slices (each slice keeps its warps busy)
    int64_t best_k = k_max;
    double best = 1e300;
    for (int64_t k = 1; k <= k_max; ++k) {
        int64_t S = G / k;
        const int64_t s_cap = int64_t(nb / (uint64_t(kBnWarps) * 2)) > 0 ? int64_t(nb / (uint64_t(kBnWarps) * 2)) : 1;
        if (S > s_cap) S = s_cap;
        if (S < 1) S = 1;
        const int64_t kk = G / S;  // channels per round the grid holds at this S
        const int64_t rounds = (a.c + kk - 1) / kk;
        const double cost = double(rounds) * (double((nb + S - 1) / S) + kBnRoundOverheadBlocks);
        if (cost < best) {
            best = cost;
            best_k = k;
        }
    }
    int64_t S = G / best_k;
    {
        const int64_t s_cap = int64_t(nb / (uint64_t(kBnWarps) * 2)) > 0 ? int64_t(nb / (uint64_t(kBnWarps) * 2)) : 1;
        if (S > s_cap) S = s_cap;
        if (S < 1) S = 1;
        if (S > bn_max_slices(*d)) S = bn_max_slices(*d);
    }
    g.S = int(S);
    const int64_t k = G / S;
    const int64_t items = a.c * S;
    int64_t grid = k * S;
    if (grid > items) grid = items;
    pl.grid = int(grid > 0 ? grid : 1);
    g.rounds = int((items + pl.grid - 1) / pl.grid);
    pl.smem = 0;
    return NRM_OK;
}

// Plan of a ring kernel: `smem` bytes of slots, `kept` tensors per element
// held in L2 between the two passes of a round (0 in eval) for `held` rounds
// at a time.  S and k trade rounds (each with a fixed cost) against L2.
inline nrm_status bn_plan_ring(BnPlan& pl, const BnArgs& a, const void* fn, size_t smem, int kept, int held,
                               int threads, double l2_budget) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    BnGeom& g = pl.g;
    pl.smem = smem;
    nrm_status st = prepare_kernel(fn, pl.smem, false);
    if (st != NRM_OK) return st;
    const int occ = cached_occupancy(fn, threads, pl.smem);
    if (occ < 1) return fail(NRM_ERR_CUDA, "batchnorm kernel cannot be resident");
    const int64_t G = int64_t(occ) * d->sms;
    const uint64_t nb = g.nb_chan;
    int64_t k_max = G;
    if (kept > 0) {
        const double chan_bytes = double(nb) * 512.0 * kept;
        k_max = int64_t(l2_budget / (double(held) * chan_bytes));
    }
    if (k_max < 1) k_max = 1;
    if (k_max > G) k_max = G;
    if (k_max > a.c) k_max = a.c;
    // a slice of at least one two-tensor chunk
    const int64_t s_cap = nb / uint64_t(chunk_span(2)) > 0 ? int64_t(nb / uint64_t(chunk_span(2))) : 1;
    int64_t best_S = 1;
    double best = 1e300;
    for (int64_t k = 1; k <= k_max; ++k) {
        int64_t S = G / k;
        if (S > s_cap) S = s_cap;
        if (S > bn_max_slices(*d)) S = bn_max_slices(*d);
        if (S < 1) S = 1;
        const int64_t kk = G / S;
        const int64_t rounds = (a.c + kk - 1) / kk;
        const double cost = double(rounds) * (double((nb + S - 1) / S) + kBnRoundOverheadBlocks);
        if (cost < best) {
            best = cost;
            best_S = S;
        }
    }
    g.S = int(best_S);
    const int64_t k = G / best_S;
    const int64_t items = a.c * best_S;
    int64_t grid = k * best_S;
    if (grid > items) grid = items;
    pl.grid = int(grid > 0 ? grid : 1);
    g.rounds = int((items + pl.grid - 1) / pl.grid);
    // the kernels rely on a CTA keeping the same slice in every round
    if (g.rounds > 1 && pl.grid % g.S != 0) return fail(NRM_ERR_CUDA, "batchnorm plan: grid not a multiple of S");
    return NRM_OK;
}

// `peer_waits`: the kernel waits for a channel's other slices (training with
// S > 1); only such a launch takes the failure-path test hook.
inline nrm_status launch_bn(const void* fn, const BnArgs& a, BnPlan& pl, void* ws, size_t ws_bytes,
                            cudaStream_t s, int threads, bool peer_waits) {
    if (a.c == 0) return NRM_OK;
    const DevInfo* d = dev_info();
    pl.g.peer_extra = 0;
    pl.g.peer_wait_ns = kBnWaitLimitNs;
    uint64_t test_ns = 0;
    if (peer_waits && pl.g.S > 1 && take_peer_wait_test(&test_ns)) {
        pl.g.peer_extra = 1;  // one arrival more than the grid makes: every such wait runs out
        pl.g.peer_wait_ns = test_ns;
    }
    if (pl.g.S > 1) {
        if (!ws || ws_bytes < bn_workspace_bytes(*d, a.c))
            return fail(NRM_ERR_WORKSPACE, "batchnorm needs a workspace of %zu bytes for this shape",
                        bn_workspace_bytes(*d, a.c));
        pl.g.counters = reinterpret_cast<uint32_t*>(ws);
        pl.g.partials = reinterpret_cast<unsigned char*>(ws) + (size_t(a.c) * 4 + 255) / 256 * 256;
        nrm_status st = cuda_status(cudaMemsetAsync(ws, 0, size_t(a.c) * 4, s), "workspace counters reset");
        if (st != NRM_OK) return st;
    }
    BnArgs args = a;
    BnGeom geom = pl.g;
    void* kargs[] = {&args, &geom};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(pl.grid));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelExC(&cfg, fn, kargs), "batchnorm launch");
}

template <typename T>
nrm_status bn_fwd(const BnArgs& a, bool training, bool vec, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (!vec) {
        // short segments: channel groups staged whole in shared memory
        nrm_status st = NRM_OK;
        if (bn_fwd_group<T>(a, training, s, st)) return st;
    }
    if (vec && a.c > 0 && a.n * a.l > 0 && training) {
        const void* fn = with_act(a.act, [&](auto act) {
            return (const void*)&bn_fwd_train_kernel<T, decltype(act)::value>;
        });
        BnPlan pl;
        bn_geometry(pl.g, a, kVec<T>);
        nrm_status st = bn_plan_ring(pl, a, fn, size_t(kTfSlotsS + kTfSlotsA) * kSlotBytes, 1, kTfLag + 1,
                                      kTrThreads, kBnL2BudgetTrainFwd);
        if (st != NRM_OK) return st;
        return launch_bn(fn, a, pl, ws, ws_bytes, s, kTrThreads, true);
    }
    if (vec && a.c > 0 && a.n * a.l > 0 && a.c <= kEsMaxChannels) {
        BnGeom g;
        bn_geometry(g, a, kVec<T>);
        const uint64_t nblocks = uint64_t(a.n) * uint64_t(a.c) * uint64_t(g.nbs);
        if (nblocks < (uint64_t(1) << 31)) {
            const void* fn = with_act(a.act, [&](auto act) {
                return (const void*)&bn_fwd_eval_stream_kernel<T, decltype(act)::value>;
            });
            const DevInfo* d = dev_info();
            const size_t smem = size_t(a.c) * sizeof(float2);
            nrm_status pst = prepare_kernel(fn, smem, false);
            if (pst != NRM_OK) return pst;
            const int occ = cached_occupancy(fn, kEsThreads, smem);
            if (occ < 1) return fail(NRM_ERR_CUDA, "batchnorm eval kernel cannot be resident");
            const uint64_t per_cta = uint64_t(kEsWarps) * kEsUnroll;
            uint64_t grid = (nblocks + per_cta - 1) / per_cta;
            if (grid > uint64_t(occ) * d->sms) grid = uint64_t(occ) * d->sms;
            const FastDivHost fc = make_fast_div(uint32_t(a.c));
            FastDiv div_c;
            div_c.d = fc.d;
            div_c.m = fc.m;
            BnArgs args = a;
            uint32_t nb = uint32_t(nblocks);
            void* kargs[] = {&args, &g, &div_c, &nb};
            return cuda_status(cudaLaunchKernel(fn, dim3(unsigned(grid)), dim3(kEsThreads), kargs, smem, s),
                               "batchnorm eval launch");
        }
    }
    if (vec && a.c > 0 && a.n * a.l > 0) {
        const void* fn = with_act(a.act, [&](auto act) {
            return (const void*)&bn_fwd_eval_kernel<T, decltype(act)::value>;
        });
        BnPlan pl;
        bn_geometry(pl.g, a, kVec<T>);
        nrm_status st = bn_plan_ring(pl, a, fn, size_t(kEvSlotsFwd) * kSlotBytes, 0, 2, kEvThreads, 0.0);
        if (st != NRM_OK) return st;
        return launch_bn(fn, a, pl, ws, ws_bytes, s, kEvThreads, false);
    }
    // unaligned tensors, channel counts the group path cannot tile, empty channels
    const void* fn = training ? (const void*)&bn_fwd_kernel<T, 1, true> : (const void*)&bn_fwd_kernel<T, 1, false>;
    BnPlan pl;
    nrm_status st = bn_plan(pl, a, 1, sizeof(T), fn);
    if (st != NRM_OK) return st;
    return launch_bn(fn, a, pl, ws, ws_bytes, s, kBnThreads, training);
}

template <typename T>
nrm_status bn_bwd(const BnArgs& a, bool training, bool vec, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (!vec) {
        nrm_status st = NRM_OK;
        if (bn_bwd_group<T>(a, training, s, st)) return st;
    }
    if (vec && a.c > 0 && a.n * a.l > 0 && training) {
        const bool need_z = bn_need_z(a.act, a.mask_in);
        const int nt = (need_z && a.res) ? 3 : 2;
        const void* fn = with_act(a.act, [&](auto act) {
            return (const void*)&bn_bwd_train_kernel<T, decltype(act)::value>;
        });
        BnPlan pl;
        bn_geometry(pl.g, a, kVec<T>);
        const size_t smem = size_t(kTbSlots1 + kTbSlots2) * (kSlotBytes + kSlotMaskWords * sizeof(uint32_t));
        nrm_status st = bn_plan_ring(pl, a, fn, smem, nt, kTbLag + 1, kTrThreads, kBnL2BudgetTrainBwd);
        if (st != NRM_OK) return st;
        return launch_bn(fn, a, pl, ws, ws_bytes, s, kTrThreads, true);
    }
    if (vec && a.c > 0 && a.n * a.l > 0) {
        const void* fn = with_act(a.act, [&](auto act) {
            return (const void*)&bn_bwd_eval_kernel<T, decltype(act)::value>;
        });
        BnPlan pl;
        bn_geometry(pl.g, a, kVec<T>);
        const size_t smem = size_t(kEvSlotsBwd) * (kSlotBytes + kSlotMaskWords * sizeof(uint32_t));
        nrm_status st = bn_plan_ring(pl, a, fn, smem, 0, 2, kEvThreads, 0.0);
        if (st != NRM_OK) return st;
        return launch_bn(fn, a, pl, ws, ws_bytes, s, kEvThreads, false);
    }
    const void* fn = training ? (const void*)&bn_bwd_kernel<T, 1, true> : (const void*)&bn_bwd_kernel<T, 1, false>;
    BnPlan pl;
    nrm_status st = bn_plan(pl, a, 1, 2 * sizeof(T), fn);
    if (st != NRM_OK) return st;
    return launch_bn(fn, a, pl, ws, ws_bytes, s, kBnThreads, training);
}

}  // namespace nrm

#define NRM_INSTANTIATE_BATCHNORM(T)                                                                  \
    template nrm_status nrm::bn_fwd<T>(const nrm::BnArgs&, bool, bool, void*, size_t, cudaStream_t); \
    template nrm_status nrm::bn_bwd<T>(const nrm::BnArgs&, bool, bool, void*, size_t, cudaStream_t);
