// batchnorm_train.cuh -- BatchNorm training forward and backward for 16-byte
// aligned tensors: the statistics (or gradient-sum) pass and the apply (or dx)
// pass of a channel run on two teams of warps of the same CTA at the same time.
// Included by batchnorm.cuh.
//
// What is computed follows the attorch normalization article
// ("attorch如何实现LayerNorm、BatchNorm与RMSNorm？3种归一化Triton核代码全解析"),
// section "BatchNorm：按特征并行 + 激活融合": per-channel statistics over batch x
// spatial in one pass over x (the blockwise online update, here per-thread
// shifted sums merged with Chan's formula), the EMA of the running statistics,
// residual and activation fused into the apply step, and a backward that first
// undoes the activation, then forms dx from the two channel sums.
//
// Schedule.  A persistent cooperative grid, one CTA per SM; a channel is cut
// into S slices and a round gives every CTA one slice of one of k channels
// (the Rounds layout of batchnorm.cuh).  A channel's second pass needs the
// channel's first-pass sums from all S CTAs, and between the two passes the
// round's data waits in L2.  Here each CTA runs
//   * team 1 (first pass of round q: statistics / gradient sums, data from
//     HBM with an evict-last policy) and
//   * team 2 (second pass of round q-1 or q-2: y / dx, the round's data
//     re-read from L2)
// concurrently, each fed by its own producer warp and ring of shared-memory
// slots (bulk copies, mbarrier completion), so that HBM keeps streaming the
// next round while the previous one is finished from L2.  Team 1 starts round
// q only after team 2 has finished round q - lag (kTfLag, kTbLag), which bounds
// the L2 held by kept data to about lag + 1 rounds.  A bookkeeper warp merges team 1's
// per-warp sums, publishes the CTA's partial to the workspace, merges a
// channel's S partials in slice order once its counter is complete and hands
// team 2 the channel's coefficients.
//
// Waits.  Every wait is bounded.  A CTA that gives up waiting for its peers
// (the channel counter, limit g.peer_wait_ns) records kErrTimeoutPeers and
// finishes its own work with the partial sums it finds; later peer waits of
// that CTA return at once.  A wait on another warp of the same CTA that runs
// out (2 s) records kErrTimeoutStage and ends every wait of the CTA (the
// shared abort word); the producers then stop issuing copies and wait,
// bounded, until each copy they issued has landed before the CTA exits.
#pragma once

namespace nrm {

constexpr int kTrThreads = 19 * 32;
// Team 1 runs at most this many rounds ahead of team 2 (forward, backward).
#ifndef NRM_BN_TRAIN_LAG_FWD
#define NRM_BN_TRAIN_LAG_FWD 3
#endif
#ifndef NRM_BN_TRAIN_LAG_BWD
#define NRM_BN_TRAIN_LAG_BWD 3
#endif
constexpr int kTfLag = NRM_BN_TRAIN_LAG_FWD;
constexpr int kTbLag = NRM_BN_TRAIN_LAG_BWD;
static_assert(kTfLag >= 1 && kTfLag <= 3 && kTbLag >= 1 && kTbLag <= 3, "the round handoffs are four deep");

// forward roles: warps [0, 4) statistics, [4, 16) apply, then two producers and the bookkeeper
constexpr int kTfStatsWarps = 4;
constexpr int kTfApplyWarps = 12;
constexpr int kTfSlotsS = 3;     // x of the statistics pass (HBM)
constexpr int kTfSlotsA = 4;     // x (L2) and the residual (HBM) of the apply pass
// backward roles: warps [0, 8) pass 1, [8, 16) pass 2, then two producers and the bookkeeper
constexpr int kTbP1Warps = 8;
constexpr int kTbP2Warps = 8;
constexpr int kTbSlots1 = 3;     // dy, x (+ residual), mask words of pass 1 (HBM)
constexpr int kTbSlots2 = 3;     // the same, re-read for pass 2 (L2)
constexpr int kTrProducer1 = 16;
constexpr int kTrProducer2 = 17;
constexpr int kTrBookkeeper = 18;

// Whether channel ch is complete (all S slices published), for a whole warp.
// Once this CTA has given up on its peers (*lost) it no longer waits.
__device__ __forceinline__ bool channel_complete(const BnGeom& g, int64_t ch, bool lost) {
    return __all_sync(0xffffffffu, lost || ld_acquire_u32(g.counters + ch) >= uint32_t(g.S) + g.peer_extra);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

struct TfShared {
    uint64_t sums_ready[2], sums_free[2];   // statistics team -> bookkeeper, by round parity
    uint64_t coef_ready[2], coef_free[2];   // bookkeeper -> apply team, by round parity
    uint64_t apply_done[4];                 // apply team finished round r (r mod 4)
    Moments warp_m[2][kTfStatsWarps];
    float2 coef[2];                         // (scale, shift)
    Moments keep[4];                        // S == 1: a round's statistics
    int abort;
    int peers_lost;
};

// Bookkeeper of the training forward (one warp).
static __device__ void tf_bookkeeper(const BnArgs& a, const BnGeom& g, const Rounds& rd, int nr, TfShared& sh, int lane) {
    volatile int* abort = &sh.abort;
    int q_pub = 0, r_mrg = 0;
    int pre_r = -1;
    float pre_w = 1.f, pre_b = 0.f;
    bool lost = false, peer_wait = false;
    uint64_t t_last = warp_now(), t_peer = 0;
    while ((q_pub < nr || r_mrg < nr) && !*abort) {
        bool moved = false;
        const uint64_t now = warp_now();
        // a statistics pass: merge the team's warps, publish the CTA's partial
        if (q_pub < nr && __all_sync(0xffffffffu, mbar_test_wait(&sh.sums_ready[q_pub & 1], (q_pub >> 1) & 1))) {
            Moments m = lane < kTfStatsWarps ? sh.warp_m[q_pub & 1][lane] : Moments{0.f, 0.f, 0.f};
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.sums_free[q_pub & 1]);
            warp_merge(m);
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(q_pub, ch, s, b0, b1);
            if (lane == 0) {
                if (g.S > 1) {
                    float4* part = reinterpret_cast<float4*>(g.partials) + ch * g.S;
                    part[s] = make_float4(m.n, m.mean, m.m2, 0.f);
                    red_release_add_u32(g.counters + ch, 1u);
                } else {
                    sh.keep[q_pub & 3] = m;
                }
            }
            ++q_pub;
            moved = true;
        }
        // a complete channel: (scale, shift) for the apply team, saved and running statistics
        if (r_mrg < q_pub) {
            const uint32_t u = uint32_t(r_mrg) >> 1;
            bool ok = u == 0 || __all_sync(0xffffffffu, mbar_test_wait(&sh.coef_free[r_mrg & 1], (u - 1) & 1));
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(r_mrg, ch, s, b0, b1);
            if (pre_r != r_mrg) {
                pre_w = a.w ? a.w[ch] : 1.f;
                pre_b = a.b ? a.b[ch] : 0.f;
                pre_r = r_mrg;
            }
            if (ok && g.S > 1 && !channel_complete(g, ch, lost)) {
                ok = false;
                if (!peer_wait) {
                    peer_wait = true;
                    t_peer = now;
                } else if (now - t_peer > g.peer_wait_ns) {
                    lost = true;  // give up on the peers: merge what has arrived
                    ok = true;
                }
            }
            if (ok) {
                peer_wait = false;
                Moments tot = sh.keep[r_mrg & 3];
                if (g.S > 1) {
                    const float4* part = reinterpret_cast<const float4*>(g.partials) + ch * g.S;
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
                    sh.coef[r_mrg & 1] = make_float2(pre_w * rs, pre_b - tot.mean * pre_w * rs);
                    mbar_arrive(&sh.coef_ready[r_mrg & 1]);
                    if (s == 0) {
                        if (a.save_mean) a.save_mean[ch] = tot.mean;
                        if (a.save_rstd) a.save_rstd[ch] = rs;
                        if (a.rm) a.rm[ch] = fmaf(a.momentum, tot.mean, (1.f - a.momentum) * a.rm[ch]);
                        if (a.rv) a.rv[ch] = fmaf(a.momentum, tot.m2 * g.inv_m1, (1.f - a.momentum) * a.rv[ch]);
                    }
                }
                ++r_mrg;
                moved = true;
            } else if (peer_wait) {
                moved = true;  // waiting for other CTAs is bounded by the peer limit, not by this one
            }
        }
        if (moved) {
            t_last = now;
        } else {
            __nanosleep(32);
            if (now - t_last > kBnWaitLimitNs) {
                if (lane == 0) *abort = 1;
                break;
            }
        }
    }
    if (lost && lane == 0) sh.peers_lost = 1;
}

template <typename T, int ACT>
__global__ void __launch_bounds__(kTrThreads, 1)
bn_fwd_train_kernel(const BnArgs a, const BnGeom g) {
    constexpr int VE = kVec<T>;
    extern __shared__ __align__(128) unsigned char ring_data[];
    __shared__ __align__(8) uint64_t full_s[kTfSlotsS], empty_s[kTfSlotsS];
    __shared__ __align__(8) uint64_t full_a[kTfSlotsA], empty_a[kTfSlotsA];
    __shared__ TfShared sh;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);
    const Rounds rd(g);
    const int nr = rd.count();
    Ring<kTfSlotsS> rs{ring_data, nullptr, full_s, empty_s};
    Ring<kTfSlotsA> ra{ring_data + size_t(kTfSlotsS) * kSlotBytes, nullptr, full_a, empty_a};
    volatile int* abort = &sh.abort;
    const uint64_t peer_limit = g.peer_wait_ns + kBnWaitLimitNs;  // waits that include other CTAs' work
    bool bad = false;

    if (threadIdx.x == 0) {
        ring_init(rs, 1, kTfStatsWarps);
        ring_init(ra, 1, kTfApplyWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.sums_ready[i], kTfStatsWarps);
            mbar_init(&sh.sums_free[i], 1);
            mbar_init(&sh.coef_ready[i], 1);
            mbar_init(&sh.coef_free[i], kTfApplyWarps);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&sh.apply_done[i], kTfApplyWarps);
        sh.abort = 0;
        sh.peers_lost = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp < kTfStatsWarps) {
        // ---------------- statistics of round q: x from HBM, kept in L2 ----------------
        const uint32_t span = chunk_span(1);
        for (int q = 0; q < nr; ++q) {
            const int qd = q - kTfLag;
            if (qd >= 0 && !ring_wait(&sh.apply_done[qd & 3], uint32_t(qd >> 2) & 1u, peer_limit, abort)) break;
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(q, ch, s, b0, b1);
            ShiftedSums acc;
            bool ok = true;
            for (uint32_t cb = b0; cb < b1 && ok; cb += span) {
                const uint32_t n = min(span, b1 - cb);
                const int slot = ring_take(rs, abort);
                if (slot < 0) {
                    ok = false;
                    break;
                }
                const uint4* sx = reinterpret_cast<const uint4*>(rs.data + size_t(slot) * kSlotBytes);
                for (uint32_t i = warp; i < n; i += kTfStatsWarps) {
                    const BlockPos p = block_pos(g, cb + i, lane, ch);
                    if (p.v < g.lv) {
                        Pack<T, VE> pk;
                        pk.u = sx[i * 32 + lane];
                        float v[VE];
                        unpack<T, VE>(pk, v);
                        acc.add(v);
                    }
                }
                ring_give(rs, slot, lane);
            }
            if (!ok) break;
            Moments m = acc.moments();
            warp_merge(m);
            if (q >= 2 && !ring_wait(&sh.sums_free[q & 1], uint32_t((q >> 1) - 1) & 1u, kBnWaitLimitNs, abort)) break;
            if (lane == 0) {
                sh.warp_m[q & 1][warp] = m;
                mbar_arrive(&sh.sums_ready[q & 1]);
            }
        }
    } else if (warp < kTfStatsWarps + kTfApplyWarps) {
        // ---------------- apply of round r: y = act(x*scale + shift (+ residual)) ----------------
        const int aw = warp - kTfStatsWarps;
        const uint64_t pol_stream = l2_evict_first();
        const uint32_t span = chunk_span(res ? 2 : 1);
        for (int r = 0; r < nr; ++r) {
            if (!ring_wait(&sh.coef_ready[r & 1], uint32_t(r >> 1) & 1u, peer_limit, abort)) break;
            const float2 sc = sh.coef[r & 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.coef_free[r & 1]);
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(r, ch, s, b0, b1);
            bool ok = true;
            for (uint32_t cb = b0; cb < b1; cb += span) {
                const uint32_t n = min(span, b1 - cb);
                const int slot = ring_take(ra, abort);
                if (slot < 0) {
                    ok = false;
                    break;
                }
                const uint4* sx = reinterpret_cast<const uint4*>(ra.data + size_t(slot) * kSlotBytes);
                const uint4* sr = sx + span * 32;
                for (uint32_t i = aw; i < n; i += kTfApplyWarps) {
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
                ring_give(ra, slot, lane);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.apply_done[r & 3]);
        }
    } else if (warp == kTrProducer1) {
        // ---------------- producer of the statistics pass ----------------
        const RingPass<T> stats{{x, nullptr, nullptr}, {l2_evict_last(), 0, 0}, 1, nullptr};
        for (int q = 0; q < nr; ++q)
            if (!ring_produce<T, VE>(rs, rd, q, stats, lane, abort)) break;
        ring_drain(rs, bad);
    } else if (warp == kTrProducer2) {
        // ---------------- producer of the apply pass: x (L2) and the residual (HBM) ----------------
        const uint64_t pol = l2_evict_first();
        const RingPass<T> apply{{x, res, nullptr}, {pol, pol, 0}, res ? 2 : 1, nullptr};
        for (int r = 0; r < nr; ++r)
            if (!ring_produce<T, VE>(ra, rd, r, apply, lane, abort)) break;
        ring_drain(ra, bad);
    } else {
        tf_bookkeeper(a, g, rd, nr, sh, lane);
    }

    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int e = 0;
        if (sh.abort) e |= kErrTimeoutStage;
        if (sh.peers_lost) e |= kErrTimeoutPeers;
        if (e) atomicOr(a.err, e);
    }
    if (bad && lane == 0) atomicOr(a.err, kErrTimeoutStage);
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------

struct TbShared {
    uint64_t sums_ready[2], sums_free[2];   // pass-1 team -> bookkeeper, by round parity
    uint64_t coef_ready[2], coef_free[2];   // bookkeeper -> pass-2 team, by round parity
    uint64_t par_ready[4], par_free[4];     // a round's channel parameters, by round mod 4
    uint64_t p2_done[4];                    // pass-2 team finished round r (r mod 4)
    float4 warp_s[2][kTbP1Warps];           // per-warp (sum dz, sum dz*(x - mean)) as float-float pairs
    float4 par[4];                          // (mean, rstd, scale, shift)
    float2 coef[2];                         // dx coefficients (c1, c2)
    double2 keep[4];                        // S == 1: a round's sums
    int abort;
    int peers_lost;
};

// Bookkeeper of the training backward (one warp).
static __device__ void tb_bookkeeper(const BnArgs& a, const BnGeom& g, const Rounds& rd, int nr, TbShared& sh, int lane) {
    volatile int* abort = &sh.abort;
    int q_par = 0, q_pub = 0, r_mrg = 0;
    bool lost = false, peer_wait = false;
    uint64_t t_last = warp_now(), t_peer = 0;
    while ((q_par < nr || q_pub < nr || r_mrg < nr) && !*abort) {
        bool moved = false;
        const uint64_t now = warp_now();
        // channel parameters of round q_par
        if (q_par < nr) {
            const uint32_t u = uint32_t(q_par) >> 2;
            if (u == 0 || __all_sync(0xffffffffu, mbar_test_wait(&sh.par_free[q_par & 3], (u - 1) & 1))) {
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
        }
        // pass-1 sums of round q_pub: merge the team's warps, publish the CTA's partial
        if (q_pub < nr && __all_sync(0xffffffffu, mbar_test_wait(&sh.sums_ready[q_pub & 1], (q_pub >> 1) & 1))) {
            double2 v = make_double2(0.0, 0.0);
            if (lane < kTbP1Warps) {
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
            if (lane == 0) {
                if (g.S > 1) {
                    double2* part = reinterpret_cast<double2*>(g.partials) + ch * g.S;
                    part[s] = v;
                    red_release_add_u32(g.counters + ch, 1u);
                } else {
                    sh.keep[q_pub & 3] = v;
                }
            }
            ++q_pub;
            moved = true;
        }
        // the dx coefficients of round r_mrg once its channel is complete; dw, db from slice 0
        if (r_mrg < q_pub) {
            const uint32_t u = uint32_t(r_mrg) >> 1;
            bool ok = u == 0 || __all_sync(0xffffffffu, mbar_test_wait(&sh.coef_free[r_mrg & 1], (u - 1) & 1));
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(r_mrg, ch, s, b0, b1);
            if (ok && g.S > 1 && !channel_complete(g, ch, lost)) {
                ok = false;
                if (!peer_wait) {
                    peer_wait = true;
                    t_peer = now;
                } else if (now - t_peer > g.peer_wait_ns) {
                    lost = true;
                    ok = true;
                }
            }
            if (ok) {
                peer_wait = false;
                double t1, t2;
                if (g.S > 1) {
                    merge_grad_partials(g, ch, lane, t1, t2);
                } else {
                    const double2 k = sh.keep[r_mrg & 3];
                    t1 = k.x;
                    t2 = k.y;
                }
                if (lane == 0) {
                    // the round's parameters stay staged until its pass 2 has finished
                    const float4 pr = sh.par[r_mrg & 3];
                    const double t2r = grad_center(a, ch, pr.x, pr.y, t1, t2, s == 0);
                    sh.coef[r_mrg & 1] = make_float2(float(t1 * double(g.inv_m)), float(t2r * double(g.inv_m)));
                    mbar_arrive(&sh.coef_ready[r_mrg & 1]);
                }
                ++r_mrg;
                moved = true;
            } else if (peer_wait) {
                moved = true;
            }
        }
        if (moved) {
            t_last = now;
        } else {
            __nanosleep(32);
            if (now - t_last > kBnWaitLimitNs) {
                if (lane == 0) *abort = 1;
                break;
            }
        }
    }
    if (lost && lane == 0) sh.peers_lost = 1;
}

template <typename T, int ACT>
__global__ void __launch_bounds__(kTrThreads, 1)
bn_bwd_train_kernel(const BnArgs a, const BnGeom g) {
    constexpr int VE = kVec<T>;
    extern __shared__ __align__(128) unsigned char ring_data[];
    __shared__ __align__(8) uint64_t full1[kTbSlots1], empty1[kTbSlots1];
    __shared__ __align__(8) uint64_t full2[kTbSlots2], empty2[kTbSlots2];
    __shared__ TbShared sh;

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
    // [ring 1: slots | mask words][ring 2: slots | mask words]
    constexpr size_t kRing1Bytes = size_t(kTbSlots1) * (kSlotBytes + kSlotMaskWords * 4);
    Ring<kTbSlots1> r1{ring_data, reinterpret_cast<uint32_t*>(ring_data + size_t(kTbSlots1) * kSlotBytes), full1,
                       empty1};
    Ring<kTbSlots2> r2{ring_data + kRing1Bytes,
                       reinterpret_cast<uint32_t*>(ring_data + kRing1Bytes + size_t(kTbSlots2) * kSlotBytes), full2,
                       empty2};
    volatile int* abort = &sh.abort;
    const uint64_t peer_limit = g.peer_wait_ns + kBnWaitLimitNs;
    bool bad = false;

    if (threadIdx.x == 0) {
        ring_init(r1, use_mask ? 33u : 1u, kTbP1Warps);
        ring_init(r2, use_mask ? 33u : 1u, kTbP2Warps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.sums_ready[i], kTbP1Warps);
            mbar_init(&sh.sums_free[i], 1);
            mbar_init(&sh.coef_ready[i], 1);
            mbar_init(&sh.coef_free[i], kTbP2Warps);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&sh.par_ready[i], 1);
            mbar_init(&sh.par_free[i], kTbP2Warps);
            mbar_init(&sh.p2_done[i], kTbP2Warps);
        }
        sh.abort = 0;
        sh.peers_lost = 0;
        mbar_init_fence();
    }
    __syncthreads();

    const uint32_t span = chunk_span(nt);
    if (warp < kTbP1Warps) {
        // ---------------- pass 1 of round q: dz, dres, the two channel sums ----------------
        const uint64_t pol_stream = l2_evict_first();
        for (int q = 0; q < nr; ++q) {
            const int qd = q - kTbLag;
            if (qd >= 0 && !ring_wait(&sh.p2_done[qd & 3], uint32_t(qd >> 2) & 1u, peer_limit, abort)) break;
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
                const int slot = ring_take(r1, abort);
                if (slot < 0) {
                    ok = false;
                    break;
                }
                const uint4* sd = reinterpret_cast<const uint4*>(r1.data + size_t(slot) * kSlotBytes);
                const uint4* sx = sd + span * 32;
                const uint4* sr = sx + span * 32;
                const uint32_t* mw = r1.mask + size_t(slot) * kSlotMaskWords;
                for (uint32_t i = warp; i < n; i += kTbP1Warps) {
                    const BlockPos p = block_pos(g, cb + i, lane, ch);
                    if (p.v >= g.lv) continue;
                    Pack<T, VE> pdy, px;
                    pdy.u = sd[i * 32 + lane];
                    px.u = sx[i * 32 + lane];
                    float dyv[VE], xv[VE], dz[VE];
                    unpack<T, VE>(pdy, dyv);
                    unpack<T, VE>(px, xv);
                    ring_dz<T, VE, ACT>(a, use_mask, need_z, mw, sr, i, lane, pr.z, pr.w, dyv, xv, dz);
                    if (dres) store_vec_pol<T, VE>(dres + (p.seg * g.lv + p.v) * VE, dz, pol_stream);
                    acc.add(dz, xv);
                }
                ring_give(r1, slot, lane);
            }
            if (!ok) break;
            const FF d1 = ff_warp_sum(acc.ff_dz());
            const FF d2 = ff_warp_sum(acc.ff_dzc());
            if (q >= 2 && !ring_wait(&sh.sums_free[q & 1], uint32_t((q >> 1) - 1) & 1u, kBnWaitLimitNs, abort)) break;
            if (lane == 0) {
                sh.warp_s[q & 1][warp] = make_float4(d1.hi, d1.lo, d2.hi, d2.lo);
                mbar_arrive(&sh.sums_ready[q & 1]);
            }
        }
    } else if (warp < kTbP1Warps + kTbP2Warps) {
        // ---------------- pass 2 of round r: dx = w*rstd*(dz - c1 - xhat*c2) ----------------
        const int pw = warp - kTbP1Warps;
        const uint64_t pol_stream = l2_evict_first();
        for (int r = 0; r < nr; ++r) {
            if (!ring_wait(&sh.par_ready[r & 3], uint32_t(r >> 2) & 1u, peer_limit, abort)) break;
            const float4 pr = sh.par[r & 3];
            const float mu = pr.x, rs = pr.y, scale = pr.z, shift = pr.w;
            if (!ring_wait(&sh.coef_ready[r & 1], uint32_t(r >> 1) & 1u, peer_limit, abort)) break;
            const float2 cc = sh.coef[r & 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.coef_free[r & 1]);
            int64_t ch;
            int s;
            uint32_t b0, b1;
            rd.range(r, ch, s, b0, b1);
            bool ok = true;
            for (uint32_t cb = b0; cb < b1; cb += span) {
                const uint32_t n = min(span, b1 - cb);
                const int slot = ring_take(r2, abort);
                if (slot < 0) {
                    ok = false;
                    break;
                }
                const uint4* sd = reinterpret_cast<const uint4*>(r2.data + size_t(slot) * kSlotBytes);
                const uint4* sx = sd + span * 32;
                const uint4* sr = sx + span * 32;
                const uint32_t* mw = r2.mask + size_t(slot) * kSlotMaskWords;
                for (uint32_t i = pw; i < n; i += kTbP2Warps) {
                    const BlockPos p = block_pos(g, cb + i, lane, ch);
                    if (p.v >= g.lv) continue;
                    Pack<T, VE> pdy, px;
                    pdy.u = sd[i * 32 + lane];
                    px.u = sx[i * 32 + lane];
                    float dyv[VE], xv[VE], dz[VE], o[VE];
                    unpack<T, VE>(pdy, dyv);
                    unpack<T, VE>(px, xv);
                    ring_dz<T, VE, ACT>(a, use_mask, need_z, mw, sr, i, lane, scale, shift, dyv, xv, dz);
#pragma unroll
                    for (int k = 0; k < VE; ++k) {
                        const float xh = (xv[k] - mu) * rs;
                        o[k] = scale * (dz[k] - cc.x - xh * cc.y);
                    }
                    store_vec_pol<T, VE>(dx + (p.seg * g.lv + p.v) * VE, o, pol_stream);
                }
                ring_give(r2, slot, lane);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sh.p2_done[r & 3]);
                mbar_arrive(&sh.par_free[r & 3]);
            }
        }
    } else if (warp == kTrProducer1) {
        // ---------------- producer of pass 1 (HBM, kept in L2) ----------------
        const uint64_t pol = l2_evict_last();
        const RingPass<T> first{{dy, x, res}, {pol, pol, pol}, nt, use_mask ? a.mask_in : nullptr};
        for (int q = 0; q < nr; ++q)
            if (!ring_produce<T, VE>(r1, rd, q, first, lane, abort)) break;
        ring_drain(r1, bad);
    } else if (warp == kTrProducer2) {
        // ---------------- producer of pass 2 (L2 re-reads) ----------------
        const uint64_t pol = l2_evict_first();
        const RingPass<T> second{{dy, x, res}, {pol, pol, pol}, nt, use_mask ? a.mask_in : nullptr};
        for (int r = 0; r < nr; ++r)
            if (!ring_produce<T, VE>(r2, rd, r, second, lane, abort)) break;
        ring_drain(r2, bad);
    } else {
        tb_bookkeeper(a, g, rd, nr, sh, lane);
    }

    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int e = 0;
        if (sh.abort) e |= kErrTimeoutStage;
        if (sh.peers_lost) e |= kErrTimeoutPeers;
        if (e) atomicOr(a.err, e);
    }
    if (bad && lane == 0) atomicOr(a.err, kErrTimeoutStage);
}

}  // namespace nrm
