// batchnorm_group.cuh -- BatchNorm for short spatial extents (l*sizeof(T) not a
// multiple of 16 bytes, e.g. the 7x7 maps of a ResNet's last stage), forward
// and backward, training and eval, with residual and activation.  Included by
// batchnorm.cuh; computes what that file states.
//
// A (sample, channel) segment of l elements is too short, and not aligned, for
// 16-byte access.  G consecutive channels of one sample (G = 16 / gcd(l*size, 16))
// form a span of G*l elements that starts and ends on a 16-byte boundary, so a
// channel group is n such spans at a fixed stride.  A thread-block cluster of
// Q CTAs owns a group: each CTA bulk-copies its n/Q samples' spans into
// shared memory, reduces its per-channel partials and pushes them into every
// cluster CTA's shared memory (distributed shared memory stores, after a
// split cluster barrier that every CTA arrived on at start), one cluster
// barrier later each CTA merges the Q partials in rank order (every CTA gets
// the same bits), and writes its outputs from shared memory with 16-byte
// stores.  Every input byte is read once.
#pragma once

namespace nrm {

constexpr int kGrpThreads = 256;
constexpr int kGrpWarps = kGrpThreads / 32;
constexpr int kGrpMaxQ = 8;  // CTAs per cluster, at most

struct GrpGeom {
    int64_t c;
    int n;
    int l;             // elements per (sample, channel)
    int G;             // channels per group (divides kGrpWarps)
    int span;          // G*l elements: a sample's run of the group
    int Q;             // CTAs per group (the cluster)
    int spc;           // samples per CTA
    int words;         // ReLU-mask words per segment
    uint32_t tile;     // bytes of one tensor's tile in shared memory
    FastDiv div_vps;   // division by the 16-byte vectors of a span
    FastDiv div_l;     // division by l
    float inv_m;       // 1 / (n*l)
    float inv_m1;      // 1 / (n*l - 1)
};

// The CTA's samples [n0, n0 + ns) of its group (whose first channel is ch0).
struct GrpPos {
    uint32_t rank;
    int64_t ch0;
    int n0, ns;
};

__device__ __forceinline__ GrpPos grp_pos(const GrpGeom& g) {
    GrpPos p;
    p.rank = cluster_ctarank();
    p.ch0 = int64_t(blockIdx.x / g.Q) * g.G;
    p.n0 = int(p.rank) * g.spc;
    const int n1 = min(g.n, p.n0 + g.spc);
    p.ns = n1 > p.n0 ? n1 - p.n0 : 0;
    return p;
}

// Warp 0 bulk-copies the CTA's spans of up to three tensors into consecutive
// tiles; completion on `bar` (phase 0).
template <typename T>
__device__ __forceinline__ void grp_load(const GrpGeom& g, const GrpPos& p, unsigned char* smem, uint64_t* bar,
                                         const T* t0, const T* t1, const T* t2) {
    const uint32_t sb = uint32_t(g.span) * sizeof(T);
    const int nt = 1 + (t1 != nullptr) + (t2 != nullptr);
    if ((threadIdx.x >> 5) != 0 || p.ns == 0) return;
    const int lane = threadIdx.x & 31;
    if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(p.ns) * sb * uint32_t(nt));
    __syncwarp();
    const uint64_t pol = l2_evict_first();
    for (int s = lane; s < p.ns; s += 32) {
        const int64_t off = (int64_t(p.n0 + s) * g.c + p.ch0) * g.l;
        bulk_g2s(smem + size_t(s) * sb, t0 + off, sb, bar, pol);
        if (t1) bulk_g2s(smem + g.tile + size_t(s) * sb, t1 + off, sb, bar, pol);
        if (t2) bulk_g2s(smem + 2 * size_t(g.tile) + size_t(s) * sb, t2 + off, sb, bar, pol);
    }
}

template <typename T>
__device__ __forceinline__ float grp_elem(const unsigned char* tile, int idx) {
    return Io<T>::load(reinterpret_cast<const typename Io<T>::bits_t*>(tile)[idx]);
}

// One 16-byte vector of a tile (element offset `e`, a multiple of kVec<T>).
template <typename T>
__device__ __forceinline__ void grp_vec(const unsigned char* tile, int e, float (&v)[kVec<T>]) {
    Pack<T, kVec<T>> pk;
    pk.u = *reinterpret_cast<const uint4*>(tile + size_t(e) * sizeof(T));
    unpack<T, kVec<T>>(pk, v);
}

// Element walk of one channel's part of a CTA's tile: element t of the
// channel's ns*l elements (sample-major) is element e of sample s, and the
// walk advances t by a fixed step with one integer division at the start.
struct GrpWalk {
    int s, e, s_step, e_step;
    __device__ __forceinline__ GrpWalk(int t0, int step, int l) {
        s = t0 / l;
        e = t0 - s * l;
        s_step = step / l;
        e_step = step - s_step * l;
    }
    __device__ __forceinline__ void next(int l) {
        e += e_step;
        s += s_step;
        if (e >= l) {
            e -= l;
            ++s;
        }
    }
};

template <typename T, bool TRAIN, int ACT>
__global__ void __launch_bounds__(kGrpThreads)
bn_fwd_group_kernel(const BnArgs a, const GrpGeom g) {
    constexpr int VE = kVec<T>;
    using bits = typename Io<T>::bits_t;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ Moments wm[kGrpWarps];
    __shared__ float4 allp[kGrpMaxQ][kGrpWarps];  // (n, mean, m2) per channel of every cluster CTA, pushed by it
    __shared__ float2 coef[kGrpWarps];            // (scale, shift) per channel
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);
    const GrpPos p = grp_pos(g);
    const unsigned char* tx = smem;
    const unsigned char* tr = smem + g.tile;

    if constexpr (TRAIN) cluster_arrive_relaxed();  // this CTA has started
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    grp_load<T>(g, p, smem, &bar, x, res, nullptr);
    bool bad = false;
    if (p.ns > 0 && !mbar_wait_bounded(&bar, 0, kBnWaitLimitNs)) bad = true;

    if constexpr (TRAIN) {
        // the warps w with w % G == j share channel j: its ns*l elements
        // (sample-major) are dealt to their lanes, so every lane's chain is
        // short even when l is 1
        const int j = warp % g.G;
        const int wpc = kGrpWarps / g.G;  // warps per channel
        const bits* tb = reinterpret_cast<const bits*>(tx) + j * g.l;
        ShiftedSums acc;
        GrpWalk wk((warp / g.G) * 32 + lane, wpc * 32, g.l);
        for (int t = (warp / g.G) * 32 + lane; t < p.ns * g.l; t += wpc * 32) {
            const float v[1] = {Io<T>::load(tb[wk.s * g.span + wk.e])};
            acc.add(v);
            wk.next(g.l);
        }
        Moments m = acc.moments();
        warp_merge(m);
        if (lane == 0) wm[warp] = m;
        __syncthreads();
        cluster_wait();  // every CTA of the cluster has started: its shared memory may be written
        if (threadIdx.x < g.G) {
            Moments t = wm[threadIdx.x];
            for (int w = threadIdx.x + g.G; w < kGrpWarps; w += g.G) chan_merge(t, wm[w].n, wm[w].mean, wm[w].m2);
            const float4 pv = make_float4(t.n, t.mean, t.m2, 0.f);
            for (int r = 0; r < g.Q; ++r) st_dsmem_f4(dsmem_addr(&allp[p.rank][threadIdx.x], uint32_t(r)), pv);
        }
        cluster_sync_all();  // every CTA's partials have landed in every CTA
        if (threadIdx.x < g.G) {
            Moments tot{0.f, 0.f, 0.f};
            for (int r = 0; r < g.Q; ++r) {
                const float4 pv = allp[r][threadIdx.x];
                chan_merge(tot, pv.x, pv.y, pv.z);
            }
            const int64_t ch = p.ch0 + threadIdx.x;
            const float wc = a.w ? a.w[ch] : 1.f;
            const float bc = a.b ? a.b[ch] : 0.f;
            const float rs = rsqrtf(tot.m2 * g.inv_m + a.eps);
            coef[threadIdx.x] = make_float2(wc * rs, bc - tot.mean * wc * rs);
            if (p.rank == 0) {
                if (a.save_mean) a.save_mean[ch] = tot.mean;
                if (a.save_rstd) a.save_rstd[ch] = rs;
                if (a.rm) a.rm[ch] = fmaf(a.momentum, tot.mean, (1.f - a.momentum) * a.rm[ch]);
                if (a.rv) a.rv[ch] = fmaf(a.momentum, tot.m2 * g.inv_m1, (1.f - a.momentum) * a.rv[ch]);
            }
        }
    } else {
        if (threadIdx.x < g.G) {
            const int64_t ch = p.ch0 + threadIdx.x;
            const float wc = a.w ? a.w[ch] : 1.f;
            const float bc = a.b ? a.b[ch] : 0.f;
            const float rs = rsqrtf(a.rv[ch] + a.eps);
            const float mu = a.rm[ch];
            coef[threadIdx.x] = make_float2(wc * rs, bc - mu * wc * rs);
            if (p.rank == 0) {
                if (a.save_mean) a.save_mean[ch] = mu;
                if (a.save_rstd) a.save_rstd[ch] = rs;
            }
        }
    }
    __syncthreads();

    // ---- y = act(x*scale + shift (+ residual)), 16 bytes per thread and step ----
    const uint64_t pol = l2_evict_first();
    const int vps = g.span / VE;
    for (int v = threadIdx.x; v < p.ns * vps; v += kGrpThreads) {
        const int s = int(fast_div(uint32_t(v), g.div_vps));
        const int o = (v - s * vps) * VE;
        float xv[VE], rv[VE], ov[VE];
        grp_vec<T>(tx, s * g.span + o, xv);
        if (res) grp_vec<T>(tr, s * g.span + o, rv);
        int j = int(fast_div(uint32_t(o), g.div_l));
        int next = (j + 1) * g.l;
        float2 cs = coef[j];  // the vector may cross into the next channel(s): reloaded there
#pragma unroll
        for (int k = 0; k < VE; ++k) {
            if (o + k == next) {
                ++j;
                next += g.l;
                cs = coef[j];
            }
            float z = fmaf(xv[k], cs.x, cs.y);
            if (res) z += rv[k];
            ov[k] = act_forward_c<ACT>(z, a.act_param, a.act);
        }
        store_vec_pol<T, VE>(y + (int64_t(p.n0 + s) * g.c + p.ch0) * g.l + o, ov, pol);
    }
    // ---- ReLU mask: one warp per (sample, channel) segment, a ballot per word ----
    if (a.mask) {
        for (int sg = warp; sg < p.ns * g.G; sg += kGrpWarps) {
            const int s = sg / g.G;
            const int j = sg - s * g.G;
            const float2 cs = coef[j];
            uint32_t* mw = a.mask + (int64_t(p.n0 + s) * g.c + p.ch0 + j) * g.words;
            for (int wi = 0; wi < g.words; ++wi) {
                const int e = wi * 32 + lane;
                bool pos = false;
                if (e < g.l) {
                    float z = fmaf(grp_elem<T>(tx, s * g.span + j * g.l + e), cs.x, cs.y);
                    if (res) z += grp_elem<T>(tr, s * g.span + j * g.l + e);
                    pos = z > 0.f;
                }
                const uint32_t word = __ballot_sync(0xffffffffu, pos);
                if (lane == 0) mw[wi] = word;
            }
        }
    }
    if (bad) {
        // the tile's copy may still be landing: wait once more (bounded) before exit
        mbar_wait_bounded(&bar, 0, kBnWaitLimitNs);
        atomicOr(a.err, kErrTimeoutStage);
    }
}

template <typename T, bool TRAIN, int ACT>
__global__ void __launch_bounds__(kGrpThreads)
bn_bwd_group_kernel(const BnArgs a, const GrpGeom g) {
    constexpr int VE = kVec<T>;
    using bits = typename Io<T>::bits_t;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ double2 ws[kGrpWarps];
    __shared__ double2 allp[kGrpMaxQ][kGrpWarps];  // (sum dz, sum dz*(x - mean)) per channel of every cluster CTA
    __shared__ float4 prm[kGrpWarps];              // (mean, rstd, scale, shift) per channel
    __shared__ float2 coef[kGrpWarps];             // dx coefficients (c1, c2) per channel
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ dy = reinterpret_cast<const T*>(a.dy);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    T* __restrict__ dres = reinterpret_cast<T*>(a.dres);
    const bool need_z = bn_need_z(ACT, a.mask_in);
    const bool use_mask = ACT == NRM_ACT_RELU && a.mask_in != nullptr;
    const bool with_res = need_z && res != nullptr;
    const GrpPos p = grp_pos(g);
    const unsigned char* tdy = smem;
    const unsigned char* tx = smem + g.tile;
    const unsigned char* tr = smem + 2 * size_t(g.tile);
    float* tz = reinterpret_cast<float*>(smem + (with_res ? 3 : 2) * size_t(g.tile));  // dz, fp32
    uint32_t* tm = reinterpret_cast<uint32_t*>(tz + size_t(g.spc) * g.span);            // mask words

    cluster_arrive_relaxed();  // this CTA has started
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    if (threadIdx.x < g.G) {
        const int64_t ch = p.ch0 + threadIdx.x;
        const float mu = a.mean_in[ch];
        const float rs = a.rstd_in[ch];
        const float wc = a.w ? a.w[ch] : 1.f;
        const float bc = a.b ? a.b[ch] : 0.f;
        prm[threadIdx.x] = make_float4(mu, rs, wc * rs, bc - mu * wc * rs);
    }
    __syncthreads();
    grp_load<T>(g, p, smem, &bar, dy, x, with_res ? res : nullptr);
    if (use_mask) {
        // the mask words of the CTA's segments: per sample, G*words consecutive words
        const int per = g.G * g.words;
        for (int i = threadIdx.x; i < p.ns * per; i += kGrpThreads) {
            const int s = i / per;
            tm[i] = a.mask_in[(int64_t(p.n0 + s) * g.c + p.ch0) * g.words + (i - s * per)];
        }
    }
    bool bad = false;
    if (p.ns > 0 && !mbar_wait_bounded(&bar, 0, kBnWaitLimitNs)) bad = true;
    __syncthreads();

    // ---- dz (kept in shared memory) and the two channel sums: warp w takes channel w % G ----
    {
        const int j = warp % g.G;
        const int wpc = kGrpWarps / g.G;
        const float4 pr = prm[j];
        const bits* bdy = reinterpret_cast<const bits*>(tdy) + j * g.l;
        const bits* bx = reinterpret_cast<const bits*>(tx) + j * g.l;
        const bits* br = reinterpret_cast<const bits*>(tr) + j * g.l;
        float* zj = tz + j * g.l;
        const uint32_t* mj = tm + j * g.words;
        GradSums acc(pr.x);
        GrpWalk wk((warp / g.G) * 32 + lane, wpc * 32, g.l);
        for (int t = (warp / g.G) * 32 + lane; t < p.ns * g.l; t += wpc * 32) {
            const int idx = wk.s * g.span + wk.e;
            const float dyv = Io<T>::load(bdy[idx]);
            const float xv[1] = {Io<T>::load(bx[idx])};
            float dz[1];
            if (use_mask) {
                dz[0] = ((mj[wk.s * g.G * g.words + (wk.e >> 5)] >> (wk.e & 31)) & 1u) ? dyv : 0.f;
            } else if (need_z) {
                const float rv = with_res ? Io<T>::load(br[idx]) : 0.f;
                dz[0] = dyv * act_derivative_c<ACT>(fmaf(xv[0], pr.z, pr.w) + rv, a.act_param, a.act);
            } else {
                dz[0] = dyv;
            }
            zj[idx] = dz[0];
            acc.add(dz, xv);
            wk.next(g.l);
        }
        const FF d1 = ff_warp_sum(acc.ff_dz());
        const FF d2 = ff_warp_sum(acc.ff_dzc());
        if (lane == 0) ws[warp] = make_double2(ff_to_double(d1), ff_to_double(d2));
    }
    __syncthreads();
    cluster_wait();  // every CTA of the cluster has started: its shared memory may be written
    if (threadIdx.x < g.G) {
        double2 t = ws[threadIdx.x];
        for (int w = threadIdx.x + g.G; w < kGrpWarps; w += g.G) {
            t.x += ws[w].x;
            t.y += ws[w].y;
        }
        for (int r = 0; r < g.Q; ++r) st_dsmem_d2(dsmem_addr(&allp[p.rank][threadIdx.x], uint32_t(r)), t);
    }
    cluster_sync_all();  // every CTA's partials have landed in every CTA
    if (threadIdx.x < g.G) {
        double t1 = 0.0, t2 = 0.0;
        for (int r = 0; r < g.Q; ++r) {
            const double2 pv = allp[r][threadIdx.x];
            t1 += pv.x;
            t2 += pv.y;
        }
        const int64_t ch = p.ch0 + threadIdx.x;
        const float4 pr = prm[threadIdx.x];
        // t2 is sum dz*(x - mean), centred on the saved mean as it was summed
        if (p.rank == 0) {
            if (a.db) a.db[ch] = float(t1);
            if (a.dw) a.dw[ch] = float(t2 * double(pr.y));
        }
        coef[threadIdx.x] = make_float2(float(t1 * double(g.inv_m)), float(t2 * double(pr.y) * double(g.inv_m)));
    }
    __syncthreads();

    // ---- dres, dx: 16 bytes per thread and step ----
    const uint64_t pol = l2_evict_first();
    const int vps = g.span / VE;
    for (int v = threadIdx.x; v < p.ns * vps; v += kGrpThreads) {
        const int s = int(fast_div(uint32_t(v), g.div_vps));
        const int o = (v - s * vps) * VE;
        float xv[VE], dzv[VE], ov[VE];
        grp_vec<T>(tx, s * g.span + o, xv);
        {
            // dz as the sums pass formed it (two 16-byte reads per 8 values)
            const float4* zp = reinterpret_cast<const float4*>(tz + s * g.span + o);
#pragma unroll
            for (int q = 0; q < VE / 4; ++q) {
                const float4 z4 = zp[q];
                dzv[4 * q] = z4.x;
                dzv[4 * q + 1] = z4.y;
                dzv[4 * q + 2] = z4.z;
                dzv[4 * q + 3] = z4.w;
            }
        }
        int j = int(fast_div(uint32_t(o), g.div_l));
        int next = (j + 1) * g.l;
        float4 pr = prm[j];  // the vector may cross into the next channel(s): reloaded there
        float2 cc = coef[j];
#pragma unroll
        for (int k = 0; k < VE; ++k) {
            if (o + k == next) {
                ++j;
                next += g.l;
                pr = prm[j];
                cc = coef[j];
            }
            if (TRAIN) {
                const float xh = (xv[k] - pr.x) * pr.y;
                ov[k] = pr.z * (dzv[k] - cc.x - xh * cc.y);
            } else {
                ov[k] = dzv[k] * pr.z;
            }
        }
        const int64_t off = (int64_t(p.n0 + s) * g.c + p.ch0) * g.l + o;
        if (dres) store_vec_pol<T, VE>(dres + off, dzv, pol);
        store_vec_pol<T, VE>(dx + off, ov, pol);
    }
    if (bad) {
        // the tile's copy may still be landing: wait once more (bounded) before exit
        mbar_wait_bounded(&bar, 0, kBnWaitLimitNs);
        atomicOr(a.err, kErrTimeoutStage);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

inline int64_t gcd64(int64_t u, int64_t v) {
    while (v) {
        const int64_t t = u % v;
        u = v;
        v = t;
    }
    return u;
}

struct GrpPlan {
    GrpGeom g;
    int grid;
    size_t smem;
};

// Chooses G and the cluster size Q (the smallest that fills the GPU while a
// CTA's tiles fit in shared memory).  False when the shape does not suit
// (then another path runs); `nt` tensors are staged, plus mask words if asked.
inline bool bn_plan_group(GrpPlan& pl, const BnArgs& a, size_t es, int nt, bool dz_buffer, bool mask_words) {
    const DevInfo* d = dev_info();
    if (!d || a.n <= 0 || a.l <= 0 || a.c <= 0) return false;
    const int64_t seg = a.l * int64_t(es);
    const int64_t G = 16 / gcd64(seg, 16);
    if (G > kGrpWarps || a.c % G != 0) return false;
    if (a.n > (int64_t(1) << 30) || a.l > (int64_t(1) << 20)) return false;
    GrpGeom& g = pl.g;
    g.c = a.c;
    g.n = int(a.n);
    g.l = int(a.l);
    g.G = int(G);
    g.span = int(G * a.l);
    g.words = int((a.l + 31) / 32);
    const double m = double(a.n) * double(a.l);
    g.inv_m = float(1.0 / m);
    g.inv_m1 = m > 1 ? float(1.0 / (m - 1.0)) : 0.f;
    const int64_t groups = a.c / G;
    const size_t span_bytes = size_t(g.span) * es;
    const size_t cap = size_t(d->max_smem_optin) - 4096;  // room for the static shared memory
    int chosen = 0;
    for (int Q = 1; Q <= kGrpMaxQ; Q *= 2) {
        if (Q > a.n) break;
        const int64_t spc = (a.n + Q - 1) / Q;
        const size_t tile = (size_t(spc) * span_bytes + 127) / 128 * 128;
        size_t smem = size_t(nt) * tile;
        if (dz_buffer) smem += size_t(spc) * size_t(g.span) * 4;
        if (mask_words) smem += size_t(spc) * size_t(G) * size_t(g.words) * 4;
        if (smem > cap) continue;
        chosen = Q;
        g.spc = int(spc);
        g.tile = uint32_t(tile);
        pl.smem = smem;
        // enough CTAs for two per SM: the elementwise work is instruction-heavy
        if (groups * Q >= 2 * d->sms) break;
    }
    if (chosen == 0) return false;
    if (groups * chosen > (int64_t(1) << 31) - 1) return false;
    g.Q = chosen;
    pl.grid = int(groups * chosen);
    const FastDivHost fv = make_fast_div(uint32_t(g.span / (16 / es)));
    const FastDivHost fl = make_fast_div(uint32_t(g.l));
    g.div_vps.d = fv.d;
    g.div_vps.m = fv.m;
    g.div_l.d = fl.d;
    g.div_l.m = fl.m;
    return true;
}

inline nrm_status launch_group(const void* fn, const BnArgs& a, GrpPlan& pl, cudaStream_t s) {
    nrm_status st = prepare_kernel(fn, pl.smem, false);
    if (st != NRM_OK) return st;
    BnArgs args = a;
    GrpGeom geom = pl.g;
    void* kargs[] = {&args, &geom};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(pl.grid));
    cfg.blockDim = dim3(kGrpThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(pl.g.Q);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelExC(&cfg, fn, kargs), "batchnorm (channel groups) launch");
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename T>
bool bn_fwd_group(const BnArgs& a, bool training, cudaStream_t s, nrm_status& st) {
    if (!aligned16(a.x) || !aligned16(a.res) || !aligned16(a.y)) return false;
    GrpPlan pl;
    if (!bn_plan_group(pl, a, sizeof(T), a.res ? 2 : 1, false, false)) return false;
    const void* fn = with_act(a.act, [&](auto act) {
        return training ? (const void*)&bn_fwd_group_kernel<T, true, decltype(act)::value>
                        : (const void*)&bn_fwd_group_kernel<T, false, decltype(act)::value>;
    });
    st = launch_group(fn, a, pl, s);
    return true;
}

template <typename T>
bool bn_bwd_group(const BnArgs& a, bool training, cudaStream_t s, nrm_status& st) {
    if (!aligned16(a.x) || !aligned16(a.res) || !aligned16(a.dy) || !aligned16(a.dx) || !aligned16(a.dres))
        return false;
    const bool need_z = bn_need_z(a.act, a.mask_in);
    const bool use_mask = a.act == NRM_ACT_RELU && a.mask_in != nullptr;
    GrpPlan pl;
    if (!bn_plan_group(pl, a, sizeof(T), (need_z && a.res) ? 3 : 2, true, use_mask)) return false;
    const void* fn = with_act(a.act, [&](auto act) {
        return training ? (const void*)&bn_bwd_group_kernel<T, true, decltype(act)::value>
                        : (const void*)&bn_bwd_group_kernel<T, false, decltype(act)::value>;
    });
    st = launch_group(fn, a, pl, s);
    return true;
}

}  // namespace nrm
