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
// shared memory.  Each thread owns one 16-byte position of the span across a
// share of the samples, so the channel of every element it touches is fixed:
// it keeps per-element partial sums and per-element coefficients in
// registers, with no per-element index arithmetic.  One warp per channel adds
// the partials in a fixed order; each CTA pushes its per-channel result into
// every cluster CTA's shared memory (distributed shared memory stores, after a
// split cluster barrier that every CTA arrived on at start), one cluster
// barrier later each CTA merges the Q results in rank order (every CTA gets
// the same bits), and writes its outputs with 16-byte stores.  Every input
// byte is read once.
#pragma once

namespace nrm {

constexpr int kGrpMinThreads = 512;   // threads per CTA, at least (one warp per channel of a group needs 256)
constexpr int kGrpMaxThreads = 1024;  // spans of up to 1024 vectors
constexpr int kGrpMaxG = 8;           // channels per group, at most
constexpr int kGrpMaxQ = 8;           // CTAs per cluster, at most

struct GrpGeom {
    int64_t c;
    int n;
    int l;             // elements per (sample, channel)
    int G;             // channels per group
    int span;          // G*l elements: a sample's run of the group
    int vps;           // 16-byte vectors per span
    int P;             // sample phases: P*vps threads take the tile
    int Q;             // CTAs per group (the cluster)
    int spc;           // samples per CTA
    int words;         // ReLU-mask words per segment
    uint32_t tile;     // bytes of one tensor's tile in shared memory
    uint32_t part;     // byte offset of the per-element partial sums (2*P*span floats)
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

// NE elements of T in 8 or 16 bytes.
template <typename T, int NE>
union GrpPack {
    static_assert(NE * sizeof(T) == 16 || NE * sizeof(T) == 8, "8 or 16 bytes");
    typename std::conditional<NE * sizeof(T) == 16, uint4, uint2>::type u;
    typename Io<T>::bits_t b[NE];
};

// NE elements at byte offset `off` of a shared-memory tile, as fp32 pairs.
template <typename T, int NE>
__device__ __forceinline__ void grp_ld(const unsigned char* tile, uint32_t off, float2 (&v)[NE / 2]) {
    GrpPack<T, NE> pk;
    pk.u = *reinterpret_cast<const decltype(pk.u)*>(tile + off);
#pragma unroll
    for (int h = 0; h < NE / 2; ++h) v[h] = make_float2(Io<T>::load(pk.b[2 * h]), Io<T>::load(pk.b[2 * h + 1]));
}

// NE elements rounded to T, stored to global memory with L2 policy `pol`.
template <typename T, int NE>
__device__ __forceinline__ void grp_st(T* p, const float2 (&v)[NE / 2], uint64_t pol) {
    GrpPack<T, NE> pk;
#pragma unroll
    for (int h = 0; h < NE / 2; ++h) {
        pk.b[2 * h] = Io<T>::store(v[h].x);
        pk.b[2 * h + 1] = Io<T>::store(v[h].y);
    }
    if constexpr (NE * sizeof(T) == 16) {
        st_v4_policy(p, pk.u, pol);
    } else {
        st_v2_policy(p, pk.u, pol);
    }
}

// NE fp32 values to / from shared memory (8-byte aligned).
template <int NE>
__device__ __forceinline__ void grp_put_f32(float* d, const float2 (&v)[NE / 2]) {
#pragma unroll
    for (int h = 0; h < NE / 2; ++h) reinterpret_cast<float2*>(d)[h] = v[h];
}
template <int NE>
__device__ __forceinline__ void grp_get_f32(const float* d, float2 (&v)[NE / 2]) {
#pragma unroll
    for (int h = 0; h < NE / 2; ++h) v[h] = reinterpret_cast<const float2*>(d)[h];
}

// The thread's place in the tile.  A span is vps positions of NE elements
// (8 or 16 bytes); thread t < P*vps owns position vp = t % vps of every span
// and takes the CTA's samples ph, ph + P, ... (ph = t / vps), so the channel
// of each of its elements (and with it every per-channel coefficient) is the
// same sample after sample: found once here, with ch[k] the group-relative
// channel of element k and pos[k] its index within that (sample, channel)
// segment.
template <int NE>
struct GrpSlot {
    int vp, ph;
    bool on;
    int ch[NE], pos[NE];
    __device__ __forceinline__ explicit GrpSlot(const GrpGeom& g) {
        vp = int(threadIdx.x) % g.vps;
        ph = int(threadIdx.x) / g.vps;
        on = ph < g.P;
        const int e0 = vp * NE;
        int j = e0 / g.l, r = e0 - j * g.l;
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            ch[k] = j;
            pos[k] = r;
            if (++r == g.l) {
                r = 0;
                ++j;
            }
        }
    }
    // element offset of the thread's position in sample s of a tile
    __device__ __forceinline__ uint32_t at(const GrpGeom& g, int s) const {
        return uint32_t(s) * uint32_t(g.span) + uint32_t(vp * NE);
    }
};

// Element k of this thread's position, summed over its samples, goes to
// part[ph][vp*NE + k]: a [P][span] array of per-(phase, element) partials.
template <int NE>
__device__ __forceinline__ void grp_put_partial(float* part, const GrpGeom& g, const GrpSlot<NE>& sl,
                                                const float2 (&v)[NE / 2]) {
    grp_put_f32<NE>(part + size_t(sl.ph) * g.span + sl.vp * NE, v);
}

template <typename T, bool TRAIN, int ACT>
__global__ void __launch_bounds__(kGrpMaxThreads)
bn_fwd_group_kernel(const BnArgs a, const GrpGeom g) {
    constexpr int NE = kVec<T>;  // 16-byte positions
    constexpr int H = NE / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ float4 allp[kGrpMaxQ][kGrpMaxG];  // (n, mean, m2) per channel of every cluster CTA, pushed by it
    __shared__ float2 coef[kGrpMaxG];            // (scale, shift) per channel
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ res = reinterpret_cast<const T*>(a.res);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);
    const GrpPos p = grp_pos(g);
    const GrpSlot<NE> sl(g);
    const unsigned char* tx = smem;
    const unsigned char* tr = smem + g.tile;

    if constexpr (TRAIN) cluster_arrive_relaxed();  // this CTA has started
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    grp_load<T>(g, p, smem, &bar, x, res, nullptr);
    // the channel's parameters (and running statistics), read while the tile lands
    float wc = 1.f, bc = 0.f, rm = 0.f, rv = 1.f;
    if (threadIdx.x < g.G) {
        const int64_t ch = p.ch0 + threadIdx.x;
        if (a.w) wc = a.w[ch];
        if (a.b) bc = a.b[ch];
        if (!TRAIN || p.rank == 0) {
            if (a.rm) rm = a.rm[ch];
            if (a.rv) rv = a.rv[ch];
        }
    }
    bool bad = false;
    if (p.ns > 0 && !mbar_wait_bounded(&bar, 0, kBnWaitLimitNs)) bad = true;

    if constexpr (TRAIN) {
        // per element of the thread's vectors: sums of (x - K) and (x - K)^2
        // over its samples, K the channel's first value in the tile; with one
        // K per channel these add across the CTA's threads
        float* ps = reinterpret_cast<float*>(smem + g.part);
        float* pq = ps + size_t(g.P) * g.span;
        if (sl.on) {
            float2 nk[H], s2[H], q2[H];
#pragma unroll
            for (int h = 0; h < H; ++h) {
                nk[h] = p.ns > 0 ? make_float2(-grp_elem<T>(tx, sl.ch[2 * h] * g.l),
                                               -grp_elem<T>(tx, sl.ch[2 * h + 1] * g.l))
                                 : make_float2(0.f, 0.f);
                s2[h] = q2[h] = make_float2(0.f, 0.f);
            }
            for (int s = sl.ph; s < p.ns; s += g.P) {
                float2 xv[H];
                grp_ld<T, NE>(tx, sl.at(g, s) * sizeof(T), xv);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 d = __fadd2_rn(xv[h], nk[h]);
                    s2[h] = __fadd2_rn(s2[h], d);
                    q2[h] = __ffma2_rn(d, d, q2[h]);
                }
            }
            grp_put_partial<NE>(ps, g, sl, s2);
            grp_put_partial<NE>(pq, g, sl, q2);
        }
        __syncthreads();
        cluster_wait();  // every CTA of the cluster has started: its shared memory may be written
        if (warp < g.G) {
            // channel `warp`: its l elements of every phase's partials, in a fixed order
            const int j = warp;
            float sum = 0.f, sq = 0.f;
            for (int i = lane; i < g.P * g.l; i += 32) {
                const int q = i / g.l;
                const int idx = q * g.span + j * g.l + (i - q * g.l);
                sum += ps[idx];
                sq += pq[idx];
            }
            sum = warp_sum(sum);
            sq = warp_sum(sq);
            if (lane == 0) {
                float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
                if (p.ns > 0) {
                    const float n = float(p.ns) * float(g.l);
                    const float sn = sum / n;
                    pv = make_float4(n, grp_elem<T>(tx, j * g.l) + sn, fmaxf(sq - sum * sn, 0.f), 0.f);
                }
                for (int r = 0; r < g.Q; ++r) st_dsmem_f4(dsmem_addr(&allp[p.rank][j], uint32_t(r)), pv);
            }
        }
        cluster_sync_all();  // every CTA's partials have landed in every CTA
        if (threadIdx.x < g.G) {
            Moments tot{0.f, 0.f, 0.f};
            for (int r = 0; r < g.Q; ++r) {
                const float4 pv = allp[r][threadIdx.x];
                chan_merge(tot, pv.x, pv.y, pv.z);
            }
            const int64_t ch = p.ch0 + threadIdx.x;
            const float rs = rsqrtf(tot.m2 * g.inv_m + a.eps);
            coef[threadIdx.x] = make_float2(wc * rs, bc - tot.mean * wc * rs);
            if (p.rank == 0) {
                if (a.save_mean) a.save_mean[ch] = tot.mean;
                if (a.save_rstd) a.save_rstd[ch] = rs;
                if (a.rm) a.rm[ch] = fmaf(a.momentum, tot.mean, (1.f - a.momentum) * rm);
                if (a.rv) a.rv[ch] = fmaf(a.momentum, tot.m2 * g.inv_m1, (1.f - a.momentum) * rv);
            }
        }
    } else {
        if (threadIdx.x < g.G) {
            const int64_t ch = p.ch0 + threadIdx.x;
            const float rs = rsqrtf(rv + a.eps);
            const float mu = rm;
            coef[threadIdx.x] = make_float2(wc * rs, bc - mu * wc * rs);
            if (p.rank == 0) {
                if (a.save_mean) a.save_mean[ch] = mu;
                if (a.save_rstd) a.save_rstd[ch] = rs;
            }
        }
    }
    __syncthreads();

    // ---- y = act(x*scale + shift (+ residual)), the thread's vector of each of its samples ----
    const uint64_t pol = l2_evict_first();
    if (sl.on) {
        float2 sc[H], sh[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float2 c0 = coef[sl.ch[2 * h]], c1 = coef[sl.ch[2 * h + 1]];
            sc[h] = make_float2(c0.x, c1.x);
            sh[h] = make_float2(c0.y, c1.y);
        }
        for (int s = sl.ph; s < p.ns; s += g.P) {
            float2 xv[H], rv[H];
            grp_ld<T, NE>(tx, sl.at(g, s) * sizeof(T), xv);
            if (res) grp_ld<T, NE>(tr, sl.at(g, s) * sizeof(T), rv);
            float2 ov[H];
#pragma unroll
            for (int h = 0; h < H; ++h) {
                float2 z = __ffma2_rn(xv[h], sc[h], sh[h]);
                if (res) z = __fadd2_rn(z, rv[h]);
                ov[h] = act_forward2_c<ACT>(z, a.act_param, a.act);
            }
            grp_st<T, NE>(y + (int64_t(p.n0 + s) * g.c + p.ch0) * g.l + sl.vp * NE, ov, pol);
        }
    }
    // ---- ReLU mask: one warp per (sample, channel) segment, a ballot per word ----
    if (a.mask) {
        for (int sg = warp; sg < p.ns * g.G; sg += nwarps) {
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
__global__ void __launch_bounds__(kGrpMaxThreads)
bn_bwd_group_kernel(const BnArgs a, const GrpGeom g) {
    constexpr int NE = kVec<T> / 2;  // 8-byte positions: half the per-element registers
    constexpr int H = NE / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ double2 allp[kGrpMaxQ][kGrpMaxG];  // (sum dz, sum dz*(x - mean)) per channel of every cluster CTA
    __shared__ float4 prm[kGrpMaxG];              // (mean, rstd, scale, shift) per channel
    __shared__ float4 dxc[kGrpMaxG];              // dx = A*dz - B - C*(x - mean): (A, B, C, mean) per channel
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
    const GrpSlot<NE> sl(g);
    const unsigned char* tdy = smem;
    const unsigned char* tx = smem + g.tile;
    const unsigned char* tr = smem + 2 * size_t(g.tile);
    float* tz = reinterpret_cast<float*>(smem + (with_res ? 3 : 2) * size_t(g.tile));  // dz, fp32
    uint32_t* tm = reinterpret_cast<uint32_t*>(tz + size_t(g.spc) * g.span);            // mask words
    // the partial sums (2*P*span floats), over the dy tile when it is large enough
    float* pd = reinterpret_cast<float*>(smem + g.part);
    float* pc = pd + size_t(g.P) * g.span;

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
        for (int i = threadIdx.x; i < p.ns * per; i += blockDim.x) {
            const int s = i / per;
            tm[i] = a.mask_in[(int64_t(p.n0 + s) * g.c + p.ch0) * g.words + (i - s * per)];
        }
    }
    bool bad = false;
    if (p.ns > 0 && !mbar_wait_bounded(&bar, 0, kBnWaitLimitNs)) bad = true;
    __syncthreads();

    // ---- dz (kept in shared memory) and, per element of the thread's vectors, sums of dz and dz*(x - mean) ----
    float2 sdz[H], sdc[H];
#pragma unroll
    for (int h = 0; h < H; ++h) sdz[h] = sdc[h] = make_float2(0.f, 0.f);
    if (sl.on) {
        float2 nmu[H], sc[H], sh[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float4 p0 = prm[sl.ch[2 * h]], p1 = prm[sl.ch[2 * h + 1]];
            nmu[h] = make_float2(-p0.x, -p1.x);
            sc[h] = make_float2(p0.z, p1.z);
            sh[h] = make_float2(p0.w, p1.w);
        }
        const int wps = g.G * g.words;  // mask words per sample
        for (int s = sl.ph; s < p.ns; s += g.P) {
            float2 dyv[H], xv[H], dz[H];
            grp_ld<T, NE>(tdy, sl.at(g, s) * sizeof(T), dyv);
            grp_ld<T, NE>(tx, sl.at(g, s) * sizeof(T), xv);
            if (use_mask) {
                const uint32_t* mw = tm + s * wps;
                float m[NE];
#pragma unroll
                for (int k = 0; k < NE; ++k)
                    m[k] = ((mw[sl.ch[k] * g.words + (sl.pos[k] >> 5)] >> (sl.pos[k] & 31)) & 1u) ? 1.f : 0.f;
#pragma unroll
                for (int h = 0; h < H; ++h) dz[h] = __fmul2_rn(dyv[h], make_float2(m[2 * h], m[2 * h + 1]));
            } else if (need_z) {
                float2 rv[H];
                if (with_res) {
                    grp_ld<T, NE>(tr, sl.at(g, s) * sizeof(T), rv);
                } else {
#pragma unroll
                    for (int h = 0; h < H; ++h) rv[h] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 z = __fadd2_rn(__ffma2_rn(xv[h], sc[h], sh[h]), rv[h]);
                    dz[h] = __fmul2_rn(dyv[h], act_derivative2_c<ACT>(z, a.act_param, a.act));
                }
            } else {
#pragma unroll
                for (int h = 0; h < H; ++h) dz[h] = dyv[h];
            }
            grp_put_f32<NE>(tz + sl.at(g, s), dz);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                sdz[h] = __fadd2_rn(sdz[h], dz[h]);
                sdc[h] = __ffma2_rn(dz[h], __fadd2_rn(xv[h], nmu[h]), sdc[h]);
            }
        }
    }
    __syncthreads();  // the dy tile is read: the partials may go over it
    if (sl.on) {
        grp_put_partial<NE>(pd, g, sl, sdz);
        grp_put_partial<NE>(pc, g, sl, sdc);
    }
    __syncthreads();
    cluster_wait();  // every CTA of the cluster has started: its shared memory may be written
    if (warp < g.G) {
        // channel `warp`: its l elements of every phase's partials, in a fixed order, in float-float
        const int j = warp;
        FF d1{0.f, 0.f}, d2{0.f, 0.f};
        for (int i = lane; i < g.P * g.l; i += 32) {
            const int q = i / g.l;
            const int idx = q * g.span + j * g.l + (i - q * g.l);
            d1 = ff_add(d1, FF{pd[idx], 0.f});
            d2 = ff_add(d2, FF{pc[idx], 0.f});
        }
        d1 = ff_warp_sum(d1);
        d2 = ff_warp_sum(d2);
        if (lane == 0) {
            const double2 t = make_double2(ff_to_double(d1), ff_to_double(d2));
            for (int r = 0; r < g.Q; ++r) st_dsmem_d2(dsmem_addr(&allp[p.rank][j], uint32_t(r)), t);
        }
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
        // dx = scale*(dz - c1 - xhat*c2) with c1 = mean(dz), c2 = mean(dz*xhat)
        const double c1 = t1 * double(g.inv_m);
        const double c2 = t2 * double(pr.y) * double(g.inv_m);
        dxc[threadIdx.x] = TRAIN ? make_float4(pr.z, float(double(pr.z) * c1), float(double(pr.z) * c2 * double(pr.y)), pr.x)
                                 : make_float4(pr.z, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    // ---- dres, dx: the thread's vector of each of its samples ----
    const uint64_t pol = l2_evict_first();
    if (sl.on) {
        float2 ca[H], cb[H], cc[H], nmu[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float4 q0 = dxc[sl.ch[2 * h]], q1 = dxc[sl.ch[2 * h + 1]];
            ca[h] = make_float2(q0.x, q1.x);
            cb[h] = make_float2(-q0.y, -q1.y);
            cc[h] = make_float2(-q0.z, -q1.z);
            nmu[h] = make_float2(-q0.w, -q1.w);
        }
        for (int s = sl.ph; s < p.ns; s += g.P) {
            float2 dzv[H], ov[H];
            grp_get_f32<NE>(tz + sl.at(g, s), dzv);
            if (TRAIN) {
                float2 xv[H];
                grp_ld<T, NE>(tx, sl.at(g, s) * sizeof(T), xv);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    ov[h] = __ffma2_rn(cc[h], __fadd2_rn(xv[h], nmu[h]), __ffma2_rn(ca[h], dzv[h], cb[h]));
            } else {
#pragma unroll
                for (int h = 0; h < H; ++h) ov[h] = __fmul2_rn(dzv[h], ca[h]);
            }
            const int64_t off = (int64_t(p.n0 + s) * g.c + p.ch0) * g.l + sl.vp * NE;
            if (dres) grp_st<T, NE>(dres + off, dzv, pol);
            grp_st<T, NE>(dx + off, ov, pol);
        }
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
    int threads;
    size_t smem;
};

// Chooses G, the block size, the cluster size Q (the smallest that fills the
// GPU while a CTA's tiles fit in shared memory) and the sample phases P for
// threads that own `pos_bytes` (8 or 16) of a span each.  False when the
// shape does not suit (then another path runs).  `nt` tensors are staged,
// plus the backward's fp32 dz buffer and mask words if asked; `sums` reserves
// the per-element partial sums (over the first tile when it is large enough
// and `over_first_tile`).
inline bool bn_plan_group(GrpPlan& pl, const BnArgs& a, size_t es, int pos_bytes, int nt, bool dz_buffer,
                          bool mask_words, bool sums, bool over_first_tile) {
    const DevInfo* d = dev_info();
    if (!d || a.n <= 0 || a.l <= 0 || a.c <= 0) return false;
    const int64_t seg = a.l * int64_t(es);
    const int64_t G = 16 / gcd64(seg, 16);
    if (G > kGrpMaxG || a.c % G != 0) return false;
    if (a.n > (int64_t(1) << 30) || a.l > (int64_t(1) << 20)) return false;
    GrpGeom& g = pl.g;
    g.c = a.c;
    g.n = int(a.n);
    g.l = int(a.l);
    g.G = int(G);
    g.span = int(G * a.l);
    g.vps = int(int64_t(g.span) * int64_t(es) / pos_bytes);
    if (g.vps > kGrpMaxThreads) return false;
    pl.threads = g.vps <= kGrpMinThreads ? kGrpMinThreads : (g.vps + 31) / 32 * 32;
    g.words = int((a.l + 31) / 32);
    const double m = double(a.n) * double(a.l);
    g.inv_m = float(1.0 / m);
    g.inv_m1 = m > 1 ? float(1.0 / (m - 1.0)) : 0.f;
    const int64_t groups = a.c / G;
    const size_t span_bytes = size_t(g.span) * es;
    const size_t cap = size_t(d->max_smem_optin) - 4096;  // room for the static shared memory
    const int pmax = pl.threads / g.vps;
    int chosen = 0;
    for (int Q = 1; Q <= kGrpMaxQ; Q *= 2) {
        if (Q > a.n) break;
        const int64_t spc = (a.n + Q - 1) / Q;
        const size_t tile = (size_t(spc) * span_bytes + 127) / 128 * 128;
        // samples per thread, then as few phases as give each thread that many
        const int64_t per = (spc + pmax - 1) / pmax;
        const int P = int((spc + per - 1) / per);
        size_t smem = size_t(nt) * tile;
        if (dz_buffer) smem += size_t(spc) * size_t(g.span) * 4;
        if (mask_words) smem += size_t(spc) * size_t(G) * size_t(g.words) * 4;
        smem = (smem + 15) / 16 * 16;
        const size_t part_bytes = sums ? 2 * size_t(P) * size_t(g.span) * 4 : 0;
        uint32_t part = 0;
        if (!(over_first_tile && part_bytes <= tile)) {
            part = uint32_t(smem);
            smem += part_bytes;
        }
        if (smem > cap) continue;
        chosen = Q;
        g.spc = int(spc);
        g.P = P;
        g.tile = uint32_t(tile);
        g.part = part;
        pl.smem = smem;
        // enough CTAs for 1.5 per SM (512-thread CTAs, two fit an SM): measured on the fp16
        // [128,512,7,7] workload against 256-thread CTAs at two to four per SM
        if (2 * groups * Q >= 3 * d->sms) break;
    }
    if (chosen == 0) return false;
    if (groups * chosen > (int64_t(1) << 31) - 1) return false;
    g.Q = chosen;
    pl.grid = int(groups * chosen);
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
    cfg.blockDim = dim3(unsigned(pl.threads));
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
    if (!bn_plan_group(pl, a, sizeof(T), 16, a.res ? 2 : 1, false, false, training, false)) return false;
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
    if (!bn_plan_group(pl, a, sizeof(T), 8, (need_z && a.res) ? 3 : 2, true, use_mask, true, true))
        return false;
    const void* fn = with_act(a.act, [&](auto act) {
        return training ? (const void*)&bn_bwd_group_kernel<T, true, decltype(act)::value>
                        : (const void*)&bn_bwd_group_kernel<T, false, decltype(act)::value>;
    });
    st = launch_group(fn, a, pl, s);
    return true;
}

}  // namespace nrm
