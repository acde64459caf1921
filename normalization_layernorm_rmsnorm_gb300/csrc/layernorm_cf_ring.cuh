// layernorm_cf_ring.cuh -- channels-first LayerNorm (x[n, c, l], normalised
// over c for every sample and position; what layernorm_cf.cuh states) with the
// tiles streamed through shared memory by TMA, for planes whose byte length
// l*sizeof(T) is a multiple of 16 (included by rownorm.cuh).
//
// A tile is [c][P] of one sample: P = PV*V consecutive positions (V values of
// 16 bytes per thread) in every channel plane.  The tensor is a 3-D tensor map
// {l, c, n}; one box {P, CB, 1} per CB channels brings the tile in with one
// instruction, zero-filling positions past l and channels past c.  A producer
// warp keeps `slots` tiles in flight.  The 16 consumer warps form two teams
// of 8 that take the CTA's tiles in turn (team 0 the even ones), so that one
// team's barriers and merge overlap the other team's passes.  In a team,
// thread t takes position vector pv = t % PV and channel group g = t / PV,
// which covers channels g, g + CG, ... (CG = 256 / PV).  Pass 1 reduces the
// group's channels from the slot; the groups are merged per position in
// shared memory in a fixed order (partials stored position-vector-minor, so
// that a warp's accesses fall in distinct banks); pass 2 re-reads the slot and
// writes the outputs with 16-byte stores.  One persistent CTA per SM takes
// tiles b, b + grid, ...
#pragma once

namespace nrm {

constexpr int kCfrTeams = 2;
constexpr int kCfrTeamWarps = 8;
constexpr int kCfrTeamThreads = kCfrTeamWarps * 32;
constexpr int kCfrConsumerWarps = kCfrTeams * kCfrTeamWarps;
constexpr int kCfrConsumers = kCfrConsumerWarps * 32;
constexpr int kCfrThreads = kCfrConsumers + 32;  // + the producer warp
constexpr int kCfrMaxSlots = 8;                   // the slot count is even (see cfr_plan)
constexpr int kCfrBarTeam = 1;                    // named barriers 1, 2: one per team
constexpr int kCfrBarAll = 3;                     // named barrier over all consumer warps
// floats of a team's shared scratch per tile position: per-warp partials
// [8][2][P] and the merged per-position values [2 parities][2][P]
constexpr int kCfrTeamFloatsPerPos = kCfrTeamWarps * 2 + 4;

struct CfrGeom {
    int pv;                // 16-byte position vectors per tile row (8, 16 or 32)
    int P;                 // positions per tile: pv * 16 / sizeof(T)
    int cb;                // channels per TMA box (<= 256)
    int nb;                // boxes per tensor and tile: nb * cb >= c
    int slots;
    uint32_t slot_bytes;   // nb*cb rows of P values per tensor (+ 2*P floats of statistics, backward)
    uint32_t tx_tensor;    // bytes one tensor's boxes deliver per tile
    uint32_t param_bytes;  // fp32 weight (and bias) at the front of dynamic shared memory
    uint32_t part_bytes;   // both teams' scratch (kCfrTeamFloatsPerPos*P floats each) + merge factors [8][2]
    uint32_t acc_bytes;    // backward: each team's dw, db partial row [2][2][c]
    int64_t tps;           // tiles per sample
    int64_t tiles;
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
           "r"(smem_addr(bar)), "l"(pol) : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 16 bytes of shared memory as fp32 pairs.
template <typename T>
__device__ __forceinline__ void cfr_load2(const unsigned char* p, float2 (&v)[kPairs<T>]) {
    unpack2<T>(*reinterpret_cast<const uint4*>(p), v);
}

// fp32 pairs rounded to T and stored as one 16-byte global store.
template <typename T>
__device__ __forceinline__ void cfr_store2(T* p, const float2 (&o)[kPairs<T>]) {
    st_v4(p, pack2x<T>(o));
}

// Producer (whole warp, lane 0 issues): the CTA's tiles into the ring, in
// order.  `map_a` is x (forward) or dy (backward); `map_b` is x (backward).
template <typename T, bool BWD>
__device__ void cfr_produce(const CfArgs& a, const CfrGeom& g, unsigned char* ring, uint64_t* full,
                            uint64_t* empty, const CUtensorMap* map_a, const CUtensorMap* map_b, int lane,
                            bool& bad) {
    const uint64_t pol = l2_evict_first();
    const size_t tensor_bytes = size_t(g.nb) * g.cb * g.P * sizeof(T);
    int q = 0;
    for (int64_t t = blockIdx.x; t < g.tiles; t += gridDim.x, ++q) {
        const int slot = q % g.slots;
        const uint32_t use = uint32_t(q / g.slots);
        if (use > 0 && !mbar_wait_bounded(&empty[slot], (use - 1) & 1u, kRowWaitLimitNs)) bad = true;
        if (lane == 0) {
            const int64_t i = t / g.tps;
            const int p0 = int((t - i * g.tps) * g.P);
            const int pa = int(a.l - p0 < g.P ? a.l - p0 : g.P);
            unsigned char* base = ring + size_t(slot) * g.slot_bytes;
            uint32_t tx = (BWD ? 2u : 1u) * g.tx_tensor;
            if (BWD) tx += 2u * uint32_t(pa) * 4u;
            mbar_arrive_expect_tx(&full[slot], tx);
            for (int b = 0; b < g.nb; ++b) {
                const size_t off = size_t(b) * g.cb * g.P * sizeof(T);
                tma_load_3d(base + off, map_a, p0, b * g.cb, int(i), &full[slot], pol);
                if (BWD) tma_load_3d(base + tensor_bytes + off, map_b, p0, b * g.cb, int(i), &full[slot], pol);
            }
            if (BWD) {
                float* st = reinterpret_cast<float*>(base + 2 * tensor_bytes);
                bulk_g2s(st, a.mean_in + i * a.l + p0, uint32_t(pa) * 4u, &full[slot], pol);
                bulk_g2s(st + g.P, a.rstd_in + i * a.l + p0, uint32_t(pa) * 4u, &full[slot], pol);
            }
        }
        __syncwarp();
    }
}

// Waits (bounded) until the last copies into every slot have landed, so that
// no copy is in flight when the CTA exits even after a wait gave up.
__device__ __forceinline__ void cfr_drain(const CfrGeom& g, uint64_t* full, int nq, bool& bad) {
    for (int s = 0; s < g.slots && s < nq; ++s) {
        const int last = s + ((nq - 1 - s) / g.slots) * g.slots;  // last tile index using slot s
        if (!mbar_wait_bounded(&full[s], uint32_t(last / g.slots) & 1u, kRowWaitLimitNs)) bad = true;
    }
}

// Channels of a group: g, g + CG, ... below c.
__device__ __forceinline__ int cfr_group_channels(int grp, int CG, int c) {
    return grp < c ? (c - 1 - grp) / CG + 1 : 0;
}

// The CTA's tiles (b, b + grid, ... below `tiles`).
__device__ __forceinline__ int cfr_cta_tiles(int64_t tiles) {
    return int((tiles - blockIdx.x + gridDim.x - 1) / gridDim.x);
}

template <typename T>
__global__ void __launch_bounds__(kCfrThreads, 1)
lncf_fwd_ring_kernel(const CfArgs a, const CfrGeom g, const __grid_constant__ CUtensorMap map_x) {
    constexpr int V = kVec<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kCfrMaxSlots];
    __shared__ __align__(8) uint64_t empty[kCfrMaxSlots];
    __shared__ int s_bad;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c = int(a.c);
    const int PV = g.pv, P = g.P;
    const int CG = kCfrTeamThreads / PV;
    float* wsm = reinterpret_cast<float*>(smem);
    float* bsm = wsm + c;
    float* scratch = reinterpret_cast<float*>(smem + g.param_bytes);
    float* fac = scratch + kCfrTeams * kCfrTeamFloatsPerPos * P;  // [8][2]: Chan merge factors per team warp
    unsigned char* ring = smem + g.param_bytes + g.part_bytes;
    bool bad = false;

    if (threadIdx.x == 0) {
        s_bad = 0;
        for (int i = 0; i < g.slots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCfrTeamWarps);
        }
        mbar_init_fence();
        // merging team warp w's (n_w, mean_w, M2_w) into the first w warps' running
        // (N, mean, M2): mean += d*n_w/N', M2 += M2_w + d^2*N*n_w/N', N' = N + n_w
        float n_before = 0.f;
        for (int w = 0; w < kCfrTeamWarps; ++w) {
            float nw = 0.f;
            for (int gg = w * 32 / PV; gg < (w + 1) * 32 / PV; ++gg) nw += float(cfr_group_channels(gg, CG, c));
            const float nt = n_before + nw;
            const float f = nt > 0.f ? nw / nt : 0.f;
            fac[2 * w] = f;
            fac[2 * w + 1] = n_before * f;
            n_before = nt;
        }
    }
    if (warp == kCfrConsumerWarps && lane == 0) tma_prefetch_map(&map_x);
    using bits = typename Io<T>::bits_t;
    for (int ch = threadIdx.x; ch < c; ch += kCfrThreads) {
        wsm[ch] = a.w ? Io<T>::load(reinterpret_cast<const bits*>(a.w)[ch]) : 1.f;
        bsm[ch] = a.b ? Io<T>::load(reinterpret_cast<const bits*>(a.b)[ch]) : 0.f;
    }
    __syncthreads();

    if (warp == kCfrConsumerWarps) {
        cfr_produce<T, false>(a, g, ring, full, empty, &map_x, nullptr, lane, bad);
    } else {
        const int team = warp / kCfrTeamWarps;
        const int tw = warp % kCfrTeamWarps;
        const int t = threadIdx.x % kCfrTeamThreads;
        const int pv = t % PV;
        const int grp = t / PV;
        const int my_ch = cfr_group_channels(grp, CG, c);
        const size_t row = size_t(P) * sizeof(T);
        const float inv_c = 1.f / float(c);
        float* part = scratch + team * kCfrTeamFloatsPerPos * P;  // [8][2][V][PV]
        float* stat = part + kCfrTeamWarps * 2 * P;               // [2 parities][2][V][PV]
        T* __restrict__ y = reinterpret_cast<T*>(a.y);
        const int nq = cfr_cta_tiles(g.tiles);
        for (int q = team; q < nq; q += kCfrTeams) {
            const int64_t tt = blockIdx.x + int64_t(q) * gridDim.x;
            const int slot = q % g.slots;
            if (!mbar_wait_bounded_sleep(&full[slot], uint32_t(q / g.slots) & 1u, kRowWaitLimitNs)) bad = true;
            const int64_t i = tt / g.tps;
            const int p0 = int((tt - i * g.tps) * P);
            const bool on = p0 + pv * V < a.l;  // V divides l: a vector is all in or all out
            const unsigned char* base = ring + size_t(slot) * g.slot_bytes + size_t(pv) * 16;
            float* st = stat + ((q / kCfrTeams) & 1) * 2 * P;
            // ---- pass 1: (count, mean, M2) of the group's channels per position,
            // from sums shifted by the group's first channel ----
            constexpr int H = kPairs<T>;
            float mean[V], m2[V];
#pragma unroll
            for (int k = 0; k < V; ++k) mean[k] = m2[k] = 0.f;
            if (on && my_ch > 0) {
                float2 kk[H], nk[H], s[H], sq[H];
                cfr_load2<T>(base + size_t(grp) * row, kk);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    nk[h] = f2neg(kk[h]);
                    s[h] = sq[h] = f2(0.f);
                }
                const unsigned char* pch = base + size_t(grp + CG) * row;
                const size_t step = size_t(CG) * row;
                for (int j = 1; j < my_ch; ++j, pch += step) {
                    float2 v[H];
                    cfr_load2<T>(pch, v);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 d = __fadd2_rn(v[h], nk[h]);
                        s[h] = __fadd2_rn(s[h], d);
                        sq[h] = __ffma2_rn(d, d, sq[h]);
                    }
                }
                const float rc = 1.f / float(my_ch);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    mean[2 * h] = fmaf(s[h].x, rc, kk[h].x);
                    mean[2 * h + 1] = fmaf(s[h].y, rc, kk[h].y);
                    m2[2 * h] = fmaxf(fmaf(-s[h].x, s[h].x * rc, sq[h].x), 0.f);
                    m2[2 * h + 1] = fmaxf(fmaf(-s[h].y, s[h].y * rc, sq[h].y), 0.f);
                }
            }
            // groups that share a warp (PV < 32) hold the same positions: merge them
            float cnt = float(my_ch);
            for (int o = PV; o < 32; o <<= 1) {
                const float nb = __shfl_xor_sync(0xffffffffu, cnt, o);
                const float nt = cnt + nb;
                const float f = nt > 0.f ? __fdividef(nb, nt) : 0.f;
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const float mb = __shfl_xor_sync(0xffffffffu, mean[k], o);
                    const float qb = __shfl_xor_sync(0xffffffffu, m2[k], o);
                    const float d = mb - mean[k];
                    mean[k] = fmaf(d, f, mean[k]);
                    m2[k] = m2[k] + qb + d * d * cnt * f;
                }
                cnt = nt;
            }
            if (lane < PV) {
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    part[(tw * 2 + 0) * P + k * PV + pv] = mean[k];
                    part[(tw * 2 + 1) * P + k * PV + pv] = m2[k];
                }
            }
            named_barrier(kCfrBarTeam + team, kCfrTeamThreads);
            // ---- Chan merge per position (index k*PV + pv), fixed warp order ----
            if (t < P) {
                const int pos = (t % PV) * V + t / PV;
                if (p0 + pos < a.l) {
                    float mu = 0.f, q2 = 0.f;
#pragma unroll
                    for (int w = 0; w < kCfrTeamWarps; ++w) {
                        const float d = part[(w * 2 + 0) * P + t] - mu;
                        mu = fmaf(d, fac[2 * w], mu);
                        q2 = q2 + part[(w * 2 + 1) * P + t] + d * d * fac[2 * w + 1];
                    }
                    const float rs = rsqrtf(q2 * inv_c + a.eps);
                    st[t] = mu;
                    st[P + t] = rs;
                    if (a.mean) a.mean[i * a.l + p0 + pos] = mu;
                    if (a.rstd) a.rstd[i * a.l + p0 + pos] = rs;
                }
            }
            named_barrier(kCfrBarTeam + team, kCfrTeamThreads);
            // ---- pass 2: y = (x - mean) * rstd * w + b ----
            if (on) {
                float2 nmu[H], rs[H];
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    nmu[h] = make_float2(-st[(2 * h) * PV + pv], -st[(2 * h + 1) * PV + pv]);
                    rs[h] = make_float2(st[P + (2 * h) * PV + pv], st[P + (2 * h + 1) * PV + pv]);
                }
                T* yb = y + i * a.c * a.l + p0 + pv * V + int64_t(grp) * a.l;
                const int64_t ystep = int64_t(CG) * a.l;
                const unsigned char* pch = base + size_t(grp) * row;
                const size_t step = size_t(CG) * row;
                for (int j = 0; j < my_ch; ++j, pch += step, yb += ystep) {
                    const int ch = grp + j * CG;
                    float2 v[H], o[H];
                    cfr_load2<T>(pch, v);
                    const float2 wc = f2(wsm[ch]), bc = f2(bsm[ch]);
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        o[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(v[h], nmu[h]), rs[h]), wc, bc);
                    cfr_store2<T>(yb, o);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        named_barrier(kCfrBarAll, kCfrConsumers);
        if (threadIdx.x == 0) cfr_drain(g, full, nq, bad);
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0 && s_bad) atomicOr(a.err, kErrTimeoutStage);
}

template <typename T>
__global__ void __launch_bounds__(kCfrThreads, 1)
lncf_bwd_ring_kernel(const CfArgs a, const CfrGeom g, const __grid_constant__ CUtensorMap map_dy,
                     const __grid_constant__ CUtensorMap map_x) {
    constexpr int V = kVec<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kCfrMaxSlots];
    __shared__ __align__(8) uint64_t empty[kCfrMaxSlots];
    __shared__ int s_bad;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c = int(a.c);
    const int PV = g.pv, P = g.P;
    const int CG = kCfrTeamThreads / PV;
    float* wsm = reinterpret_cast<float*>(smem);
    float* scratch = reinterpret_cast<float*>(smem + g.param_bytes);
    float* acc = reinterpret_cast<float*>(smem + g.param_bytes + g.part_bytes);  // [team][dw, db][c]
    unsigned char* ring = smem + g.param_bytes + g.part_bytes + g.acc_bytes;
    const bool grads = a.ws_dw != nullptr;
    bool bad = false;

    if (threadIdx.x == 0) {
        s_bad = 0;
        for (int i = 0; i < g.slots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCfrTeamWarps);
        }
        mbar_init_fence();
    }
    if (warp == kCfrConsumerWarps && lane == 0) {
        tma_prefetch_map(&map_dy);
        tma_prefetch_map(&map_x);
    }
    using bits = typename Io<T>::bits_t;
    for (int ch = threadIdx.x; ch < c; ch += kCfrThreads) {
        wsm[ch] = a.w ? Io<T>::load(reinterpret_cast<const bits*>(a.w)[ch]) : 1.f;
#pragma unroll
        for (int k = 0; k < 2 * kCfrTeams; ++k) acc[k * c + ch] = 0.f;
    }
    __syncthreads();

    if (warp == kCfrConsumerWarps) {
        cfr_produce<T, true>(a, g, ring, full, empty, &map_dy, &map_x, lane, bad);
    } else {
        const int team = warp / kCfrTeamWarps;
        const int tw = warp % kCfrTeamWarps;
        const int t = threadIdx.x % kCfrTeamThreads;
        const int pv = t % PV;
        const int grp = t / PV;
        const int nch = (c + CG - 1) / CG;  // uniform trip count (the channel shuffles need it)
        const int my_ch = cfr_group_channels(grp, CG, c);
        const size_t row = size_t(P) * sizeof(T);
        const size_t tensor_bytes = size_t(g.nb) * g.cb * row;
        const float inv_c = 1.f / float(c);
        float* part = scratch + team * kCfrTeamFloatsPerPos * P;  // [8][2][V][PV]
        float* coef = part + kCfrTeamWarps * 2 * P;               // [2 parities][2][V][PV]
        float* tacc = acc + team * 2 * c;
        T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
        const int nq = cfr_cta_tiles(g.tiles);
        for (int q = team; q < nq; q += kCfrTeams) {
            const int64_t tt = blockIdx.x + int64_t(q) * gridDim.x;
            const int slot = q % g.slots;
            if (!mbar_wait_bounded_sleep(&full[slot], uint32_t(q / g.slots) & 1u, kRowWaitLimitNs)) bad = true;
            const int64_t i = tt / g.tps;
            const int p0 = int((tt - i * g.tps) * P);
            const bool on = p0 + pv * V < a.l;
            const unsigned char* sbase = ring + size_t(slot) * g.slot_bytes;
            const unsigned char* dyb = sbase + size_t(pv) * 16;
            const float* sst = reinterpret_cast<const float*>(sbase + 2 * tensor_bytes);  // mean [P], rstd [P]
            float* cf = coef + ((q / kCfrTeams) & 1) * 2 * P;
            constexpr int H = kPairs<T>;
            float2 nmu[H], rs[H];
            if (on) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 m = *reinterpret_cast<const float2*>(sst + pv * V + 2 * h);
                    nmu[h] = f2neg(m);
                    rs[h] = *reinterpret_cast<const float2*>(sst + P + pv * V + 2 * h);
                }
            }
            const size_t step = size_t(CG) * row;
            // ---- pass 1: sum g and sum g*xhat over the group's channels, g = dy*w ----
            float2 s1[H], s2[H];
#pragma unroll
            for (int h = 0; h < H; ++h) s1[h] = s2[h] = f2(0.f);
            if (on) {
                const unsigned char* pd = dyb + size_t(grp) * row;
                for (int j = 0; j < my_ch; ++j, pd += step) {
                    const int ch = grp + j * CG;
                    float2 dv[H], xv[H];
                    cfr_load2<T>(pd, dv);
                    cfr_load2<T>(pd + tensor_bytes, xv);
                    const float2 wc = f2(wsm[ch]);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 gg = __fmul2_rn(dv[h], wc);
                        s1[h] = __fadd2_rn(s1[h], gg);
                        s2[h] = __ffma2_rn(gg, __fmul2_rn(__fadd2_rn(xv[h], nmu[h]), rs[h]), s2[h]);
                    }
                }
            }
            for (int o = PV; o < 32; o <<= 1) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    s1[h].x += __shfl_xor_sync(0xffffffffu, s1[h].x, o);
                    s1[h].y += __shfl_xor_sync(0xffffffffu, s1[h].y, o);
                    s2[h].x += __shfl_xor_sync(0xffffffffu, s2[h].x, o);
                    s2[h].y += __shfl_xor_sync(0xffffffffu, s2[h].y, o);
                }
            }
            if (lane < PV) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    part[(tw * 2 + 0) * P + (2 * h) * PV + pv] = s1[h].x;
                    part[(tw * 2 + 0) * P + (2 * h + 1) * PV + pv] = s1[h].y;
                    part[(tw * 2 + 1) * P + (2 * h) * PV + pv] = s2[h].x;
                    part[(tw * 2 + 1) * P + (2 * h + 1) * PV + pv] = s2[h].y;
                }
            }
            named_barrier(kCfrBarTeam + team, kCfrTeamThreads);
            if (t < P) {
                float S1 = 0.f, S2 = 0.f;
#pragma unroll
                for (int w = 0; w < kCfrTeamWarps; ++w) {
                    S1 += part[(w * 2 + 0) * P + t];
                    S2 += part[(w * 2 + 1) * P + t];
                }
                cf[t] = S1 * inv_c;
                cf[P + t] = S2 * inv_c;
            }
            named_barrier(kCfrBarTeam + team, kCfrTeamThreads);
            // ---- pass 2: dx; this tile's dw, db per channel ----
            float2 nc1[H], nc2[H];
#pragma unroll
            for (int h = 0; h < H; ++h) {
                nc1[h] = make_float2(-cf[(2 * h) * PV + pv], -cf[(2 * h + 1) * PV + pv]);
                nc2[h] = make_float2(-cf[P + (2 * h) * PV + pv], -cf[P + (2 * h + 1) * PV + pv]);
            }
            T* dxb = dx + i * a.c * a.l + p0 + pv * V + int64_t(grp) * a.l;
            const int64_t dstep = int64_t(CG) * a.l;
            const unsigned char* pd = dyb + size_t(grp) * row;
            for (int j = 0; j < nch; ++j, pd += step, dxb += dstep) {
                const int ch = grp + j * CG;
                float pw = 0.f, pb = 0.f;
                if (on && j < my_ch) {
                    float2 dv[H], xv[H], o[H];
                    cfr_load2<T>(pd, dv);
                    cfr_load2<T>(pd + tensor_bytes, xv);
                    const float2 wc = f2(wsm[ch]);
                    float2 pw2 = f2(0.f), pb2 = f2(0.f);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 xh = __fmul2_rn(__fadd2_rn(xv[h], nmu[h]), rs[h]);
                        // rstd * (dy*w - c1 - xhat*c2)
                        const float2 u = __ffma2_rn(xh, nc2[h], __fadd2_rn(__fmul2_rn(dv[h], wc), nc1[h]));
                        o[h] = __fmul2_rn(rs[h], u);
                        pw2 = __ffma2_rn(dv[h], xh, pw2);
                        pb2 = __fadd2_rn(pb2, dv[h]);
                    }
                    cfr_store2<T>(dxb, o);
                    pw = pw2.x + pw2.y;
                    pb = pb2.x + pb2.y;
                }
                if (grads) {
                    // the PV threads of this channel are PV consecutive lanes
                    for (int o = 1; o < PV; o <<= 1) {
                        pw += __shfl_xor_sync(0xffffffffu, pw, o);
                        pb += __shfl_xor_sync(0xffffffffu, pb, o);
                    }
                    if (pv == 0 && j < my_ch) {
                        tacc[ch] += pw;
                        tacc[c + ch] += pb;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        named_barrier(kCfrBarAll, kCfrConsumers);
        if (threadIdx.x == 0) cfr_drain(g, full, nq, bad);
        pdl_trigger();
        if (grads) {
            for (int ch = threadIdx.x; ch < c; ch += kCfrConsumers) {
                a.ws_dw[int64_t(blockIdx.x) * c + ch] = acc[ch] + acc[2 * c + ch];
                if (a.ws_db) a.ws_db[int64_t(blockIdx.x) * c + ch] = acc[c + ch] + acc[3 * c + ch];
            }
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0 && s_bad) atomicOr(a.err, kErrTimeoutStage);
}

}  // namespace nrm
