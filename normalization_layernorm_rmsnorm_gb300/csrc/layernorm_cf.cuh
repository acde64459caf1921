// layernorm_cf.cuh -- LayerNorm over the channels of an NCHW tensor (channels
// first: x[n, c, l], l = H*W, normalised over c for every sample and spatial
// position), forward and backward, for one storage dtype T (included by
// rownorm.cuh).
//
// What is computed is the LayerNorm of the attorch normalization article
// ("attorch如何实现LayerNorm、BatchNorm与RMSNorm？3种归一化Triton核代码全解析",
// section "LayerNorm：一个程序归一化一批行"), taken for each (sample, position)
// over its c channels, as ConvNeXt -- which the article's application
// paragraph lists as a LayerNorm user -- normalises channels.
//
// Design: a CTA of 8 warps owns a tile of 32*V*K positions of one sample: each
// lane K groups of V consecutive positions, 32*V apart (V = 16/sizeof(T) when
// rows are 16-byte aligned, else 1; K > 1 only for those scalar planes), so
// every load is a coalesced run of the tile in one channel plane.
// Warp w takes channels w, w+8, ...; per-position statistics are merged across
// the 8 warps in shared memory in a fixed order.  The second pass re-reads the
// tile (L2: a CTA's tile is c*32*V*K elements).  The backward keeps the per-CTA
// dw/db partial row in shared memory (channel ch belongs to warp ch % 8, so
// no atomics) and writes it to the workspace for the fixed-order column sum.
#pragma once

namespace nrm {

constexpr int kCfWarps = 8;
constexpr int kCfThreads = kCfWarps * 32;

template <typename T, int V>
__device__ __forceinline__ void cf_load(const T* p, float (&v)[V]) {
    if constexpr (V > 1) {
        Pack<T, V> pk;
        pk.u = ld_cached_v4(p);
#pragma unroll
        for (int k = 0; k < V; ++k) v[k] = Io<T>::load(pk.b[k]);
    } else {
        v[0] = Io<T>::load(*reinterpret_cast<const typename Io<T>::bits_t*>(p));
    }
}

template <typename T, int V>
__device__ __forceinline__ void cf_store(T* p, const float (&v)[V]) {
    if constexpr (V > 1) {
        store_vec<T, V>(p, v);
    } else {
        *reinterpret_cast<typename Io<T>::bits_t*>(p) = Io<T>::store(v[0]);
    }
}

template <typename T>
__device__ __forceinline__ float cf_wb(const void* p, int64_t ch, float dflt) {
    if (!p) return dflt;
    return Io<T>::load(reinterpret_cast<const typename Io<T>::bits_t*>(p)[ch]);
}

// Tile t of the grid: sample i, first position p_base.
struct CfTile {
    int64_t i, p_base;
};
__device__ __forceinline__ CfTile cf_tile(int64_t t, int64_t tiles_per_sample, int pw) {
    CfTile r;
    r.i = t / tiles_per_sample;
    r.p_base = (t - r.i * tiles_per_sample) * pw;
    return r;
}

// K groups of V positions per lane, strided by 32*V: a tile of PW = 32*V*K
// positions.  K > 1 serves planes that are not 16-byte multiples (V = 1), so
// that a 7x7 or 14x14 plane is one tile rather than two to seven of 32.
template <typename T, int V, int K = 1>
__global__ void __launch_bounds__(kCfThreads)
lncf_fwd_kernel(const CfArgs a) {
    constexpr int PW = 32 * V * K;  // positions per tile
    __shared__ float part[kCfWarps][3][PW];  // per warp and position: n, mean, m2
    __shared__ float stat[2][PW];            // mean, rstd per position
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t c = a.c, l = a.l;
    const int64_t tps = (l + PW - 1) / PW;
    const int64_t tiles = a.n * tps;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    T* __restrict__ y = reinterpret_cast<T*>(a.y);

    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const CfTile tl = cf_tile(t, tps, PW);
        int64_t p0[K];
        bool on[K];
        bool any = false;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            p0[j] = tl.p_base + (j * 32 + lane) * V;
            on[j] = p0[j] < l;  // V divides l on the vector path
            any |= on[j];
        }
        const T* xs = x + tl.i * c * l;
        // ---- pass 1: shifted sums over this warp's channels ----
        float kk[K][V], s[K][V], q[K][V];
        int cnt = 0;
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int k = 0; k < V; ++k) kk[j][k] = s[j][k] = q[j][k] = 0.f;
        if (any) {
            for (int64_t ch = warp; ch < c; ch += kCfWarps) {
                float v[K][V];
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (on[j]) {
                        cf_load<T, V>(xs + ch * l + p0[j], v[j]);
                    } else {
#pragma unroll
                        for (int k = 0; k < V; ++k) v[j][k] = 0.f;
                    }
                }
                if (cnt == 0) {
#pragma unroll
                    for (int j = 0; j < K; ++j)
#pragma unroll
                        for (int k = 0; k < V; ++k) kk[j][k] = v[j][k];
                }
#pragma unroll
                for (int j = 0; j < K; ++j)
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        const float d = v[j][k] - kk[j][k];
                        s[j][k] += d;
                        q[j][k] = fmaf(d, d, q[j][k]);
                    }
                ++cnt;
            }
        }
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int pi = (j * 32 + lane) * V + k;
                const float fn = on[j] ? float(cnt) : 0.f;
                part[warp][0][pi] = fn;
                part[warp][1][pi] = fn > 0.f ? kk[j][k] + s[j][k] / fn : 0.f;
                part[warp][2][pi] = fn > 0.f ? fmaxf(q[j][k] - s[j][k] * (s[j][k] / fn), 0.f) : 0.f;
            }
        __syncthreads();
        // ---- merge the 8 warps per position (fixed order) ----
        for (int pi = threadIdx.x; pi < PW; pi += kCfThreads) {
            Moments m{0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kCfWarps; ++w) chan_merge(m, part[w][0][pi], part[w][1][pi], part[w][2][pi]);
            const float rs = rsqrtf(m.m2 / float(c) + a.eps);
            stat[0][pi] = m.mean;
            stat[1][pi] = rs;
            const int64_t p = tl.p_base + pi;
            if (p < l) {
                if (a.mean) a.mean[tl.i * l + p] = m.mean;
                if (a.rstd) a.rstd[tl.i * l + p] = rs;
            }
        }
        __syncthreads();
        // ---- pass 2: y = (x - mean)*rstd*w + b ----
        if (any) {
            float mu[K][V], rs[K][V];
#pragma unroll
            for (int j = 0; j < K; ++j)
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    mu[j][k] = stat[0][(j * 32 + lane) * V + k];
                    rs[j][k] = stat[1][(j * 32 + lane) * V + k];
                }
            T* ys = y + tl.i * c * l;
            for (int64_t ch = warp; ch < c; ch += kCfWarps) {
                const float wc = cf_wb<T>(a.w, ch, 1.f);
                const float bc = cf_wb<T>(a.b, ch, 0.f);
                float v[K][V];
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (on[j]) cf_load<T, V>(xs + ch * l + p0[j], v[j]);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (on[j]) {
                        float o[V];
#pragma unroll
                        for (int k = 0; k < V; ++k) o[k] = fmaf((v[j][k] - mu[j][k]) * rs[j][k], wc, bc);
                        cf_store<T, V>(ys + ch * l + p0[j], o);
                    }
                }
            }
        }
        __syncthreads();  // part / stat are rewritten by the next tile
    }
}

template <typename T, int V, int K = 1>
__global__ void __launch_bounds__(kCfThreads)
lncf_bwd_kernel(const CfArgs a) {
    constexpr int PW = 32 * V * K;
    __shared__ float part[kCfWarps][2][PW];  // per warp and position: sum g, sum g*xhat
    __shared__ float coef[2][PW];            // c1, c2 per position
    extern __shared__ float acc[];           // [2][c]: this CTA's dw, db partial row
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t c = a.c, l = a.l;
    const int64_t tps = (l + PW - 1) / PW;
    const int64_t tiles = a.n * tps;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ dy = reinterpret_cast<const T*>(a.dy);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    const bool grads = a.ws_dw != nullptr;
    if (grads)
        for (int64_t i = threadIdx.x; i < 2 * c; i += kCfThreads) acc[i] = 0.f;
    __syncthreads();

    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const CfTile tl = cf_tile(t, tps, PW);
        int64_t p0[K];
        bool on[K];
        bool any = false;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            p0[j] = tl.p_base + (j * 32 + lane) * V;
            on[j] = p0[j] < l;
            any |= on[j];
        }
        const int64_t base = tl.i * c * l;
        float mu[K][V], rs[K][V];
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int k = 0; k < V; ++k) {
                mu[j][k] = on[j] ? a.mean_in[tl.i * l + p0[j] + k] : 0.f;
                rs[j][k] = on[j] ? a.rstd_in[tl.i * l + p0[j] + k] : 0.f;
            }
        // ---- pass 1: sum g and sum g*xhat over this warp's channels, g = dy*w ----
        float s1[K][V], s2[K][V];
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int k = 0; k < V; ++k) s1[j][k] = s2[j][k] = 0.f;
        if (any) {
            for (int64_t ch = warp; ch < c; ch += kCfWarps) {
                float dv[K][V], xv[K][V];
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (on[j]) {
                        cf_load<T, V>(dy + base + ch * l + p0[j], dv[j]);
                        cf_load<T, V>(x + base + ch * l + p0[j], xv[j]);
                    }
                }
                const float wc = cf_wb<T>(a.w, ch, 1.f);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (on[j]) {
#pragma unroll
                        for (int k = 0; k < V; ++k) {
                            const float g = dv[j][k] * wc;
                            s1[j][k] += g;
                            s2[j][k] = fmaf(g, (xv[j][k] - mu[j][k]) * rs[j][k], s2[j][k]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int k = 0; k < V; ++k) {
                part[warp][0][(j * 32 + lane) * V + k] = s1[j][k];
                part[warp][1][(j * 32 + lane) * V + k] = s2[j][k];
            }
        __syncthreads();
        for (int pi = threadIdx.x; pi < PW; pi += kCfThreads) {
            float t1 = 0.f, t2 = 0.f;
#pragma unroll
            for (int w = 0; w < kCfWarps; ++w) {
                t1 += part[w][0][pi];
                t2 += part[w][1][pi];
            }
            coef[0][pi] = t1 / float(c);
            coef[1][pi] = t2 / float(c);
        }
        __syncthreads();
        // ---- pass 2: dx; this tile's dw, db per channel ----
        float c1[K][V], c2[K][V];
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int k = 0; k < V; ++k) {
                c1[j][k] = coef[0][(j * 32 + lane) * V + k];
                c2[j][k] = coef[1][(j * 32 + lane) * V + k];
            }
        for (int64_t ch = warp; ch < c; ch += kCfWarps) {
            float pw = 0.f, pb = 0.f;
            if (any) {
                float dv[K][V], xv[K][V];
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (on[j]) {
                        cf_load<T, V>(dy + base + ch * l + p0[j], dv[j]);
                        cf_load<T, V>(x + base + ch * l + p0[j], xv[j]);
                    }
                }
                const float wc = cf_wb<T>(a.w, ch, 1.f);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (on[j]) {
                        float o[V];
#pragma unroll
                        for (int k = 0; k < V; ++k) {
                            const float xh = (xv[j][k] - mu[j][k]) * rs[j][k];
                            o[k] = rs[j][k] * (dv[j][k] * wc - c1[j][k] - xh * c2[j][k]);
                            pw = fmaf(dv[j][k], xh, pw);
                            pb += dv[j][k];
                        }
                        cf_store<T, V>(dx + base + ch * l + p0[j], o);
                    }
                }
            }
            if (grads) {
                pw = warp_sum(pw);
                pb = warp_sum(pb);
                if (lane == 0) {
                    acc[ch] += pw;
                    acc[c + ch] += pb;
                }
            }
        }
        __syncthreads();
    }
    pdl_trigger();
    if (grads) {
        for (int64_t ch = threadIdx.x; ch < c; ch += kCfThreads) {
            a.ws_dw[int64_t(blockIdx.x) * c + ch] = acc[ch];
            if (a.ws_db) a.ws_db[int64_t(blockIdx.x) * c + ch] = acc[c + ch];
        }
    }
}

}  // namespace nrm
