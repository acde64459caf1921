// rownorm.cuh -- LayerNorm and RMSNorm over the last dimension, forward and
// backward, for one storage dtype T (included by rownorm_<dtype>.cu).
//
// What is computed follows the attorch normalization article
// ("attorch如何实现LayerNorm、BatchNorm与RMSNorm？3种归一化Triton核代码全解析"):
//   section "LayerNorm：一个程序归一化一批行" -- a program normalises a block of
//     rows held whole in registers: row mean, variance from squared deviations
//     of that mean, a reciprocal square root, optional stats, weight and bias;
//     the backward needs two row sums and finishes a row in one launch;
//   section "RMSNorm：去掉均值的极简版 LayerNorm" -- the same without the mean,
//     backward with one row sum of input * output_grad * weight;
//   section "三种核共享的工程技巧" -- fp32 accumulation, masks for ragged sizes,
//     weight/bias gradients written per row block and then summed.
//
// GB300 design:
//   * A row is held in registers by a group of TPR threads (a power of two from
//     32 to 1024), each thread holding up to 4 (forward) or 2 (backward) raw
//     16-byte vectors, unpacked to fp32 where used, so x is read from HBM once.
//     Vector j of thread t is vector j*TPR + t of the row: a warp's accesses
//     for one j are 512 contiguous bytes.
//   * Group sums are warp butterflies, plus a named barrier and a fixed-order
//     pass over shared memory when a group spans several warps.  The mean is
//     subtracted from the registers before the variance sum (exact two-pass).
//   * Grids are persistent: at most (resident CTAs per SM) x (SMs) CTAs, each
//     looping over row groups with a stride, so each CTA's dw/db partials cover
//     a fixed set of rows.
//   * dw/db: each thread accumulates its columns over its rows in fp32
//     registers; the CTA reduces its row groups in a fixed order and writes one
//     partial row to the workspace; a second kernel (launched with programmatic
//     dependent launch) sums the partial rows column-wise in a fixed order.  No
//     atomics, so the result is bitwise reproducible.
//   * The backward of 16-byte-aligned rows up to 2048 vectors streams rows
//     through shared memory with bulk copies (rowring.cuh).  The register
//     backward (other rows) prefetches the next row of its group into
//     registers while the current row is being reduced, so two rows per group
//     are in flight.
//   * Rows too wide for registers (more than 4096 vectors forward or 1024
//     backward; elements on the unaligned path) take a two-pass "wide" kernel: Welford/Chan
//     statistics in one pass over global memory, then a normalising pass.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace nrm {

constexpr int kRowFwdVpt = 4;         // 16-byte vectors per thread, forward
constexpr int kRowBwdVpt = 2;         // 16-byte vectors per thread, backward
constexpr int kRowBwdBlock = 512;     // threads per backward CTA
constexpr int kRowWideBlock = 1024;   // threads per CTA of the wide-row kernels
constexpr int kRowMaxFwdTpr = 1024;
constexpr int kRowMaxBwdTpr = 512;

// Threads per forward CTA: 128 for rows of up to 128 threads (finer occupancy
// steps: measured faster than 256 on the ViT-B LayerNorm and LLaMA RMSNorm rows).
__host__ __device__ constexpr int row_fwd_block(int tpr) { return tpr > 128 ? (tpr > 256 ? tpr : 256) : 128; }

// Sum of NV values over the TPR threads of row group `group`.  For TPR > 32
// the per-warp sums meet in shared memory `buf` ([2][TPR/32][NV] floats for
// this group), double-buffered by `phase`, behind named barrier 1 + group.
template <int TPR, int NV>
__device__ __forceinline__ void group_sum(float (&v)[NV], float* buf, int& phase, int group) {
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = warp_sum(v[k]);
    if constexpr (TPR > 32) {
        constexpr int NW = TPR / 32;
        const int lane = threadIdx.x & 31;
        const int wig = (threadIdx.x % TPR) >> 5;
        float* b = buf + phase * NW * NV;
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < NV; ++k) b[wig * NV + k] = v[k];
        }
        named_barrier(1 + group, TPR);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += b[w * NV + k];
            v[k] = s;
        }
        phase ^= 1;
    }
}

template <typename T, int VE>
__device__ __forceinline__ void load_raw(const T* p, Pack<T, VE>& pk, bool stream) {
    if constexpr (VE > 1) {
        pk.u = stream ? ld_stream_v4(p) : ld_cached_v4(p);
    } else {
        const typename Io<T>::bits_t* q = reinterpret_cast<const typename Io<T>::bits_t*>(p);
        pk.b[0] = stream ? q[0] : __ldg(q);
    }
}

template <typename T, int VE>
__device__ __forceinline__ float elem(const Pack<T, VE>& pk, int k) {
    return Io<T>::load(pk.b[k]);
}

template <typename T, int VE>
__device__ __forceinline__ void load_param(const void* p, int vi, float (&out)[VE], float dflt) {
    if (p) {
        load_vec<T, VE, false>(reinterpret_cast<const T*>(p) + int64_t(vi) * VE, out);
    } else {
#pragma unroll
        for (int k = 0; k < VE; ++k) out[k] = dflt;
    }
}

// Row `row` of a [rows, cols] tensor as this thread's VPT packs (zero where
// the vector lies past the end of the row).
template <typename T, int TPR, int VPT, int VE>
__device__ __forceinline__ void load_row(const T* base, int64_t row, int cols, int t,
                                         Pack<T, VE> (&pk)[VPT]) {
    const int nvec = cols / VE;
    const T* r = base + row * cols;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int vi = j * TPR + t;
        if (vi < nvec) {
            load_raw<T, VE>(r + int64_t(vi) * VE, pk[j], true);
        } else {
            pk[j].u = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// ---------------------------------------------------------------------------
// forward, rows held in registers
// ---------------------------------------------------------------------------
// TO: the output's storage type (T, or float for a 16-bit input whose output
// is kept in float32).
template <typename T, bool LN, int TPR, int VE, int VPT = kRowFwdVpt, typename TO = T>
__global__ void __launch_bounds__(row_fwd_block(TPR))
row_fwd_kernel(const RowArgs a) {
    constexpr int BLOCK = row_fwd_block(TPR);
    constexpr int RPC = BLOCK / TPR;
    constexpr int NW = TPR / 32;
    __shared__ float red[RPC][2 * NW];

    const int group = threadIdx.x / TPR;
    const int t = threadIdx.x % TPR;
    const int cols = a.cols;
    const int nvec = cols / VE;
    const float fcols = float(cols);
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    TO* __restrict__ y = reinterpret_cast<TO*>(a.y);
    int phase = 0;

    const int64_t stride = int64_t(gridDim.x) * RPC;
    int64_t row = int64_t(blockIdx.x) * RPC + group;
    const float inv_cols = 1.f / fcols;  // mean = sum * (1/cols): one division per thread
    if constexpr (VE > 1) {
        // 16-byte vectors: the element arithmetic on fp32 pairs, and the next
        // row of the group loaded while this one is normalised
        constexpr int H = VE / 2;
        // this thread's columns of w and b, the same for every row: for one-warp
        // rows (short rows, where per-row work is small) loaded once, as fp32
        // pairs for up to 3 vectors per thread and as packed T for 4 (fp32
        // pairs would take 32 more registers there); wider rows reload them
        // per row (registers for occupancy)
        constexpr bool kHoist = TPR == 32;
        constexpr bool kHoistF = kHoist && VPT <= 3;
        float2 wf[kHoistF ? VPT : 1][H], bf[kHoistF ? VPT : 1][H];
        Pack<T, VE> wpk[kHoist && !kHoistF ? VPT : 1], bpk[kHoist && !kHoistF ? VPT : 1];
        if constexpr (kHoist) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int vi = j * TPR + t;
                Pack<T, VE> pw, pb;
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    pw.b[k] = Io<T>::store(1.f);
                    pb.b[k] = Io<T>::store(0.f);
                }
                if (vi < nvec) {
                    if (a.w) pw.u = ld_cached_v4(reinterpret_cast<const T*>(a.w) + int64_t(vi) * VE);
                    if (a.b) pb.u = ld_cached_v4(reinterpret_cast<const T*>(a.b) + int64_t(vi) * VE);
                }
                if constexpr (kHoistF) {
                    unpack2<T>(pw.u, wf[j]);
                    unpack2<T>(pb.u, bf[j]);
                } else {
                    wpk[j] = pw;
                    bpk[j] = pb;
                }
            }
        }
        Pack<T, VE> xp[VPT];
        if (row < a.rows) load_row<T, TPR, VPT, VE>(x, row, cols, t, xp);
        for (; row < a.rows; row += stride) {
            Pack<T, VE> xn[VPT];
            if (row + stride < a.rows) load_row<T, TPR, VPT, VE>(x, row + stride, cols, t, xn);
            TO* yr = y + row * cols;
            float2 xv[VPT][H];
#pragma unroll
            for (int j = 0; j < VPT; ++j) unpack2<T>(xp[j].u, xv[j]);
            float mu = 0.f;
            float2 q2 = f2(0.f);
            if constexpr (LN) {
                float2 s2 = f2(0.f);
#pragma unroll
                for (int j = 0; j < VPT; ++j)
#pragma unroll
                    for (int h = 0; h < H; ++h) s2 = __fadd2_rn(s2, xv[j][h]);
                float s[1] = {s2.x + s2.y};
                group_sum<TPR, 1>(s, &red[group][0], phase, group);
                mu = s[0] * inv_cols;
                const float2 nmu = f2(-mu);
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (j * TPR + t < nvec) {  // the zero padding past the row is not centred
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            xv[j][h] = __fadd2_rn(xv[j][h], nmu);
                            q2 = __ffma2_rn(xv[j][h], xv[j][h], q2);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < VPT; ++j)
#pragma unroll
                    for (int h = 0; h < H; ++h) q2 = __ffma2_rn(xv[j][h], xv[j][h], q2);
            }
            float q[1] = {q2.x + q2.y};
            group_sum<TPR, 1>(q, &red[group][0], phase, group);
            const float rs = rsqrtf(q[0] * inv_cols + a.eps);
            if (t == 0) {
                if (LN && a.mean) a.mean[row] = mu;
                if (a.rstd) a.rstd[row] = rs;
            }
            const float2 rs2 = f2(rs);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int vi = j * TPR + t;
                if (vi < nvec) {
                    float2 wv[H], bv[H], o[H];
                    if constexpr (kHoistF) {
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            wv[h] = wf[j][h];
                            bv[h] = bf[j][h];  // LayerNorm's bias, or RMSNorm's optional one (else 0)
                        }
                    } else if constexpr (kHoist) {
                        unpack2<T>(wpk[j].u, wv);
                        unpack2<T>(bpk[j].u, bv);
                    } else {
                        if (a.w) {
                            unpack2<T>(ld_cached_v4(reinterpret_cast<const T*>(a.w) + int64_t(vi) * VE), wv);
                        } else {
#pragma unroll
                            for (int h = 0; h < H; ++h) wv[h] = f2(1.f);
                        }
                        if (a.b) {  // LayerNorm's bias, or RMSNorm's optional one
                            unpack2<T>(ld_cached_v4(reinterpret_cast<const T*>(a.b) + int64_t(vi) * VE), bv);
                        } else {
#pragma unroll
                            for (int h = 0; h < H; ++h) bv[h] = f2(0.f);
                        }
                    }
#pragma unroll
                    for (int h = 0; h < H; ++h) o[h] = __ffma2_rn(__fmul2_rn(xv[j][h], rs2), wv[h], bv[h]);
                    if constexpr (sizeof(TO) == sizeof(T)) {
                        st_v4(yr + int64_t(vi) * VE, pack2x<T>(o));
                    } else {  // float32 output of a 16-bit input: two 16-byte stores
                        st_v4(yr + int64_t(vi) * VE, make_uint4(__float_as_uint(o[0].x), __float_as_uint(o[0].y),
                                                                __float_as_uint(o[1].x), __float_as_uint(o[1].y)));
                        st_v4(yr + int64_t(vi) * VE + 4,
                              make_uint4(__float_as_uint(o[2].x), __float_as_uint(o[2].y), __float_as_uint(o[3].x),
                                         __float_as_uint(o[3].y)));
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < VPT; ++j) xp[j] = xn[j];
        }
    } else {
        for (; row < a.rows; row += stride) {
            Pack<T, VE> xp[VPT];
            load_row<T, TPR, VPT, VE>(x, row, cols, t, xp);
            TO* yr = y + row * cols;
            float mu = 0.f;
            float q[1] = {0.f};
            if constexpr (LN) {
                float s[1] = {0.f};
#pragma unroll
                for (int j = 0; j < VPT; ++j) s[0] += elem(xp[j], 0);
                group_sum<TPR, 1>(s, &red[group][0], phase, group);
                mu = s[0] * inv_cols;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (j * TPR + t < nvec) {
                        const float d = elem(xp[j], 0) - mu;
                        q[0] = fmaf(d, d, q[0]);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < VPT; ++j) q[0] = fmaf(elem(xp[j], 0), elem(xp[j], 0), q[0]);
            }
            group_sum<TPR, 1>(q, &red[group][0], phase, group);
            const float rs = rsqrtf(q[0] * inv_cols + a.eps);
            if (t == 0) {
                if (LN && a.mean) a.mean[row] = mu;
                if (a.rstd) a.rstd[row] = rs;
            }
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int vi = j * TPR + t;
                if (vi < nvec) {
                    float wv[1], bv[1], o[1];
                    load_param<T, 1>(a.w, vi, wv, 1.f);
                    load_param<T, 1>(a.b, vi, bv, 0.f);
                    o[0] = fmaf((elem(xp[j], 0) - mu) * rs, wv[0], bv[0]);
                    store_vec<TO, 1>(yr + vi, o);
                }
            }
        }
    }
}

// Writes the CTA's partial row: the sum over its RPC row groups (in group
// order) of each thread's per-column accumulators.  `part` holds
// [RPC][TPR*VE] floats when RPC > 1.  Called by all threads of the CTA.
template <int TPR, int VPT, int VE, int RPC>
__device__ __forceinline__ void write_partial_row(const float (&acc)[VPT][VE], float* ws,
                                                  float* part, int group, int t, int cols) {
    const int nvec = cols / VE;
    if constexpr (RPC == 1) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int vi = j * TPR + t;
            if (vi < nvec) {
#pragma unroll
                for (int k = 0; k < VE; ++k) ws[vi * VE + k] = acc[j][k];
            }
        }
    } else {
        constexpr int BLOCK = TPR * RPC;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (j * TPR * VE >= cols) break;
#pragma unroll
            for (int k = 0; k < VE; ++k) part[group * TPR * VE + t * VE + k] = acc[j][k];
            __syncthreads();
            for (int i = threadIdx.x; i < TPR * VE; i += BLOCK) {
                const int col = j * TPR * VE + i;
                if (col < cols) {
                    float sum = 0.f;
#pragma unroll
                    for (int g = 0; g < RPC; ++g) sum += part[g * TPR * VE + i];
                    ws[col] = sum;
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// backward, rows held in registers, next row prefetched; dw/db partials per CTA
// ---------------------------------------------------------------------------
// DB: accumulate db = sum dy (LayerNorm, or RMSNorm with a bias).
template <typename T, bool LN, int TPR, int VE, bool DB = LN>
__global__ void __launch_bounds__(kRowBwdBlock)
row_bwd_kernel(const RowArgs a) {
    constexpr int VPT = kRowBwdVpt;
    constexpr int BLOCK = kRowBwdBlock;
    constexpr int RPC = BLOCK / TPR;
    constexpr int NW = TPR / 32;
    constexpr int NV = LN ? 2 : 1;
    __shared__ float red[RPC][2 * NW * NV];
    __shared__ float part[RPC > 1 ? RPC : 1][RPC > 1 ? TPR * VE : 1];

    const int group = threadIdx.x / TPR;
    const int t = threadIdx.x % TPR;
    const int cols = a.cols;
    const int nvec = cols / VE;
    const float fcols = float(cols);
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const T* __restrict__ dy = reinterpret_cast<const T*>(a.dy);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    int phase = 0;

    float accw[VPT][VE];
    float accb[VPT][VE];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int k = 0; k < VE; ++k) accw[j][k] = accb[j][k] = 0.f;

    // weight for this thread's columns, read once
    float wv[VPT][VE];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int vi = j * TPR + t;
        if (vi < nvec) {
            load_param<T, VE>(a.w, vi, wv[j], 1.f);
        } else {
#pragma unroll
            for (int k = 0; k < VE; ++k) wv[j][k] = 0.f;
        }
    }

    const int64_t stride = int64_t(gridDim.x) * RPC;
    int64_t row = int64_t(blockIdx.x) * RPC + group;
    Pack<T, VE> xp[VPT], dp[VPT];
    if (row < a.rows) {
        load_row<T, TPR, VPT, VE>(x, row, cols, t, xp);
        load_row<T, TPR, VPT, VE>(dy, row, cols, t, dp);
    }
    for (; row < a.rows; row += stride) {
        // prefetch the next row of this group while this one is reduced
        Pack<T, VE> xn[VPT], dn[VPT];
        const int64_t nrow = row + stride;
        if (nrow < a.rows) {
            load_row<T, TPR, VPT, VE>(x, nrow, cols, t, xn);
            load_row<T, TPR, VPT, VE>(dy, nrow, cols, t, dn);
        }
        const float rs = a.rstd_in[row];
        const float mu = LN ? a.mean_in[row] : 0.f;

        float s[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) s[i] = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
#pragma unroll
            for (int k = 0; k < VE; ++k) {
                const float g = elem(dp[j], k) * wv[j][k];
                if constexpr (LN) {
                    const float xh = (elem(xp[j], k) - mu) * rs;
                    s[0] += g;
                    s[NV - 1] = fmaf(g, xh, s[NV - 1]);
                } else {
                    s[0] = fmaf(g, elem(xp[j], k), s[0]);
                }
            }
        }
        group_sum<TPR, NV>(s, &red[group][0], phase, group);

        T* dxr = dx + row * cols;
        const float c1 = s[0] / fcols;
        const float c2 = LN ? s[NV - 1] / fcols : c1 * rs * rs;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int vi = j * TPR + t;
            if (vi < nvec) {
                float o[VE];
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    const float xv = elem(xp[j], k);
                    const float dv = elem(dp[j], k);
                    const float g = dv * wv[j][k];
                    if constexpr (LN) {
                        const float xh = (xv - mu) * rs;
                        o[k] = rs * (g - c1 - xh * c2);
                        accw[j][k] = fmaf(dv, xh, accw[j][k]);
                        accb[j][k] += dv;
                    } else {
                        o[k] = rs * (g - xv * c2);
                        accw[j][k] = fmaf(dv, xv * rs, accw[j][k]);
                        if constexpr (DB) accb[j][k] += dv;
                    }
                }
                store_vec<T, VE>(dxr + int64_t(vi) * VE, o);
            }
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            xp[j] = xn[j];
            dp[j] = dn[j];
        }
    }

    // the column-sum kernel may be scheduled now; it waits for this grid
    pdl_trigger();

    // one partial row per CTA: fixed-order sum over the CTA's row groups
    if (a.ws_dw)
        write_partial_row<TPR, VPT, VE, RPC>(accw, a.ws_dw + int64_t(blockIdx.x) * cols, &part[0][0],
                                             group, t, cols);
    if constexpr (DB) {
        if (a.ws_db)
            write_partial_row<TPR, VPT, VE, RPC>(accb, a.ws_db + int64_t(blockIdx.x) * cols, &part[0][0],
                                                 group, t, cols);
    }
}

// Compensated fp32 sum (Neumaier's variant of Kahan's): exact to about two
// ulps of the result even when the terms are much larger than their sum.
struct NeumaierSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float v) {
        const float t = s + v;
        c += fabsf(s) >= fabsf(v) ? (s - t) + v : (v - t) + s;
        s = t;
    }
    __device__ __forceinline__ float value() const { return s + c; }
};

// dw/db[col] = sum over the P partial rows, in a fixed order, rounded to T.
// The partial rows can be much larger than their sum (dw of a column whose
// per-row terms cancel), so the sum is compensated.
constexpr int kColsumWarps = 32;  // partial rows are split over the warps: short dependent chains

template <typename T>
__global__ void __launch_bounds__(kColsumWarps * 32)
row_colsum_kernel(const float* __restrict__ ws_dw, const float* __restrict__ ws_db, int P,
                  int cols, T* dw, T* db) {
    pdl_wait();
    const float* ws = blockIdx.y == 0 ? ws_dw : ws_db;
    T* out = blockIdx.y == 0 ? dw : db;
    if (out == nullptr) return;
    __shared__ float part[kColsumWarps][2][33];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;
    NeumaierSum s;
    if (col < cols) {
#pragma unroll 4
        for (int p = warp; p < P; p += kColsumWarps) s.add(ws[int64_t(p) * cols + col]);
    }
    part[warp][0][lane] = s.s;
    part[warp][1][lane] = s.c;
    __syncthreads();
    if (warp == 0 && col < cols) {
        NeumaierSum tot;
#pragma unroll 8
        for (int w = 0; w < kColsumWarps; ++w) {
            tot.add(part[w][0][lane]);
            tot.add(part[w][1][lane]);
        }
        reinterpret_cast<typename Io<T>::bits_t*>(out)[col] = Io<T>::store(tot.value());
    }
}

// The same for a few partial rows (at most kColsumSerialMax): one thread per
// column adds its P values in order (Neumaier-compensated), 256 columns per CTA.
constexpr int kColsumSerialMax = 64;
constexpr int kColsumSerialBlock = 256;
template <typename T>
__global__ void __launch_bounds__(kColsumSerialBlock)
row_colsum_serial_kernel(const float* __restrict__ ws_dw, const float* __restrict__ ws_db, int P, int cols, T* dw,
                         T* db) {
    pdl_wait();
    const float* ws = blockIdx.y == 0 ? ws_dw : ws_db;
    T* out = blockIdx.y == 0 ? dw : db;
    const int col = blockIdx.x * kColsumSerialBlock + threadIdx.x;
    if (out == nullptr || col >= cols) return;
    NeumaierSum s;
#pragma unroll 8
    for (int p = 0; p < P; ++p) s.add(ws[int64_t(p) * cols + col]);
    reinterpret_cast<typename Io<T>::bits_t*>(out)[col] = Io<T>::store(s.value());
}

// ---------------------------------------------------------------------------
// wide rows: one CTA per row, two passes over global memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ Moments block_merge(Moments m, Moments* sm /* [33] */) {
    warp_merge(m);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (lane == 0) sm[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        Moments tot = sm[0];
        for (int w = 1; w < int(blockDim.x >> 5); ++w) chan_merge(tot, sm[w].n, sm[w].mean, sm[w].m2);
        sm[32] = tot;
    }
    __syncthreads();
    const Moments r = sm[32];
    __syncthreads();
    return r;
}

template <int NV>
__device__ __forceinline__ void block_sum(float (&v)[NV], float* sm /* [32*NV] */) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = warp_sum(v[k]);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < NV; ++k) sm[warp * NV + k] = v[k];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        float s = 0.f;
        for (int w = 0; w < int(blockDim.x >> 5); ++w) s += sm[w * NV + k];
        v[k] = s;
    }
    __syncthreads();
}

// VE fp32 values of type TD at p (fp32 values of a 16-bit VE-vector are two
// 16-byte vectors; p is 16-byte aligned when VE > 1), and the stores of them.
template <typename TD, int VE, bool STREAM = true>
__device__ __forceinline__ void load_as(const TD* p, float (&out)[VE]) {
    if constexpr (VE == 1 || VE == kVec<TD>) {
        load_vec<TD, VE, STREAM>(p, out);
    } else {
        static_assert(VE == 2 * kVec<TD>, "fp32 values of a 16-bit vector");
        constexpr int H = kVec<TD>;
        float lo[H], hi[H];
        load_vec<TD, H, STREAM>(p, lo);
        load_vec<TD, H, STREAM>(p + H, hi);
#pragma unroll
        for (int k = 0; k < H; ++k) {
            out[k] = lo[k];
            out[H + k] = hi[k];
        }
    }
}
template <typename TO, int VE>
__device__ __forceinline__ void store_as(TO* p, const float (&in)[VE]) {
    if constexpr (VE == 1 || VE == kVec<TO>) {
        store_vec<TO, VE>(p, in);
    } else {
        static_assert(VE == 2 * kVec<TO>, "fp32 values of a 16-bit vector");
        constexpr int H = kVec<TO>;
        float lo[H], hi[H];
#pragma unroll
        for (int k = 0; k < H; ++k) {
            lo[k] = in[k];
            hi[k] = in[H + k];
        }
        store_vec<TO, H>(p, lo);
        store_vec<TO, H>(p + H, hi);
    }
}

// 16-byte raw loads of VE elements of T (one or two 16-byte accesses), kept
// packed until they are used, so that several can be in flight per thread.
template <typename T, int VE>
struct RawVec {
    static constexpr int N = int(sizeof(T)) * VE / 16;
    uint4 u[N];
    __device__ __forceinline__ void load(const T* p) {
#pragma unroll
        for (int i = 0; i < N; ++i) u[i] = ld_stream_v4(p + i * (16 / int(sizeof(T))));
    }
    // with an L2 eviction policy
    __device__ __forceinline__ void load(const T* p, uint64_t pol) {
#pragma unroll
        for (int i = 0; i < N; ++i) u[i] = ld_v4_policy(p + i * (16 / int(sizeof(T))), pol);
    }
    __device__ __forceinline__ void unpack(float (&out)[VE]) const {
        constexpr int E = 16 / int(sizeof(T));
#pragma unroll
        for (int i = 0; i < N; ++i) {
            Pack<T, E> pk;
            pk.u = u[i];
#pragma unroll
            for (int k = 0; k < E; ++k) out[i * E + k] = Io<T>::load(pk.b[k]);
        }
    }
};
constexpr int kWideBatch = 4;  // 16-byte vectors per thread whose loads the wide kernels issue together
constexpr int kWideFwdBlock = 512;  // threads per CTA of the wide forward: 512 / 1024 measured 143 / 174 us (fp16 [2048,65536])

// TO: the output's storage type (T, or float for a 16-bit input whose output
// is kept in fp32).
template <typename T, bool LN, int VE, typename TO = T>
__global__ void __launch_bounds__(kRowWideBlock)
row_fwd_wide_kernel(const RowArgs a) {
    __shared__ Moments msm[33];
    __shared__ float ssm[32];
    const int cols = a.cols;
    const int nvec = cols / VE;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    TO* __restrict__ y = reinterpret_cast<TO*>(a.y);
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const T* xr = x + row * cols;
        float mu = 0.f, var;
        if constexpr (LN) {
            Moments m{0.f, 0.f, 0.f};
            auto add = [&](const float (&v)[VE]) {
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < VE; ++k) s += v[k];
                const float vm = s * (1.f / VE);
                float q = 0.f;
#pragma unroll
                for (int k = 0; k < VE; ++k) q = fmaf(v[k] - vm, v[k] - vm, q);
                chan_merge(m, float(VE), vm, q);
            };
            if constexpr (VE == kVec<T>) {
                // kWideBatch vectors' loads in flight per thread; the row stays in
                // L2 (evict_last) for the normalising pass
                const uint64_t keep = l2_evict_last();
                for (int v0 = threadIdx.x; v0 < nvec; v0 += kWideBatch * int(blockDim.x)) {
                    RawVec<T, VE> r[kWideBatch];
#pragma unroll
                    for (int u = 0; u < kWideBatch; ++u)
                        if (v0 + u * int(blockDim.x) < nvec)
                            r[u].load(xr + int64_t(v0 + u * int(blockDim.x)) * VE, keep);
#pragma unroll
                    for (int u = 0; u < kWideBatch; ++u) {
                        if (v0 + u * int(blockDim.x) < nvec) {
                            float v[VE];
                            r[u].unpack(v);
                            add(v);
                        }
                    }
                }
            } else {
                for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
                    float v[VE];
                    load_vec<T, VE, false>(xr + int64_t(vi) * VE, v);
                    add(v);
                }
            }
            const Moments tot = block_merge(m, msm);
            mu = tot.mean;
            var = tot.m2 / float(cols);
        } else {
            float s[1] = {0.f};
            for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
                float v[VE];
                load_vec<T, VE, false>(xr + int64_t(vi) * VE, v);
#pragma unroll
                for (int k = 0; k < VE; ++k) s[0] = fmaf(v[k], v[k], s[0]);
            }
            block_sum<1>(s, ssm);
            var = s[0] / float(cols);
        }
        const float rs = rsqrtf(var + a.eps);
        if (threadIdx.x == 0) {
            if (LN && a.mean) a.mean[row] = mu;
            if (a.rstd) a.rstd[row] = rs;
        }
        TO* yr = y + row * cols;
        auto out = [&](int vi, const float (&v)[VE]) {
            float wv[VE], bv[VE], o[VE];
            load_param<T, VE>(a.w, vi, wv, 1.f);
            load_param<T, VE>(a.b, vi, bv, 0.f);
#pragma unroll
            for (int k = 0; k < VE; ++k) {
                const float xh = (v[k] - mu) * rs;
                o[k] = fmaf(xh, wv[k], bv[k]);
            }
            store_as<TO, VE>(yr + int64_t(vi) * VE, o);
        };
        if constexpr (VE == kVec<T>) {
            const uint64_t drop = l2_evict_first();  // the row's last read
            for (int v0 = threadIdx.x; v0 < nvec; v0 += kWideBatch * int(blockDim.x)) {
                RawVec<T, VE> r[kWideBatch];
#pragma unroll
                for (int u = 0; u < kWideBatch; ++u)
                    if (v0 + u * int(blockDim.x) < nvec)
                        r[u].load(xr + int64_t(v0 + u * int(blockDim.x)) * VE, drop);
#pragma unroll
                for (int u = 0; u < kWideBatch; ++u) {
                    if (v0 + u * int(blockDim.x) < nvec) {
                        float v[VE];
                        r[u].unpack(v);
                        out(v0 + u * int(blockDim.x), v);
                    }
                }
            }
        } else {
            for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
                float v[VE];
                load_vec<T, VE>(xr + int64_t(vi) * VE, v);
                out(vi, v);
            }
        }
    }
}

// TD: the storage type of dy (T, or float when the forward's output was kept in fp32).
template <typename T, bool LN, int VE, typename TD = T>
__global__ void __launch_bounds__(kRowWideBlock)
row_bwd_wide_kernel(const RowArgs a) {
    __shared__ float ssm[32 * 2];
    const int cols = a.cols;
    const int nvec = cols / VE;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const TD* __restrict__ dy = reinterpret_cast<const TD*>(a.dy);
    T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
    float* wsw = a.ws_dw ? a.ws_dw + int64_t(blockIdx.x) * cols : nullptr;
    float* wsb = a.ws_db ? a.ws_db + int64_t(blockIdx.x) * cols : nullptr;
    // this CTA's partial rows; each column is always updated by the same thread.
    // When the row has at most one vector per thread the sums stay in registers
    // and are written once at the end; wider rows update the workspace row.
    const bool in_regs = nvec <= int(blockDim.x);
    float racc_w[VE], racc_b[VE];
#pragma unroll
    for (int k = 0; k < VE; ++k) racc_w[k] = racc_b[k] = 0.f;
    if (!in_regs) {
        for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
#pragma unroll
            for (int k = 0; k < VE; ++k) {
                if (wsw) wsw[vi * VE + k] = 0.f;
                if (wsb) wsb[vi * VE + k] = 0.f;
            }
        }
    }
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const T* xr = x + row * cols;
        const TD* dyr = dy + row * cols;
        const float rs = a.rstd_in[row];
        const float mu = LN ? a.mean_in[row] : 0.f;
        constexpr int NV = LN ? 2 : 1;
        float s[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) s[i] = 0.f;
        for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
            float xv[VE], dv[VE], wv[VE];
            load_vec<T, VE, false>(xr + int64_t(vi) * VE, xv);
            load_as<TD, VE, false>(dyr + int64_t(vi) * VE, dv);
            load_param<T, VE>(a.w, vi, wv, 1.f);
#pragma unroll
            for (int k = 0; k < VE; ++k) {
                const float g = dv[k] * wv[k];
                if constexpr (LN) {
                    s[0] += g;
                    s[NV - 1] = fmaf(g, (xv[k] - mu) * rs, s[NV - 1]);
                } else {
                    s[0] = fmaf(g, xv[k], s[0]);
                }
            }
        }
        block_sum<NV>(s, ssm);
        const float c1 = s[0] / float(cols);
        const float c2 = s[NV - 1] / float(cols);
        T* dxr = dx + row * cols;
        for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
            float xv[VE], dv[VE], wv[VE], o[VE], xs[VE];
            load_vec<T, VE>(xr + int64_t(vi) * VE, xv);
            load_as<TD, VE>(dyr + int64_t(vi) * VE, dv);
            load_param<T, VE>(a.w, vi, wv, 1.f);
#pragma unroll
            for (int k = 0; k < VE; ++k) {
                const float g = dv[k] * wv[k];
                xs[k] = LN ? (xv[k] - mu) * rs : xv[k] * rs;  // xhat (LN) or x*inv_rms
                if constexpr (LN) {
                    o[k] = rs * (g - c1 - xs[k] * c2);
                } else {
                    o[k] = rs * (g - xv[k] * (c1 * rs * rs));
                }
                if (in_regs) {
                    racc_w[k] = fmaf(dv[k], xs[k], racc_w[k]);
                    racc_b[k] += dv[k];
                }
            }
            if (!in_regs) {
                if constexpr (VE >= 4) {
                    // the partial rows by 16-byte accesses (the workspace and every
                    // CTA's row in it are 16-byte aligned; cols is a multiple of VE)
#pragma unroll
                    for (int h = 0; h < VE; h += 4) {
                        if (wsw) {
                            float4* p = reinterpret_cast<float4*>(wsw + vi * VE + h);
                            float4 u = *p;
                            u.x = fmaf(dv[h], xs[h], u.x);
                            u.y = fmaf(dv[h + 1], xs[h + 1], u.y);
                            u.z = fmaf(dv[h + 2], xs[h + 2], u.z);
                            u.w = fmaf(dv[h + 3], xs[h + 3], u.w);
                            *p = u;
                        }
                        if (wsb) {
                            float4* p = reinterpret_cast<float4*>(wsb + vi * VE + h);
                            float4 u = *p;
                            u.x += dv[h];
                            u.y += dv[h + 1];
                            u.z += dv[h + 2];
                            u.w += dv[h + 3];
                            *p = u;
                        }
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < VE; ++k) {
                        if (wsw) wsw[vi * VE + k] = fmaf(dv[k], xs[k], wsw[vi * VE + k]);
                        if (wsb) wsb[vi * VE + k] += dv[k];
                    }
                }
            }
            store_vec<T, VE>(dxr + int64_t(vi) * VE, o);
        }
    }
    if (in_regs && threadIdx.x < nvec) {
#pragma unroll
        for (int k = 0; k < VE; ++k) {
            if (wsw) wsw[threadIdx.x * VE + k] = racc_w[k];
            if (wsb) wsb[threadIdx.x * VE + k] = racc_b[k];
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// backward of rows too wide for the ring, in two kernels: the per-row sums,
// then a column pass in which each thread keeps its columns' dw/db sums in
// registers over a chunk of rows (one partial row per chunk, no
// read-modify-write of a workspace row per row)
// ---------------------------------------------------------------------------
constexpr int kWideColsBlock = 256;  // threads per CTA of the column pass
constexpr int kWideColsRows = 8;     // rows whose loads the column pass issues together

constexpr int kWideSumsBlock = 512;  // threads per CTA of the per-row sums (two CTAs share an SM)

// c[row] = (sum(g)/cols, sum(g*xhat)/cols) for LayerNorm, (sum(g*x)/cols, the
// same) for RMSNorm, g = dy*w: one CTA per row.
template <typename T, bool LN, int VE, typename TD = T>
__global__ void __launch_bounds__(kWideSumsBlock)
row_bwd_wide_sums_kernel(const RowArgs a, float2* __restrict__ c) {
    __shared__ float ssm[32 * 2];
    constexpr int NV = LN ? 2 : 1;
    constexpr int U = kWideBatch;
    const int cols = a.cols;
    const int nvec = cols / VE;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const TD* __restrict__ dy = reinterpret_cast<const TD*>(a.dy);
    const int bd = blockDim.x;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const T* xr = x + row * cols;
        const TD* dyr = dy + row * cols;
        const float rs = a.rstd_in[row];
        const float mu = LN ? a.mean_in[row] : 0.f;
        float s[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) s[i] = 0.f;
        for (int v0 = threadIdx.x; v0 < nvec; v0 += U * bd) {
            RawVec<T, VE> rx[U];
            RawVec<TD, VE> rd[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vi = v0 + u * bd;
                if (vi < nvec) {
                    rx[u].load(xr + int64_t(vi) * VE);
                    rd[u].load(dyr + int64_t(vi) * VE);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vi = v0 + u * bd;
                if (vi < nvec) {
                    float xv[VE], dv[VE], wv[VE];
                    rx[u].unpack(xv);
                    rd[u].unpack(dv);
                    load_param<T, VE>(a.w, vi, wv, 1.f);
#pragma unroll
                    for (int k = 0; k < VE; ++k) {
                        const float g = dv[k] * wv[k];
                        if constexpr (LN) {
                            s[0] += g;
                            s[NV - 1] = fmaf(g, (xv[k] - mu) * rs, s[NV - 1]);
                        } else {
                            s[0] = fmaf(g, xv[k], s[0]);
                        }
                    }
                }
            }
        }
        block_sum<NV>(s, ssm);
        if (threadIdx.x == 0) c[row] = make_float2(s[0] / float(cols), s[NV - 1] / float(cols));
    }
}

// dx for rows [blockIdx.y*rpc, +rpc) and this thread's column vector, and the
// chunk's partial dw/db row.
template <typename T, bool LN, int VE, typename TD = T>
__global__ void __launch_bounds__(kWideColsBlock)
row_bwd_wide_cols_kernel(const RowArgs a, const float2* __restrict__ c, int rpc) {
    // rows in flight: 8, or 4 when dy is fp32 (twice the raw bytes per row)
    constexpr int R = sizeof(TD) == sizeof(T) ? kWideColsRows : kWideColsRows / 2;
    const int cols = a.cols;
    const int nvec = cols / VE;
    const int vi = blockIdx.x * kWideColsBlock + threadIdx.x;
    if (vi < nvec) {
        const int64_t r0 = int64_t(blockIdx.y) * rpc;
        const int64_t r1 = a.rows - r0 < rpc ? a.rows : r0 + rpc;
        const T* __restrict__ x = reinterpret_cast<const T*>(a.x) + int64_t(vi) * VE;
        const TD* __restrict__ dy = reinterpret_cast<const TD*>(a.dy) + int64_t(vi) * VE;
        T* __restrict__ dx = reinterpret_cast<T*>(a.dx) + int64_t(vi) * VE;
        float wv[VE], accw[VE], accb[VE];
        load_param<T, VE>(a.w, vi, wv, 1.f);
#pragma unroll
        for (int k = 0; k < VE; ++k) accw[k] = accb[k] = 0.f;
        for (int64_t rb = r0; rb < r1; rb += R) {
            const int nr = r1 - rb < R ? int(r1 - rb) : R;
            // the rows' raw bytes, all loads in flight before the arithmetic
            RawVec<T, VE> rx[R];
            RawVec<TD, VE> rd[R];
#pragma unroll
            for (int u = 0; u < R; ++u) {
                if (u < nr) {
                    rx[u].load(x + (rb + u) * cols);
                    rd[u].load(dy + (rb + u) * cols);
                }
            }
#pragma unroll
            for (int u = 0; u < R; ++u) {
                if (u < nr) {
                    const int64_t r = rb + u;
                    const float rs = a.rstd_in[r];
                    const float mu = LN ? a.mean_in[r] : 0.f;
                    const float2 cc = c[r];
                    float xv[VE], dv[VE], o[VE];
                    rx[u].unpack(xv);
                    rd[u].unpack(dv);
#pragma unroll
                    for (int k = 0; k < VE; ++k) {
                        const float g = dv[k] * wv[k];
                        const float xs = LN ? (xv[k] - mu) * rs : xv[k] * rs;  // xhat or x*inv_rms
                        if constexpr (LN) {
                            o[k] = rs * (g - cc.x - xs * cc.y);
                        } else {
                            o[k] = rs * (g - xv[k] * (cc.x * rs * rs));
                        }
                        accw[k] = fmaf(dv[k], xs, accw[k]);
                        accb[k] += dv[k];
                    }
                    store_vec<T, VE>(dx + r * cols, o);
                }
            }
        }
        const int64_t off = int64_t(blockIdx.y) * cols + int64_t(vi) * VE;
#pragma unroll
        for (int k = 0; k < VE; ++k) {
            if (a.ws_dw) a.ws_dw[off + k] = accw[k];
            if (a.ws_db) a.ws_db[off + k] = accb[k];
        }
    }
    pdl_trigger();
}

constexpr uint64_t kRowWaitLimitNs = 2000000000ull;  // 2 s

}  // namespace nrm

#include "rowring.cuh"
#include "layernorm_cf.cuh"
#include "layernorm_cf_ring.cuh"

namespace nrm {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Plan of a backward ring kernel: TPR (rows of at most kRrVpt*512 vectors), R rows per
// chunk (a multiple of the row groups per CTA, about 48 KB per slot) and at
// least three slots where they fit.  False when the row does not suit.
inline bool rr_plan(RrGeom& g, int& tpr, size_t& smem, const RowArgs& a, size_t es, bool ln, size_t es_dy) {
    const DevInfo* d = dev_info();
    if (!d || a.rows <= 0) return false;
    const int nvec = int(size_t(a.cols) * es / 16);
    tpr = 32;
    while (tpr * kRrVpt < nvec && tpr < kRrMaxConsumers) tpr *= 2;
    if (tpr * kRrVpt < nvec) return false;
    const int rpc = rr_consumers(tpr) / tpr;
    const size_t row_bytes = size_t(a.cols) * (es + es_dy);  // a row of dy and a row of x
    const size_t param = (size_t(a.cols) * 4 + 127) / 128 * 128;
    const size_t cap = size_t(d->max_smem_optin) - 4096;  // room for the static shared memory
    if (param >= cap) return false;
    const size_t avail = cap - param;
    int m = int(49152 / (size_t(rpc) * row_bytes));
    if (m < 1) m = 1;
    size_t slot = 0;
    int slots = 0;
    for (;; --m) {
        const size_t R = size_t(m) * rpc;
        slot = (R * row_bytes + R * 4 * (ln ? 2 : 1) + 127) / 128 * 128;
        slots = int(avail / slot < size_t(kRrMaxSlots) ? avail / slot : size_t(kRrMaxSlots));
        if (slots >= 3 || m == 1) break;
    }
    if (slots < 2) return false;
    g.R = m * rpc;
    g.slots = slots;
    g.slot_bytes = uint32_t(slot);
    g.param_bytes = uint32_t(param);
    g.chunks = (a.rows + g.R - 1) / g.R;
    smem = param + size_t(slots) * slot;
    return true;
}

template <typename T, bool LN, bool DB, int VPT, typename TD>
const void* rr_fn_v(int tpr) {
    switch (tpr) {
    case 32: return (const void*)&row_bwd_ring_kernel<T, LN, 32, DB, VPT, TD>;
    case 64: return (const void*)&row_bwd_ring_kernel<T, LN, 64, DB, VPT, TD>;
    case 128: return (const void*)&row_bwd_ring_kernel<T, LN, 128, DB, VPT, TD>;
    case 256: return (const void*)&row_bwd_ring_kernel<T, LN, 256, DB, VPT, TD>;
    default: return (const void*)&row_bwd_ring_kernel<T, LN, 512, DB, VPT, TD>;
    }
}

// The ring kernel for rows of `nvec` vectors at TPR threads per row: 3
// vectors per thread when that covers the row, else 4.
template <typename T, bool LN, bool DB, typename TD = T>
const void* rr_fn(int tpr, int nvec) {
    return nvec <= 3 * tpr ? rr_fn_v<T, LN, DB, 3, TD>(tpr) : rr_fn_v<T, LN, DB, kRrVpt, TD>(tpr);
}

// Launches a ring kernel (row groups of `tpr` threads) on `grid` CTAs (one per SM at most).
inline nrm_status rr_launch(const void* fn, const RowArgs& a, const RrGeom& g, int tpr, size_t smem, int grid,
                            cudaStream_t s) {
    nrm_status st = prepare_kernel(fn, smem, false);
    if (st != NRM_OK) return st;
    RowArgs args = a;
    args.err = dev_info()->err;
    RrGeom geom = g;
    void* kargs[] = {&args, &geom};
    return cuda_status(cudaLaunchKernel(fn, dim3(grid), dim3(rr_threads(tpr)), kargs, smem, s), "row ring launch");
}

template <typename T, bool LN, int VE, int VPT, typename TO>
const void* row_fwd_fn_v(int tpr) {
    switch (tpr) {
    case 32: return (const void*)&row_fwd_kernel<T, LN, 32, VE, VPT, TO>;
    case 64: return (const void*)&row_fwd_kernel<T, LN, 64, VE, VPT, TO>;
    case 128: return (const void*)&row_fwd_kernel<T, LN, 128, VE, VPT, TO>;
    case 256: return (const void*)&row_fwd_kernel<T, LN, 256, VE, VPT, TO>;
    case 512: return (const void*)&row_fwd_kernel<T, LN, 512, VE, VPT, TO>;
    case 1024: return (const void*)&row_fwd_kernel<T, LN, 1024, VE, VPT, TO>;
    default: return (const void*)&row_fwd_wide_kernel<T, LN, VE, TO>;
    }
}

// The forward for rows of `nvec` vectors at TPR threads per row (0: the wide
// kernel): on the 16-byte path 3 vectors per thread when that covers the row
// (no idle fourth vector, e.g. 768 fp16 columns at 32 threads), else 4.
template <typename T, bool LN, int VE, typename TO = T>
const void* row_fwd_fn(int tpr, int nvec) {
    if constexpr (VE > 1) {
        if (tpr && nvec <= 3 * tpr) return row_fwd_fn_v<T, LN, VE, 3, TO>(tpr);
    }
    return row_fwd_fn_v<T, LN, VE, kRowFwdVpt, TO>(tpr);
}

template <typename T, bool LN, int VE>
const void* row_bwd_fn(int tpr, bool db) {
    if (!LN && db) {
        switch (tpr) {  // RMSNorm with a bias
        case 32: return (const void*)&row_bwd_kernel<T, LN, 32, VE, true>;
        case 64: return (const void*)&row_bwd_kernel<T, LN, 64, VE, true>;
        case 128: return (const void*)&row_bwd_kernel<T, LN, 128, VE, true>;
        case 256: return (const void*)&row_bwd_kernel<T, LN, 256, VE, true>;
        case 512: return (const void*)&row_bwd_kernel<T, LN, 512, VE, true>;
        default: return (const void*)&row_bwd_wide_kernel<T, LN, VE>;
        }
    }
    switch (tpr) {
    case 32: return (const void*)&row_bwd_kernel<T, LN, 32, VE>;
    case 64: return (const void*)&row_bwd_kernel<T, LN, 64, VE>;
    case 128: return (const void*)&row_bwd_kernel<T, LN, 128, VE>;
    case 256: return (const void*)&row_bwd_kernel<T, LN, 256, VE>;
    case 512: return (const void*)&row_bwd_kernel<T, LN, 512, VE>;
    default: return (const void*)&row_bwd_wide_kernel<T, LN, VE>;
    }
}

// Threads per row group: the smallest power of two >= 32 holding the row in
// `vpt` vectors per thread, or 0 for the wide-row kernel.
inline int row_tpr(int nvec, int vpt, int max_tpr) {
    int tpr = 32;
    while (tpr * vpt < nvec && tpr < max_tpr) tpr *= 2;
    return tpr * vpt < nvec ? 0 : tpr;
}

// The forward with output storage type TO (T, or float for a 16-bit T).
template <typename T, typename TO>
nrm_status row_fwd_to(const RowArgs& a, bool layernorm, bool vec, cudaStream_t s) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    if (a.rows == 0) return NRM_OK;
    const int ve = vec ? kVec<T> : 1;
    const int tpr = row_tpr(a.cols / ve, kRowFwdVpt, kRowMaxFwdTpr);
    const int nvec = a.cols / ve;
    const void* fn = layernorm ? (vec ? row_fwd_fn<T, true, kVec<T>, TO>(tpr, nvec)
                                      : row_fwd_fn<T, true, 1, TO>(tpr, nvec))
                               : (vec ? row_fwd_fn<T, false, kVec<T>, TO>(tpr, nvec)
                                      : row_fwd_fn<T, false, 1, TO>(tpr, nvec));
    const int block = tpr ? row_fwd_block(tpr) : kWideFwdBlock;
    const int rpc = tpr ? block / tpr : 1;
    const int occ = cached_occupancy(fn, block, 0);
    if (occ <= 0) return fail(NRM_ERR_CUDA, "row forward kernel cannot be resident");
    const int64_t groups = (a.rows + rpc - 1) / rpc;
    const int grid = int(groups < int64_t(occ) * d->sms ? groups : int64_t(occ) * d->sms);
    RowArgs args = a;
    void* kargs[] = {&args};
    return cuda_status(cudaLaunchKernel(fn, dim3(grid), dim3(block), kargs, 0, s), "row forward launch");
}

template <typename T>
nrm_status row_fwd(const RowArgs& a, bool layernorm, bool vec, cudaStream_t s) {
    return row_fwd_to<T, T>(a, layernorm, vec, s);
}

// The fixed-order column sums of P partial dw/db rows (programmatic dependent
// launch after the kernel that wrote them).
template <typename T>
nrm_status row_colsum_launch(const RowArgs& a, int P, cudaStream_t s) {
    const float* wsw = a.ws_dw;
    const float* wsb = a.ws_db;
    int P_ = P;
    int cols = a.cols;
    T* dw = reinterpret_cast<T*>(a.dw);
    T* db = reinterpret_cast<T*>(a.db);
    void* cargs[] = {&wsw, &wsb, &P_, &cols, &dw, &db};
    if (P <= kColsumSerialMax)
        return launch_pdl((const void*)&row_colsum_serial_kernel<T>,
                          dim3((a.cols + kColsumSerialBlock - 1) / kColsumSerialBlock, 2), dim3(kColsumSerialBlock),
                          cargs, s);
    return launch_pdl((const void*)&row_colsum_kernel<T>, dim3((a.cols + 31) / 32, 2), dim3(kColsumWarps * 32),
                      cargs, s);
}

// Threads per CTA of a wide-row kernel used for rows of `nvec` vectors: a
// warp multiple that covers the row, at most kRowWideBlock.
inline int wide_block(int nvec) {
    int b = (nvec + 31) / 32 * 32;
    return b < 32 ? 32 : (b > kRowWideBlock ? kRowWideBlock : b);
}

// The wide-row backward in two kernels (per-row sums, then the column pass)
// for 16-byte vectors.  The per-row sums take 2*rows floats of the dw
// workspace after the chunks' partial rows; returns the chunk count (the
// partial rows for the column sums), or 0 when the workspace has no room for
// them (the one-kernel wide path runs instead).
template <typename T, typename TD>
int row_bwd_wide_split(const RowArgs& a, float* ws0, bool layernorm, cudaStream_t s, nrm_status& st) {
    constexpr int VE = kVec<T>;
    const DevInfo* d = dev_info();
    st = NRM_OK;
    if (!d || !ws0 || a.rows <= 0) return 0;
    const int nvec = a.cols / VE;
    const int slabs = (nvec + kWideColsBlock - 1) / kWideColsBlock;
    int64_t cap = row_bwd_max_partials(*d);
    if (a.max_partials > 0 && cap > a.max_partials) cap = a.max_partials;
    const int64_t c_rows = (2 * a.rows + a.cols - 1) / a.cols;  // workspace rows the sums take
    int64_t rc = (int64_t(4) * d->sms + slabs - 1) / slabs;   // about four CTAs per SM
    if (rc > a.rows) rc = a.rows;
    if (rc > cap - c_rows) rc = cap - c_rows;
    if (rc < 1) return 0;
    const int rpc = int((a.rows + rc - 1) / rc);
    rc = (a.rows + rpc - 1) / rpc;
    float2* c = reinterpret_cast<float2*>(ws0 + size_t(rc) * size_t(a.cols));
    const void* sums = layernorm ? (const void*)&row_bwd_wide_sums_kernel<T, true, VE, TD>
                                 : (const void*)&row_bwd_wide_sums_kernel<T, false, VE, TD>;
    const void* colk = layernorm ? (const void*)&row_bwd_wide_cols_kernel<T, true, VE, TD>
                                 : (const void*)&row_bwd_wide_cols_kernel<T, false, VE, TD>;
    const int block = kWideSumsBlock;
    const int occ = cached_occupancy(sums, block, 0);
    if (occ <= 0) {
        st = fail(NRM_ERR_CUDA, "row backward (sums) kernel cannot be resident");
        return 0;
    }
    const int64_t g1 = a.rows < int64_t(occ) * d->sms ? a.rows : int64_t(occ) * d->sms;
    RowArgs args = a;
    void* k1[] = {&args, &c};
    st = cuda_status(cudaLaunchKernel(sums, dim3(unsigned(g1)), dim3(block), k1, 0, s), "row backward (sums) launch");
    if (st != NRM_OK) return 0;
    const float2* cc = c;
    int rpc_ = rpc;
    void* k2[] = {&args, &cc, &rpc_};
    st = cuda_status(cudaLaunchKernel(colk, dim3(unsigned(slabs), unsigned(rc)), dim3(kWideColsBlock), k2, 0, s),
                     "row backward (columns) launch");
    return st == NRM_OK ? int(rc) : 0;
}

template <typename T>
nrm_status row_bwd(RowArgs a, bool layernorm, bool vec, cudaStream_t s) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    const bool want = a.dw || a.db;
    float* const ws0 = a.ws_dw;
    if (!want) a.ws_dw = a.ws_db = nullptr;
    const int ve = vec ? kVec<T> : 1;
    RrGeom rg;
    int rtpr = 0;
    size_t rsmem = 0;
    const bool ring = vec && rr_plan(rg, rtpr, rsmem, a, sizeof(T), layernorm, sizeof(T));
    const int tpr = ring ? 0 : row_tpr(a.cols / ve, kRowBwdVpt, kRowMaxBwdTpr);
    const void* fn;
    int64_t groups, p;
    int block = 0;
    if (ring) {
        const int nv = a.cols / kVec<T>;
        fn = layernorm ? rr_fn<T, true, true>(rtpr, nv)
                       : (a.ws_db ? rr_fn<T, false, true>(rtpr, nv) : rr_fn<T, false, false>(rtpr, nv));
        groups = rg.chunks;
        p = d->sms;
    } else {
        if (tpr == 0 && vec) {
            nrm_status st = NRM_OK;
            const int rc = row_bwd_wide_split<T, T>(a, ws0, layernorm, s, st);
            if (st != NRM_OK) return st;
            if (rc > 0) return want ? row_colsum_launch<T>(a, rc, s) : NRM_OK;
        }
        const bool db = a.ws_db != nullptr;
        fn = layernorm ? (vec ? row_bwd_fn<T, true, kVec<T>>(tpr, db) : row_bwd_fn<T, true, 1>(tpr, db))
                       : (vec ? row_bwd_fn<T, false, kVec<T>>(tpr, db) : row_bwd_fn<T, false, 1>(tpr, db));
        block = tpr ? kRowBwdBlock : kRowWideBlock;
        const int rpc = tpr ? block / tpr : 1;
        const int occ = cached_occupancy(fn, block, 0);
        if (occ <= 0) return fail(NRM_ERR_CUDA, "row backward kernel cannot be resident");
        groups = (a.rows + rpc - 1) / rpc;
        p = int64_t(occ) * d->sms;
    }
    if (p > row_bwd_max_partials(*d)) p = row_bwd_max_partials(*d);
    if (a.max_partials > 0 && p > a.max_partials) p = a.max_partials;
    if (groups < p) p = groups;
    const int P = int(p);
    if (ring && P > 0) {
        nrm_status st = rr_launch(fn, a, rg, rtpr, rsmem, P, s);
        if (st != NRM_OK) return st;
    } else if (P > 0) {
        RowArgs args = a;
        void* kargs[] = {&args};
        nrm_status st = cuda_status(cudaLaunchKernel(fn, dim3(P), dim3(block), kargs, 0, s),
                                    "row backward launch");
        if (st != NRM_OK) return st;
    }
    if (!want) return NRM_OK;
    const float* wsw = a.ws_dw;
    const float* wsb = a.ws_db;
    int P_ = P;
    int cols = a.cols;
    T* dw = reinterpret_cast<T*>(a.dw);
    T* db = reinterpret_cast<T*>(a.db);
    void* cargs[] = {&wsw, &wsb, &P_, &cols, &dw, &db};
    return launch_pdl((const void*)&row_colsum_kernel<T>, dim3((a.cols + 31) / 32, 2), dim3(kColsumWarps * 32),
                      cargs, s);
}


// Forward with the output kept in fp32 for a 16-bit input: the same kernels
// as the plain forward, storing float32 (two 16-byte stores per input vector).
template <typename T>
nrm_status row_fwd_f32out(const RowArgs& a, bool layernorm, bool vec, cudaStream_t s) {
    return row_fwd_to<T, float>(a, layernorm, vec, s);
}

// Backward whose dy is fp32 (the forward kept its output in fp32) for a
// 16-bit x: the wide-row kernels with TD = float, then the column sums.
template <typename T>
nrm_status row_bwd_f32dy(RowArgs a, bool layernorm, bool vec, cudaStream_t s) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    const bool want = a.dw || a.db;
    float* const ws0 = a.ws_dw;
    if (!want) a.ws_dw = a.ws_db = nullptr;
    constexpr int V = kVec<T>;
    RrGeom rg;
    int rtpr = 0;
    size_t rsmem = 0;
    int P = 0;
    bool ring = false;
    if constexpr (sizeof(T) == 2) {
        // dy rows as float32 in the ring slots beside x
        ring = vec && rr_plan(rg, rtpr, rsmem, a, sizeof(T), layernorm, sizeof(float));
        if (ring) {
            const int nv = a.cols / V;
            const void* fn = layernorm ? rr_fn<T, true, true, float>(rtpr, nv)
                                       : (a.ws_db ? rr_fn<T, false, true, float>(rtpr, nv)
                                                  : rr_fn<T, false, false, float>(rtpr, nv));
            int64_t p = d->sms;
            if (p > row_bwd_max_partials(*d)) p = row_bwd_max_partials(*d);
            if (rg.chunks < p) p = rg.chunks;
            P = int(p);
            if (P > 0) {
                nrm_status st = rr_launch(fn, a, rg, rtpr, rsmem, P, s);
                if (st != NRM_OK) return st;
            }
        }
    }
    if (!ring && vec && sizeof(T) == 2) {
        nrm_status st = NRM_OK;
        const int rc = row_bwd_wide_split<T, float>(a, ws0, layernorm, s, st);
        if (st != NRM_OK) return st;
        if (rc > 0) return want ? row_colsum_launch<T>(a, rc, s) : NRM_OK;
    }
    if (!ring) {
        const void* fn = layernorm ? (vec ? (const void*)&row_bwd_wide_kernel<T, true, V, float>
                                          : (const void*)&row_bwd_wide_kernel<T, true, 1, float>)
                                   : (vec ? (const void*)&row_bwd_wide_kernel<T, false, V, float>
                                          : (const void*)&row_bwd_wide_kernel<T, false, 1, float>);
        const int block = wide_block(a.cols / (vec ? V : 1));
        const int occ = cached_occupancy(fn, block, 0);
        if (occ <= 0) return fail(NRM_ERR_CUDA, "row backward kernel cannot be resident");
        int64_t p = int64_t(occ) * d->sms;
        if (p > row_bwd_max_partials(*d)) p = row_bwd_max_partials(*d);
        if (a.rows < p) p = a.rows;
        P = int(p);
        if (P > 0) {
            RowArgs args = a;
            void* kargs[] = {&args};
            nrm_status st = cuda_status(cudaLaunchKernel(fn, dim3(P), dim3(block), kargs, 0, s), "row backward launch");
            if (st != NRM_OK) return st;
        }
    }
    if (!want) return NRM_OK;
    const float* wsw = a.ws_dw;
    const float* wsb = a.ws_db;
    int P_ = P;
    int cols = a.cols;
    T* dw = reinterpret_cast<T*>(a.dw);
    T* db = reinterpret_cast<T*>(a.db);
    void* cargs[] = {&wsw, &wsb, &P_, &cols, &dw, &db};
    return launch_pdl((const void*)&row_colsum_kernel<T>, dim3((a.cols + 31) / 32, 2), dim3(kColsumWarps * 32),
                      cargs, s);
}

// Plan of a channels-first ring kernel: positions per tile (the widest of 32,
// 16, 8 vectors per channel row that the plane needs and that leaves at least
// four slots, else three, else two), channel boxes of at most 256 rows, and
// the shared-memory layout.  False when a tile does not fit (the register kernel runs instead).
inline bool cfr_plan(CfrGeom& g, size_t& smem, const CfArgs& a, size_t es, bool bwd) {
    const DevInfo* d = dev_info();
    if (!d || a.n <= 0 || a.l <= 0 || a.c > 4096) return false;
    if (a.l >= (int64_t(1) << 31) || a.n >= (int64_t(1) << 31)) return false;
    const int V = int(16 / es);
    const auto r128 = [](size_t b) { return (b + 127) / 128 * 128; };
    const size_t param = r128(size_t(a.c) * 4 * (bwd ? 1 : 2));
    const size_t acc = bwd ? r128(size_t(a.c) * 4 * 2 * kCfrTeams) : 0;
    const size_t cap = size_t(d->max_smem_optin) - 1024;  // room for the static shared memory
    const int nb = int((a.c + 255) / 256);
    const int cb = int((a.c + nb - 1) / nb);
    int pv = 8;
    while (pv < 32 && int64_t(pv) * V < a.l) pv *= 2;
    bool found = false;
    // two tiles are being consumed at a time (one per team): four slots keep two loading
    for (int want = 4; want >= 2 && !found; want -= 2) {
        for (int p = pv; p >= 8; p /= 2) {
            const int P = p * V;
            const size_t part = r128((size_t(kCfrTeams) * kCfrTeamFloatsPerPos * P + 2 * kCfrTeamWarps) * 4);
            const size_t tensor = size_t(nb) * cb * P * es;
            const size_t slot = r128(tensor * (bwd ? 2 : 1) + (bwd ? size_t(2) * P * 4 : 0));
            if (param + part + acc >= cap) continue;
            // an even number of slots: the tile that used a slot before tile q is then
            // q - slots, which the same team consumed (so it has landed).  With an odd
            // count it belongs to the other team and may still be in flight, and a wait
            // on the slot's barrier for tile q (parity of phase q / slots) would see the
            // phase before it pending and return at once.
            size_t n_slots = (cap - param - part - acc) / slot;
            if (n_slots > size_t(kCfrMaxSlots)) n_slots = kCfrMaxSlots;
            n_slots &= ~size_t(1);
            if (n_slots < size_t(want)) continue;
            g.pv = p;
            g.P = P;
            g.cb = cb;
            g.nb = nb;
            g.slots = int(n_slots);
            g.slot_bytes = uint32_t(slot);
            g.tx_tensor = uint32_t(tensor);
            g.param_bytes = uint32_t(param);
            g.part_bytes = uint32_t(part);
            g.acc_bytes = uint32_t(acc);
            smem = param + part + acc + size_t(g.slots) * slot;
            found = true;
            break;
        }
    }
    if (!found) return false;
    g.tps = (a.l + g.P - 1) / g.P;
    g.tiles = a.n * g.tps;
    return true;
}

// Position groups per lane of the scalar register kernels: the fewest of 1, 2,
// 4, 8 (32 positions each) that cover a plane of l positions.
inline int cf_scalar_groups(int64_t l) { return l <= 32 ? 1 : (l <= 64 ? 2 : (l <= 128 ? 4 : 8)); }
template <typename T, bool BWD>
const void* cf_scalar_fn(int K) {
    switch (K) {
    case 1: return BWD ? (const void*)&lncf_bwd_kernel<T, 1, 1> : (const void*)&lncf_fwd_kernel<T, 1, 1>;
    case 2: return BWD ? (const void*)&lncf_bwd_kernel<T, 1, 2> : (const void*)&lncf_fwd_kernel<T, 1, 2>;
    case 4: return BWD ? (const void*)&lncf_bwd_kernel<T, 1, 4> : (const void*)&lncf_fwd_kernel<T, 1, 4>;
    default: return BWD ? (const void*)&lncf_bwd_kernel<T, 1, 8> : (const void*)&lncf_fwd_kernel<T, 1, 8>;
    }
}

template <typename T>
nrm_status cf_fwd(const CfArgs& a, bool vec, cudaStream_t s) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    if (a.n == 0 || a.l == 0) return NRM_OK;
    CfrGeom g{};
    size_t smem = 0;
    if (vec && cfr_plan(g, smem, a, sizeof(T), false)) {
        alignas(64) CUtensorMap map_x;
        nrm_status st = encode_ncl_map(&map_x, a.x, sizeof(T), a.n, a.c, a.l, g.P, g.cb);
        if (st != NRM_OK) return st;
        const void* fn = (const void*)&lncf_fwd_ring_kernel<T>;
        if ((st = prepare_kernel(fn, smem, false)) != NRM_OK) return st;
        CfArgs args = a;
        args.err = d->err;
        const int grid = int(g.tiles < d->sms ? g.tiles : d->sms);
        void* kargs[] = {&args, &g, &map_x};
        return cuda_status(cudaLaunchKernel(fn, dim3(grid), dim3(kCfrThreads), kargs, smem, s),
                           "channels-first LayerNorm forward launch");
    }
    // groups only where they fold a mostly idle second tile into the first
    // (planes of up to 64 positions): the forward has no per-channel warp
    // reductions to save, and fewer tiles are fewer CTAs (fp16 [256,384,14,14]:
    // 51 us with 32-position tiles, 62 with one 256-position tile per plane)
    const int K = vec ? 1 : (a.l <= 64 ? cf_scalar_groups(a.l) : 1);
    const void* fn = vec ? (const void*)&lncf_fwd_kernel<T, kVec<T>> : cf_scalar_fn<T, false>(K);
    const int pw = 32 * (vec ? kVec<T> : K);
    const int64_t tiles = a.n * ((a.l + pw - 1) / pw);
    const int occ = cached_occupancy(fn, kCfThreads, 0);
    if (occ <= 0) return fail(NRM_ERR_CUDA, "channels-first LayerNorm forward cannot be resident");
    const int64_t cap = int64_t(occ) * d->sms;
    const int grid = int(tiles < cap ? tiles : cap);
    CfArgs args = a;
    void* kargs[] = {&args};
    return cuda_status(cudaLaunchKernel(fn, dim3(grid), dim3(kCfThreads), kargs, 0, s),
                       "channels-first LayerNorm forward launch");
}

template <typename T>
nrm_status cf_bwd(CfArgs a, bool vec, cudaStream_t s) {
    const DevInfo* d = dev_info();
    if (!d) return fail(NRM_ERR_CUDA, "no usable CUDA device");
    const bool want = a.dw || a.db;
    if (!want) a.ws_dw = a.ws_db = nullptr;
    if (a.n == 0 || a.l == 0) {
        if (!want) return NRM_OK;
        // no positions: dw = db = 0 (the column sum over zero partial rows)
        const float* none = nullptr;
        int P0 = 0;
        int cols = int(a.c);
        T* dw = reinterpret_cast<T*>(a.dw);
        T* db = reinterpret_cast<T*>(a.db);
        void* cargs[] = {&none, &none, &P0, &cols, &dw, &db};
        return launch_pdl((const void*)&row_colsum_kernel<T>, dim3((cols + 31) / 32, 2),
                          dim3(kColsumWarps * 32), cargs, s);
    }
    CfrGeom g{};
    size_t rsmem = 0;
    const bool stats16 = ((reinterpret_cast<uintptr_t>(a.mean_in) | reinterpret_cast<uintptr_t>(a.rstd_in)) & 15) == 0;
    if (vec && stats16 && cfr_plan(g, rsmem, a, sizeof(T), true)) {
        alignas(64) CUtensorMap map_dy;
        alignas(64) CUtensorMap map_x;
        nrm_status st = encode_ncl_map(&map_dy, a.dy, sizeof(T), a.n, a.c, a.l, g.P, g.cb);
        if (st == NRM_OK) st = encode_ncl_map(&map_x, a.x, sizeof(T), a.n, a.c, a.l, g.P, g.cb);
        if (st != NRM_OK) return st;
        const void* fn = (const void*)&lncf_bwd_ring_kernel<T>;
        if ((st = prepare_kernel(fn, rsmem, false)) != NRM_OK) return st;
        CfArgs args = a;
        args.err = d->err;
        const int grid = int(g.tiles < d->sms ? g.tiles : d->sms);
        void* kargs[] = {&args, &g, &map_dy, &map_x};
        st = cuda_status(cudaLaunchKernel(fn, dim3(grid), dim3(kCfrThreads), kargs, rsmem, s),
                         "channels-first LayerNorm backward launch");
        if (st != NRM_OK || !want) return st;
        const float* wsw = a.ws_dw;
        const float* wsb = a.ws_db;
        int P_ = grid;
        int cols = int(a.c);
        T* dw = reinterpret_cast<T*>(a.dw);
        T* db = reinterpret_cast<T*>(a.db);
        void* cargs[] = {&wsw, &wsb, &P_, &cols, &dw, &db};
        return launch_pdl((const void*)&row_colsum_kernel<T>, dim3((cols + 31) / 32, 2),
                          dim3(kColsumWarps * 32), cargs, s);
    }
    // one dw/db warp reduction per channel and tile: a plane in one tile where
    // it fits 256 positions (fp16 [256,384,14,14] 158 -> 127 us, [2048,768,7,7]
    // 676 -> 545 us)
    const int K = vec ? 1 : cf_scalar_groups(a.l);
    const void* fn = vec ? (const void*)&lncf_bwd_kernel<T, kVec<T>> : cf_scalar_fn<T, true>(K);
    const int pw = 32 * (vec ? kVec<T> : K);
    const int64_t tiles = a.n * ((a.l + pw - 1) / pw);
    // the CTA's dw, db partial row
    const size_t smem = size_t(a.c) * 2 * sizeof(float);
    nrm_status st = prepare_kernel(fn, smem, false);
    if (st != NRM_OK) return st;
    const int occ = cached_occupancy(fn, kCfThreads, smem);
    if (occ <= 0) return fail(NRM_ERR_CUDA, "channels-first LayerNorm backward cannot be resident");
    int64_t p = int64_t(occ) * d->sms;
    if (p > row_bwd_max_partials(*d)) p = row_bwd_max_partials(*d);
    if (tiles < p) p = tiles;
    const int P = int(p);
    CfArgs args = a;
    void* kargs[] = {&args};
    st = cuda_status(cudaLaunchKernel(fn, dim3(P), dim3(kCfThreads), kargs, smem, s),
                     "channels-first LayerNorm backward launch");
    if (st != NRM_OK || !want) return st;
    const float* wsw = a.ws_dw;
    const float* wsb = a.ws_db;
    int P_ = P;
    int cols = int(a.c);
    T* dw = reinterpret_cast<T*>(a.dw);
    T* db = reinterpret_cast<T*>(a.db);
    void* cargs[] = {&wsw, &wsb, &P_, &cols, &dw, &db};
    return launch_pdl((const void*)&row_colsum_kernel<T>, dim3((cols + 31) / 32, 2), dim3(kColsumWarps * 32),
                      cargs, s);
}

}  // namespace nrm

#define NRM_INSTANTIATE_ROWNORM(T)                                                      \
    template nrm_status nrm::row_fwd<T>(const nrm::RowArgs&, bool, bool, cudaStream_t); \
    template nrm_status nrm::row_bwd<T>(nrm::RowArgs, bool, bool, cudaStream_t);        \
    template nrm_status nrm::row_fwd_f32out<T>(const nrm::RowArgs&, bool, bool, cudaStream_t); \
    template nrm_status nrm::row_bwd_f32dy<T>(nrm::RowArgs, bool, bool, cudaStream_t);  \
    template nrm_status nrm::cf_fwd<T>(const nrm::CfArgs&, bool, cudaStream_t);         \
    template nrm_status nrm::cf_bwd<T>(nrm::CfArgs, bool, cudaStream_t);
