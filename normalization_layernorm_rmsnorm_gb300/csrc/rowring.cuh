// rowring.cuh -- LayerNorm and RMSNorm backward for rows that are 16-byte
// aligned and at most 2048 vectors long, with the rows streamed through shared
// memory (included by rownorm.cuh; computes what that file states).
//
// Rows of a [rows, cols] tensor are contiguous, so a chunk of R rows is one
// bulk copy per tensor.  A producer warp streams the CTA's chunks of dy and x
// (CTA b takes chunks b, b + grid, ...) through a ring of shared-memory slots;
// the rows' rstd and mean ride along as 4-byte async copies.  16 consumer
// warps process the rows in groups of TPR threads (vector j*TPR + t of a row
// belongs to thread t of its group): the row sums from the slot, then dx from
// a second read of the slot, stored with 16-byte stores, and dw/db
// accumulated per thread in fp32; the element arithmetic runs on fp32 pairs
// with the packed FP32 instructions.  The weight is converted to fp32 once per
// CTA and kept in shared memory.  Memory parallelism comes from the ring
// (several chunks in flight per SM), not from registers.  (The forward keeps
// the register kernel: its rows need one read, and many resident CTAs hide
// its reduction latency better than one ring CTA per SM.)
#pragma once

namespace nrm {

// Consumer warps per CTA.  One-warp rows (TPR 32) take 15, so that the CTA
// with its producer warp has 16 warps: 4 per SM sub-partition, and 128
// registers per thread, enough to keep the thread's columns of the weight in
// registers (a 17th warp would leave 96).  Wider rows take 16, a multiple of
// their row groups.
__host__ __device__ constexpr int rr_consumer_warps(int tpr) { return tpr == 32 ? 15 : 16; }
__host__ __device__ constexpr int rr_consumers(int tpr) { return rr_consumer_warps(tpr) * 32; }
__host__ __device__ constexpr int rr_threads(int tpr) { return rr_consumers(tpr) + 32; }  // + the producer warp
constexpr int kRrMaxConsumers = 16 * 32;
constexpr int kRrVpt = 4;                      // 16-byte vectors per thread and row, at most
constexpr int kRrMaxSlots = 8;
constexpr int kRrBarConsumers = 15;            // named barrier over the consumer warps

struct RrGeom {
    int R;                 // rows per chunk
    int slots;             // ring slots
    uint32_t slot_bytes;   // bytes of a slot: R rows of dy, R rows of x, R floats of rstd (and of mean)
    uint32_t param_bytes;  // fp32 weight (and bias) at the front of dynamic shared memory
    int64_t chunks;        // ceil(rows / R)
};

// Producer (whole warp): the CTA's chunks of dy (storage type TD) and x (T)
// (and the rows' rstd, mean) into the ring, in order.  If a wait for a free
// slot gives up, it issues nothing more; either way it then waits (bounded)
// until the last copy issued into each slot has landed, so that none is in
// flight at exit.
template <typename T, bool LN, typename TD>
__device__ void rr_produce(const RowArgs& a, const RrGeom& g, unsigned char* ring, uint64_t* full,
                           uint64_t* empty, int lane, bool& bad) {
    const size_t row_bytes = size_t(a.cols) * sizeof(T);
    const size_t dy_row_bytes = size_t(a.cols) * sizeof(TD);
    const uint64_t pol = l2_evict_first();
    int q = 0;
    for (int64_t c = blockIdx.x; c < g.chunks; c += gridDim.x, ++q) {
        const int slot = q % g.slots;
        const uint32_t use = uint32_t(q / g.slots);
        if (use > 0 && !__all_sync(0xffffffffu, mbar_wait_bounded(&empty[slot], (use - 1) & 1u, kRowWaitLimitNs))) {
            bad = true;
            break;
        }
        const int64_t r0 = c * g.R;
        const int ra = int(a.rows - r0 < g.R ? a.rows - r0 : g.R);
        unsigned char* base = ring + size_t(slot) * g.slot_bytes;
        const uint32_t bytes = uint32_t(size_t(ra) * row_bytes);
        const uint32_t dy_bytes = uint32_t(size_t(ra) * dy_row_bytes);
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[slot], dy_bytes + bytes);
            bulk_g2s(base, reinterpret_cast<const TD*>(a.dy) + r0 * a.cols, dy_bytes, &full[slot], pol);
            bulk_g2s(base + size_t(g.R) * dy_row_bytes, reinterpret_cast<const T*>(a.x) + r0 * a.cols, bytes,
                     &full[slot], pol);
        }
        float* st = reinterpret_cast<float*>(base + size_t(g.R) * (dy_row_bytes + row_bytes));
        for (int i = lane; i < ra; i += 32) {
            cp_async_4(st + i, a.rstd_in + r0 + i);
            if (LN) cp_async_4(st + g.R + i, a.mean_in + r0 + i);
        }
        cp_async_mbar_arrive_noinc(&full[slot]);
    }
    for (int s = 0; s < g.slots && s < q; ++s) {
        const int last = s + ((q - 1 - s) / g.slots) * g.slots;  // last chunk index that used slot s
        if (!mbar_wait_bounded(&full[s], uint32_t(last / g.slots) & 1u, kRowWaitLimitNs)) bad = true;
    }
}

// The fp32 weight in shared memory is laid out [VE/4][nvec][4]: quarter h of
// vector vi at float4 index h*nvec + vi, so a warp's 16-byte reads of one
// quarter for consecutive vectors are contiguous (no bank conflicts).
template <int VE>
__device__ __forceinline__ void rr_params2(const float* wsm, int vi, int nvec, float2 (&v)[VE / 2]) {
#pragma unroll
    for (int h = 0; h < VE / 4; ++h) {
        const float4 f = reinterpret_cast<const float4*>(wsm)[h * nvec + vi];
        v[2 * h] = make_float2(f.x, f.y);
        v[2 * h + 1] = make_float2(f.z, f.w);
    }
}

// Pair accumulators back to per-element form.
template <int VPT, int VE>
__device__ __forceinline__ void unpair(const float2 (&in)[VPT][VE / 2], float (&out)[VPT][VE]) {
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int h = 0; h < VE / 2; ++h) {
            out[j][2 * h] = in[j][h].x;
            out[j][2 * h + 1] = in[j][h].y;
        }
}

// The weight of the row as fp32 in shared memory, in rr_params2's layout
// (consumer threads).
template <typename T>
__device__ __forceinline__ void rr_stage_weight(const RowArgs& a, float* wsm, int consumers) {
    using bits = typename Io<T>::bits_t;
    constexpr int VE = kVec<T>;
    const int nvec = a.cols / VE;
    for (int i = threadIdx.x; i < a.cols; i += consumers) {
        const int vi = i / VE, k = i - vi * VE;
        wsm[((k >> 2) * nvec + vi) * 4 + (k & 3)] = a.w ? Io<T>::load(reinterpret_cast<const bits*>(a.w)[i]) : 1.f;
    }
}

// The CTA's dw (or db) partial row: each thread's per-column sums, summed over
// the row groups in group order.  Consumer threads only; `part` is scratch
// shared memory of RPC*TPR*VE floats (the drained ring), staged element-major
// (element k of thread t at k*TPR + t) so that the stores do not conflict.
template <int TPR, int VPT, int VE, int RPC, int NC = RPC * TPR>
__device__ __forceinline__ void rr_partial_row(const float (&acc)[VPT][VE], float* ws, float* part, int group,
                                               int t, int cols) {
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
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (j * TPR * VE >= cols) break;
#pragma unroll
            for (int k = 0; k < VE; ++k) part[group * TPR * VE + k * TPR + t] = acc[j][k];
            named_barrier(kRrBarConsumers, NC);
            for (int i = threadIdx.x; i < TPR * VE; i += NC) {
                const int k = i / TPR;
                const int col = j * TPR * VE + (i - k * TPR) * VE + k;
                if (col < cols) {
                    float sum = 0.f;
#pragma unroll
                    for (int gg = 0; gg < RPC; ++gg) sum += part[gg * TPR * VE + i];
                    ws[col] = sum;
                }
            }
            named_barrier(kRrBarConsumers, NC);
        }
    }
}

// DB: accumulate db = sum dy (LayerNorm, or RMSNorm with a bias); a template
// parameter so that RMSNorm without one keeps those registers free.  VPT: the
// row's vectors per thread (3 or 4): the dw/db accumulators are VPT*VE floats
// each, and at 544 threads a CTA has 96 registers per thread, so rows that
// need 3 vectors per thread do not carry a fourth's accumulators (they spilled).
// Vector vi (VE elements of a row of T) of a dy row stored as TD in the slot:
// one 16-byte read when TD is T, two when dy is float32 for a 16-bit x.
template <typename T, typename TD>
__device__ __forceinline__ void rr_load_dy(const unsigned char* dr, int vi, float2 (&dv)[kPairs<T>]) {
    if constexpr (sizeof(TD) == sizeof(T)) {
        unpack2<T>(*reinterpret_cast<const uint4*>(dr + size_t(vi) * 16), dv);
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(dr + size_t(vi) * 32);
        const uint4 u0 = p[0], u1 = p[1];
        dv[0] = make_float2(__uint_as_float(u0.x), __uint_as_float(u0.y));
        dv[1] = make_float2(__uint_as_float(u0.z), __uint_as_float(u0.w));
        dv[2] = make_float2(__uint_as_float(u1.x), __uint_as_float(u1.y));
        dv[3] = make_float2(__uint_as_float(u1.z), __uint_as_float(u1.w));
    }
}

// TD: dy's storage type (T, or float32 when the forward kept its output in
// float32 for a 16-bit x).
template <typename T, bool LN, int TPR, bool DB, int VPT, typename TD = T>
__global__ void __launch_bounds__(rr_threads(TPR), 1)
row_bwd_ring_kernel(const RowArgs a, const RrGeom g) {
    constexpr int VE = kVec<T>;
    static_assert(VPT <= kRrVpt, "at most kRrVpt vectors per thread");
    constexpr int CW = rr_consumer_warps(TPR);
    constexpr int NC = CW * 32;
    constexpr int RPC = NC / TPR;
    // one-warp rows of up to 3 vectors per thread keep the thread's columns of
    // the weight in registers (with a fourth vector's accumulators they would spill)
    constexpr bool kRegW = TPR == 32 && VPT <= 3;
    constexpr int NW = TPR / 32;
    constexpr int NV = LN ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kRrMaxSlots];
    __shared__ __align__(8) uint64_t empty[kRrMaxSlots];
    __shared__ float red[RPC][2 * NW * NV];
    __shared__ int s_bad;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    float* wsm = reinterpret_cast<float*>(smem);
    unsigned char* ring = smem + g.param_bytes;
    bool bad = false;

    if (threadIdx.x == 0) {
        s_bad = 0;
        for (int i = 0; i < g.slots; ++i) {
            mbar_init(&full[i], 33);  // the bulk copies' arrival + one per producer lane (mean/rstd)
            mbar_init(&empty[i], CW);
        }
        mbar_init_fence();
    }
    if (warp < CW) rr_stage_weight<T>(a, wsm, NC);
    __syncthreads();

    if (warp == CW) {
        rr_produce<T, LN, TD>(a, g, ring, full, empty, lane, bad);
    } else {
        const int group = threadIdx.x / TPR;
        const int t = threadIdx.x % TPR;
        const int cols = a.cols;
        const int nvec = cols / VE;
        const float fcols = float(cols);
        const float inv_cols = 1.f / fcols;
        const size_t row_bytes = size_t(cols) * sizeof(T);
        const size_t dy_row_bytes = size_t(cols) * sizeof(TD);
        T* __restrict__ dx = reinterpret_cast<T*>(a.dx);
        int phase = 0;
        // the element arithmetic runs on fp32 pairs (packed FP32 instructions)
        constexpr int H = VE / 2;
        float2 accw[VPT][H];
        float2 accb[VPT][H];
        float2 wreg[kRegW ? VPT : 1][H];
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int h = 0; h < H; ++h) accw[j][h] = accb[j][h] = f2(0.f);
        if constexpr (kRegW) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int vi = j * TPR + t;
                if (vi < nvec) {
                    rr_params2<VE>(wsm, vi, nvec, wreg[j]);
                } else {
#pragma unroll
                    for (int h = 0; h < H; ++h) wreg[j][h] = f2(0.f);
                }
            }
        }

        int q = 0;
        for (int64_t c = blockIdx.x; c < g.chunks; c += gridDim.x, ++q) {
            const int slot = q % g.slots;
            if (!mbar_wait_bounded(&full[slot], uint32_t(q / g.slots) & 1u, kRowWaitLimitNs)) bad = true;
            const int64_t r0 = c * g.R;
            const int ra = int(a.rows - r0 < g.R ? a.rows - r0 : g.R);
            const unsigned char* base = ring + size_t(slot) * g.slot_bytes;
            const float* st = reinterpret_cast<const float*>(base + size_t(g.R) * (dy_row_bytes + row_bytes));
            for (int r = group; r < ra; r += RPC) {
                const unsigned char* dr = base + size_t(r) * dy_row_bytes;
                const unsigned char* xr = base + size_t(g.R) * dy_row_bytes + size_t(r) * row_bytes;
                const float rs = st[r];
                const float mu = LN ? st[g.R + r] : 0.f;
                const float2 rs2 = f2(rs);
                const float2 nmu = f2(-mu);
                // the row sums: sum(dy*w) and sum(dy*w*xhat) (LN) / sum(dy*w*x) (RMS),
                // one accumulator per vector (short dependency chains)
                float2 s2[VPT][NV];
#pragma unroll
                for (int j = 0; j < VPT; ++j)
#pragma unroll
                    for (int i = 0; i < NV; ++i) s2[j][i] = f2(0.f);
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int vi = j * TPR + t;
                    if (vi < nvec) {
                        float2 dv[H], xv[H], wv[H];
                        rr_load_dy<T, TD>(dr, vi, dv);
                        unpack2<T>(*reinterpret_cast<const uint4*>(xr + size_t(vi) * 16), xv);
                        if constexpr (kRegW) {
#pragma unroll
                            for (int h = 0; h < H; ++h) wv[h] = wreg[j][h];
                        } else {
                            rr_params2<VE>(wsm, vi, nvec, wv);
                        }
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            const float2 gw = __fmul2_rn(dv[h], wv[h]);
                            if constexpr (LN) {
                                const float2 xh = __fmul2_rn(__fadd2_rn(xv[h], nmu), rs2);
                                s2[j][0] = __fadd2_rn(s2[j][0], gw);
                                s2[j][NV - 1] = __ffma2_rn(gw, xh, s2[j][NV - 1]);
                            } else {
                                s2[j][0] = __ffma2_rn(gw, xv[h], s2[j][0]);
                            }
                        }
                    }
                }
                float s[NV];
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    float2 acc = s2[0][i];
#pragma unroll
                    for (int j = 1; j < VPT; ++j) acc = __fadd2_rn(acc, s2[j][i]);
                    s[i] = acc.x + acc.y;
                }
                group_sum<TPR, NV>(s, &red[group][0], phase, group);
                const float c1 = s[0] * inv_cols;
                const float c2 = LN ? s[NV - 1] * inv_cols : c1 * rs * rs;
                const float2 nc1 = f2(-c1);
                const float2 nc2 = f2(-c2);
                T* dxr = dx + (r0 + r) * cols;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int vi = j * TPR + t;
                    if (vi < nvec) {
                        float2 dv[H], xv[H], wv[H], o[H];
                        rr_load_dy<T, TD>(dr, vi, dv);
                        unpack2<T>(*reinterpret_cast<const uint4*>(xr + size_t(vi) * 16), xv);
                        if constexpr (kRegW) {
#pragma unroll
                            for (int h = 0; h < H; ++h) wv[h] = wreg[j][h];
                        } else {
                            rr_params2<VE>(wsm, vi, nvec, wv);
                        }
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            const float2 gw = __fmul2_rn(dv[h], wv[h]);
                            if constexpr (LN) {
                                // dx = rs * (dy*w - c1 - xhat*c2)
                                const float2 xh = __fmul2_rn(__fadd2_rn(xv[h], nmu), rs2);
                                o[h] = __fmul2_rn(rs2, __ffma2_rn(xh, nc2, __fadd2_rn(gw, nc1)));
                                accw[j][h] = __ffma2_rn(dv[h], xh, accw[j][h]);
                                accb[j][h] = __fadd2_rn(accb[j][h], dv[h]);
                            } else {
                                // dx = rs * (dy*w - x*c2)
                                o[h] = __fmul2_rn(rs2, __ffma2_rn(xv[h], nc2, gw));
                                accw[j][h] = __ffma2_rn(dv[h], __fmul2_rn(xv[h], rs2), accw[j][h]);
                                if constexpr (DB) accb[j][h] = __fadd2_rn(accb[j][h], dv[h]);
                            }
                        }
                        st_v4(dxr + int64_t(vi) * VE, pack2x<T>(o));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // the column-sum kernel may be scheduled now; it waits for this grid
        pdl_trigger();
        // every chunk has been consumed (and its copies have landed): the ring is scratch now
        named_barrier(kRrBarConsumers, NC);
        float* part = reinterpret_cast<float*>(ring);
        float acc[VPT][VE];
        if (a.ws_dw) {
            unpair<VPT, VE>(accw, acc);
            rr_partial_row<TPR, VPT, VE, RPC, NC>(acc, a.ws_dw + int64_t(blockIdx.x) * cols, part, group, t, cols);
        }
        if constexpr (DB) {
            if (a.ws_db) {
                unpair<VPT, VE>(accb, acc);
                rr_partial_row<TPR, VPT, VE, RPC, NC>(acc, a.ws_db + int64_t(blockIdx.x) * cols, part, group, t,
                                                      cols);
            }
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0 && s_bad) atomicOr(a.err, kErrTimeoutStage);
}

}  // namespace nrm
