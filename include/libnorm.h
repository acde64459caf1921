/*
 * libnorm.h -- C ABI of libnorm: forward and backward passes of LayerNorm,
 * RMSNorm and BatchNorm (with fused residual add and activation) on one NVIDIA
 * GB300 GPU (sm_103a), computed by hand-written CUDA kernels.
 *
 * Sources for what each call computes (web articles on the attorch
 * normalization kernels):
 *   [NK] "attorch如何实现LayerNorm、BatchNorm与RMSNorm？3种归一化Triton核代码全解析"
 *   [AM] "如何用attorch.math快速开发自定义GPU算子：面向进阶开发者的算子融合实战指南"
 *   [AF] "算子融合实战：attorch激活函数与Dropout融合核的完整实现原理"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every pointer is a device pointer owned by the caller (cudaMalloc,
 *           PyTorch, a pool...).  The library allocates nothing; it keeps only
 *           per-device caches of device properties and kernel attributes.
 *           Tensors are dense and row-major (C order).  Pointers must be aligned
 *           to their element size; 16-byte alignment of every tensor (and a row
 *           or segment length that is a multiple of 16 bytes) selects the
 *           128-bit vector path, anything else a scalar path inside the same
 *           kernels.  In-place use (y == x, dx == dy) is not supported.
 * Streams.  Every call only enqueues work on `stream` (0 = legacy default
 *           stream) and returns without synchronising.  Argument errors are
 *           found on the host and returned before anything is enqueued.
 * Dtypes.   `dt` is the storage type of the activations (x, y, dy, dx, residual,
 *           dres).  Row-norm weight, bias and their gradients use the same `dt`;
 *           BatchNorm weight, bias, running statistics and their gradients are
 *           always float32.  Saved statistics are always float32.  All
 *           arithmetic is float32; stores round to nearest even.
 * Results.  For a fixed device, shape and set of pointers' alignment, every
 *           output is bitwise reproducible from run to run (no atomics in any
 *           reduction; all partial sums are combined in a fixed order).
 * Errors.   NRM_ERR_INVALID_ARG for a bad pointer, size, flag or dtype;
 *           NRM_ERR_UNSUPPORTED for a size beyond the limits below;
 *           NRM_ERR_WORKSPACE when workspace_bytes is too small;
 *           NRM_ERR_CUDA when a CUDA runtime call or launch fails;
 *           NRM_ERR_TIMEOUT (from nrm_sync_status) when a kernel's bounded wait
 *           gave up: on its own asynchronous copies, on another warp of its
 *           CTA, or on the other CTAs of a BatchNorm channel.  nrm_last_error_message()
 *           gives a human-readable reason for the last failure on this thread.
 * Limits.   rows, n*c*l < 2^40; cols < 2^31; a BatchNorm channel holds fewer
 *           than 2^31 elements (n*l).
 */
#ifndef LIBNORM_H
#define LIBNORM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NRM_API __attribute__((visibility("default")))
#else
#define NRM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so callers need no CUDA header. */
typedef struct CUstream_st *nrm_stream_t;

typedef enum nrm_status {
    NRM_OK = 0,
    NRM_ERR_INVALID_ARG = 1,
    NRM_ERR_UNSUPPORTED = 2,
    NRM_ERR_WORKSPACE = 3,
    NRM_ERR_CUDA = 4,
    NRM_ERR_TIMEOUT = 5
} nrm_status;

typedef enum nrm_dtype { NRM_F32 = 0, NRM_F16 = 1, NRM_BF16 = 2 } nrm_dtype;

/* Activation fused after BatchNorm ([NK] BatchNorm section, act_func, which
 * lists relu, gelu, silu and mish among the fusable activations; [AF] section
 * "六、一个内核通吃 21 种激活" for the set and section "五、反向传播融合同样成立"
 * for the derivative taken from the pre-activation input).  ReLU'(0) = 0.
 * GELU is the exact erf form z * Phi(z).  SiLU is z * sigmoid(z); Mish is
 * z * tanh(softplus(z)), softplus(z) = log(1 + e^z) (PyTorch's definitions:
 * the articles name the activations without formulas).  Two take a parameter,
 * passed as act_param (the [AF] article encodes it in the name, e.g.
 * "leaky_relu_0.01"): LEAKY_RELU is z for z > 0, else act_param*z (derivative
 * 1, else act_param); ELU is z for z > 0, else act_param*(e^z - 1) (derivative
 * 1, else act_param*e^z); CELU is z for z > 0, else act_param*(e^(z/act_param)
 * - 1) (derivative 1, else e^(z/act_param); act_param != 0).  SIGMOID is
 * 1/(1 + e^-z).  SELU is L*z for z > 0, else L*A*(e^z - 1), L and A the
 * constants of Klambauer et al. (2017).  RELU6 and HARDTANH are the clamps the
 * [AF] article names beside ReLU (section 七): min(max(z, 0), 6) and
 * min(max(z, -1), 1), each with derivative 1 strictly inside its range and 0
 * outside it and at both ends.  act_param is ignored by the others. */
typedef enum nrm_act {
    NRM_ACT_NONE = 0,
    NRM_ACT_RELU = 1,
    NRM_ACT_GELU = 2,
    NRM_ACT_SILU = 3,
    NRM_ACT_MISH = 4,
    NRM_ACT_LEAKY_RELU = 5,
    NRM_ACT_ELU = 6,
    NRM_ACT_SIGMOID = 7,
    NRM_ACT_CELU = 8,
    NRM_ACT_SELU = 9,
    NRM_ACT_RELU6 = 10,
    NRM_ACT_HARDTANH = 11
} nrm_act;

/* Operations that need a workspace (for nrm_workspace_bytes). */
typedef enum nrm_op {
    NRM_OP_LAYERNORM_BWD = 1,
    NRM_OP_RMSNORM_BWD = 2,
    NRM_OP_LAYERNORM_CF_BWD = 3 /* rows: n*l (unused), cols: c */
} nrm_op;

/* ------------------------------------------------------------------------ */
/* LayerNorm over the last dimension                                         */
/* ------------------------------------------------------------------------ */

/*
 * nrm_layernorm_fwd -- [NK] section "LayerNorm：一个程序归一化一批行", forward
 * steps 1-4; [AM] function table, calc_mean_and_inv_std and standardize.
 * For each row r of x[rows, cols]:
 *   mean = sum_j x_j / cols;  var = sum_j (x_j - mean)^2 / cols  (biased)
 *   rstd = (var + eps)^(-1/2);  y_j = (x_j - mean) * rstd * w_j + b_j
 * x, y: [rows, cols] in dt.  w, b: [cols] in dt, each may be NULL (1 and 0).
 * mean, rstd: float32 [rows], each may be NULL (the "save_stats" option).
 * rows >= 0 (0 is a no-op), cols >= 1, eps > 0.
 */
NRM_API nrm_status nrm_layernorm_fwd(const void *x, const void *w, const void *b, void *y,
                             float *mean, float *rstd, int64_t rows, int64_t cols,
                             float eps, nrm_dtype dt, nrm_stream_t stream);

/*
 * nrm_layernorm_bwd -- [NK] section "LayerNorm：一个程序归一化一批行", backward
 * paragraph (the two per-row sums "term1" and "term2" in one launch), and
 * section "三种核共享的工程技巧" (weight/bias gradients written per row block
 * into an intermediate buffer, then summed).  With g = dy*w and
 * xhat = (x - mean)*rstd:
 *   dx = rstd * (g - sum(g)/cols - xhat * sum(g*xhat)/cols)
 *   dw = sum over rows of dy*xhat;  db = sum over rows of dy
 * dy, x, dx: [rows, cols] in dt.  w: [cols] in dt or NULL (1).  mean, rstd:
 * float32 [rows] as written by nrm_layernorm_fwd.  dw, db: [cols] in dt, each
 * may be NULL.  workspace: device memory of at least
 * nrm_workspace_bytes(NRM_OP_LAYERNORM_BWD, rows, cols, dt) bytes, 16-byte
 * aligned, used as scratch for the per-block dw/db partial sums (its contents
 * on entry do not matter and are clobbered); may be NULL when dw and db are
 * both NULL.  The call enqueues two kernels when dw or db is requested.
 */
NRM_API nrm_status nrm_layernorm_bwd(const void *dy, const void *x, const void *w,
                             const float *mean, const float *rstd, void *dx,
                             void *dw, void *db, int64_t rows, int64_t cols,
                             nrm_dtype dt, void *workspace, size_t workspace_bytes,
                             nrm_stream_t stream);

/*
 * nrm_layernorm_bwd_noalloc -- nrm_layernorm_bwd without a workspace argument,
 * for callers that cannot allocate device memory when they run the backward:
 * code running under another framework's allocator (a plugin or custom op
 * whose host runtime forbids or accounts every allocation), loops that must
 * never enter the allocator after start-up (cudaMalloc can synchronise the
 * device and stall), and C callers that were handed device pointers and have no
 * allocator of their own.  The articles have no counterpart of this call; it is
 * a property of this library's interface, not of the method.
 * The dw/db partial rows live in a library-owned static device array of 8 MiB
 * (2^21 floats), which every GPU that loads libnorm holds until the process
 * exits.  cols must be <= 65536 (else NRM_ERR_UNSUPPORTED); the call allocates
 * nothing.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  All calls share the one
 * array, so calls that overlap on the GPU (unordered streams) race on it;
 * calls ordered on one stream are safe.
 * Its contents need no initialisation: every call writes each partial value it
 * reads.  The looked-up address is kept for the life of the process: do not
 * reset a device (cudaDeviceReset) or destroy its primary context while the
 * library is loaded and this call is in use, since the kept address would then
 * point into a released module.  Arguments, results and errors are otherwise
 * those of nrm_layernorm_bwd.
 */
NRM_API nrm_status nrm_layernorm_bwd_noalloc(const void *dy, const void *x, const void *w,
                                     const float *mean, const float *rstd, void *dx,
                                     void *dw, void *db, int64_t rows, int64_t cols,
                                     nrm_dtype dt, nrm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* LayerNorm over the channels of an NCHW tensor (channels first)            */
/* ------------------------------------------------------------------------ */

/*
 * nrm_layernorm_cf_fwd -- the LayerNorm of nrm_layernorm_fwd ([NK] section
 * "LayerNorm：一个程序归一化一批行", forward steps 1-4) taken over the channels:
 * for x of shape [n, c, l] (NCHW, l = H*W), for every sample i and spatial
 * position p,
 *   mean = sum_ch x[i,ch,p] / c;  var = sum_ch (x[i,ch,p] - mean)^2 / c
 *   rstd = (var + eps)^(-1/2);  y[i,ch,p] = (x[i,ch,p] - mean)*rstd*w[ch] + b[ch]
 * (the layout of ConvNeXt, which [NK] section "三种核共享的工程技巧" lists as a
 * LayerNorm user; it normalises the channels of each position).  x, y:
 * [n, c, l] in dt.  w, b: [c] in dt, each may be NULL (1 and 0).  mean,
 * rstd: float32 [n, l], each may be NULL.  n, l >= 0 (an empty tensor is a
 * no-op), 1 <= c <= 16384, eps > 0.
 */
NRM_API nrm_status nrm_layernorm_cf_fwd(const void *x, const void *w, const void *b, void *y,
                                float *mean, float *rstd, int64_t n, int64_t c, int64_t l,
                                float eps, nrm_dtype dt, nrm_stream_t stream);

/*
 * nrm_layernorm_cf_bwd -- backward of nrm_layernorm_cf_fwd: per (sample,
 * position), with g = dy*w and xhat = (x - mean)*rstd over its channels,
 *   dx = rstd * (g - sum(g)/c - xhat * sum(g*xhat)/c)
 *   dw[ch] = sum over (i, p) of dy*xhat;  db[ch] = sum over (i, p) of dy
 * dy, x, dx: [n, c, l] in dt.  w: [c] in dt or NULL (1).  mean, rstd:
 * float32 [n, l] as written by nrm_layernorm_cf_fwd.  dw, db: [c] in dt, each
 * may be NULL.  workspace: at least
 * nrm_workspace_bytes(NRM_OP_LAYERNORM_CF_BWD, n*l, c, dt) bytes, 16-byte
 * aligned, scratch for the per-block dw/db partial sums (clobbered); may be
 * NULL when dw and db are both NULL.  Two kernels are enqueued when dw or db
 * is requested.  Errors as nrm_layernorm_bwd.
 */
NRM_API nrm_status nrm_layernorm_cf_bwd(const void *dy, const void *x, const void *w,
                                const float *mean, const float *rstd, void *dx, void *dw,
                                void *db, int64_t n, int64_t c, int64_t l, nrm_dtype dt,
                                void *workspace, size_t workspace_bytes, nrm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* RMSNorm over the last dimension                                           */
/* ------------------------------------------------------------------------ */

/*
 * nrm_rmsnorm_fwd -- [NK] section "RMSNorm：去掉均值的极简版 LayerNorm": no mean
 * is subtracted; output = input * inv_rms * weight (+ bias) with
 *   inv_rms = (sum_j x_j^2 / cols + eps)^(-1/2).
 * x, y: [rows, cols] in dt.  w: [cols] in dt or NULL (1).  b: [cols] in dt or
 * NULL: the article's formula has no bias; a bias is added after the weight,
 * as LayerNorm's is.  rstd: float32 [rows] receives inv_rms, may be NULL.
 */
NRM_API nrm_status nrm_rmsnorm_fwd(const void *x, const void *w, const void *b, void *y,
                           float *rstd, int64_t rows, int64_t cols, float eps, nrm_dtype dt,
                           nrm_stream_t stream);

/*
 * nrm_rmsnorm_bwd -- [NK] RMSNorm section, backward sentence (the LayerNorm
 * reduction reused with the row sum of input * output_grad * weight).  With
 * g = dy*w and s = sum(g*x):
 *   dx = inv_rms * g - x * inv_rms^3 * s / cols;  dw = sum over rows of dy*x*inv_rms
 *   db = sum over rows of dy (the bias, when the forward had one)
 * Arguments as nrm_layernorm_bwd, with rstd = inv_rms from nrm_rmsnorm_fwd and
 * NRM_OP_RMSNORM_BWD for the workspace size.  dw, db may be NULL.
 */
NRM_API nrm_status nrm_rmsnorm_bwd(const void *dy, const void *x, const void *w,
                           const float *rstd, void *dx, void *dw, void *db, int64_t rows,
                           int64_t cols, nrm_dtype dt, void *workspace,
                           size_t workspace_bytes, nrm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Output kept in float32 for a 16-bit input                                 */
/* ------------------------------------------------------------------------ */

/*
 * nrm_layernorm_fwd_ex, nrm_rmsnorm_fwd_ex -- [NK] LayerNorm section, layer
 * paragraph: the layer's autocast_to_fp32 flag chooses between keeping the
 * input precision and PyTorch's mixed-precision behaviour of returning
 * float32.  As nrm_layernorm_fwd / nrm_rmsnorm_fwd, with y stored in y_dt:
 * y_dt == dt (the plain calls) or NRM_F32 for a float16/bfloat16 x (the
 * arithmetic is float32 either way; only the output's rounding differs).
 * Any other y_dt returns NRM_ERR_UNSUPPORTED.  y must be aligned to y_dt's
 * size.
 */
NRM_API nrm_status nrm_layernorm_fwd_ex(const void *x, const void *w, const void *b, void *y,
                                float *mean, float *rstd, int64_t rows, int64_t cols, float eps,
                                nrm_dtype dt, nrm_dtype y_dt, nrm_stream_t stream);
NRM_API nrm_status nrm_rmsnorm_fwd_ex(const void *x, const void *w, const void *b, void *y,
                              float *rstd, int64_t rows, int64_t cols, float eps, nrm_dtype dt,
                              nrm_dtype y_dt, nrm_stream_t stream);

/*
 * nrm_layernorm_bwd_ex, nrm_rmsnorm_bwd_ex -- the backward of the _ex
 * forwards: dy is stored in dy_dt (the forward's y_dt); x, dx, w, dw, db in
 * dt.  Otherwise as nrm_layernorm_bwd / nrm_rmsnorm_bwd (same workspace).
 */
NRM_API nrm_status nrm_layernorm_bwd_ex(const void *dy, const void *x, const void *w,
                                const float *mean, const float *rstd, void *dx, void *dw,
                                void *db, int64_t rows, int64_t cols, nrm_dtype dt,
                                nrm_dtype dy_dt, void *workspace, size_t workspace_bytes,
                                nrm_stream_t stream);
NRM_API nrm_status nrm_rmsnorm_bwd_ex(const void *dy, const void *x, const void *w,
                              const float *rstd, void *dx, void *dw, void *db, int64_t rows,
                              int64_t cols, nrm_dtype dt, nrm_dtype dy_dt, void *workspace,
                              size_t workspace_bytes, nrm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* BatchNorm over (batch, spatial) per channel, NCHW                         */
/* ------------------------------------------------------------------------ */

/*
 * nrm_batchnorm_fwd -- [NK] section "BatchNorm：按特征并行 + 激活融合" (statistics
 * per channel over batch and spatial positions, accumulated block by block with
 * an online mean/variance update; running statistics updated with momentum in
 * training and read directly in inference; residual add and activation fused in
 * the same kernel); [AM] section "实战二 Welford EMA 组合手写 BatchNorm 融合统计"
 * (Welford update, EMA (1-momentum)*old + momentum*new).
 * Per channel ch, over the M = n*l elements of x[:, ch, :]:
 *   training:  mean = batch mean;  var = biased batch variance;
 *              running_mean = (1-momentum)*running_mean + momentum*mean
 *              running_var  = (1-momentum)*running_var  + momentum*var*M/(M-1)
 *   eval:      mean = running_mean;  var = running_var (no update)
 *   rstd = (var + eps)^(-1/2);  z = (x - mean)*rstd*w + b (+ residual);  y = act(z)
 * x, residual, y: [n, c, l] in dt (NCHW with l = H*W; residual may be NULL).
 * w, b: float32 [c] or NULL (1, 0).  running_mean, running_var: float32 [c],
 * both NULL or both set in training (updated in place), both required in eval.
 * save_mean, save_rstd: float32 [c] or NULL; training writes the batch mean and
 * rstd, eval writes running_mean and (running_var+eps)^(-1/2); the backward
 * reads them.
 * workspace: device memory, 16-byte aligned, of at least
 * nrm_batchnorm_workspace_bytes(n, c, l, dt) bytes; the call splits large
 * channels over several CTAs, which meet there (per-channel counters reset by
 * the call with an enqueued memset, and per-slice partial statistics).  It may
 * be NULL when every channel fits one CTA; otherwise a NULL or short workspace
 * returns NRM_ERR_WORKSPACE.  Calls that overlap on the GPU need separate
 * workspaces.
 * act_mask: NULL or, for act == NRM_ACT_RELU, nrm_act_mask_words(n, c, l)
 * uint32 words receiving bit (z > 0) per element: segment (i, ch) owns
 * ceil(l/32) words starting at word (i*c + ch)*ceil(l/32) and element j of the
 * segment is bit j%32 of word j/32 (unused high bits are 0).  It must be NULL
 * for other activations.  act_param: the slope or alpha of LEAKY_RELU / ELU
 * (finite; ignored otherwise).
 * training requires M >= 2.  eps > 0, 0 <= momentum <= 1.
 */
NRM_API nrm_status nrm_batchnorm_fwd(const void *x, const void *residual, const float *w,
                             const float *b, void *y, float *running_mean,
                             float *running_var, float *save_mean, float *save_rstd,
                             uint32_t *act_mask, int64_t n, int64_t c, int64_t l,
                             float eps, float momentum, int training, nrm_act act,
                             float act_param, nrm_dtype dt, void *workspace,
                             size_t workspace_bytes, nrm_stream_t stream);

/*
 * nrm_batchnorm_bwd -- [NK] BatchNorm section, last sentences: with a fused
 * activation the backward first recovers the pre-activation gradient, then
 * computes the BatchNorm gradient.  With xhat = (x - save_mean)*save_rstd and
 * z = xhat*w + b (+ residual):
 *   dz   = dy * act'(z)   (ReLU: the act_mask bit when act_mask != NULL,
 *                          otherwise z is recomputed from x and residual)
 *   dres = dz;  db = sum dz;  dw = sum dz*xhat          (per channel)
 *   training: dx = w*rstd*(dz - db/M - xhat*dw/M)
 *   eval:     dx = w*rstd*dz
 * dy, x, residual, dx, dres: [n, c, l] in dt.  residual is needed only to
 * recompute z (GELU, or ReLU without a mask) when the forward used one.
 * w, b: float32 [c] or NULL (1, 0), as in the forward.  save_mean, save_rstd:
 * float32 [c] from nrm_batchnorm_fwd with the same `training` flag.
 * act_mask: NULL, or the mask the forward wrote (ReLU only).  act, act_param:
 * those of the forward.  dres, dw, db may be NULL.  workspace: as for
 * nrm_batchnorm_fwd.
 */
NRM_API nrm_status nrm_batchnorm_bwd(const void *dy, const void *x, const void *residual,
                             const float *w, const float *b, const float *save_mean,
                             const float *save_rstd, const uint32_t *act_mask,
                             void *dx, void *dres, float *dw, float *db, int64_t n,
                             int64_t c, int64_t l, int training, nrm_act act,
                             float act_param, nrm_dtype dt, void *workspace,
                             size_t workspace_bytes, nrm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Activation with fused dropout                                             */
/* ------------------------------------------------------------------------ */

/*
 * nrm_act_dropout_fwd -- "算子融合实战：attorch激活函数与Dropout融合核的完整实现原理",
 * sections "三、融合内核的骨架" and "四、Dropout 融合的关键：可复现的随机掩码": the
 * activation's result goes through inverted dropout in the same pass,
 *   y[e] = act(x[e]) / (1 - drop_p)  if element e is kept,  else 0.
 * The mask is not stored: element e's random value is a function of (seed, e)
 * alone.  Generator (this library's reading of the article's tl.rand(seed,
 * offset)): Philox4x32-10 (Salmon et al., SC 2011) with key (seed, 0) and
 * counter (e / 4 as two 32-bit words, 0, 0); element e takes output word e % 4,
 * u = (word >> 8) * 2^-24, and is dropped when u < drop_p (compared in single
 * precision).  x, y: count elements in dt (contiguous; y may equal x).
 * act: NRM_ACT_NONE (plain dropout) or any activation of nrm_act, with
 * act_param for LEAKY_RELU and ELU.  drop_p in
 * [0, 1]: 0 keeps every element, 1 drops every one.  Any seed; the article
 * draws a 16-bit one.  One kernel is enqueued (none for count == 0).
 * Errors: NRM_ERR_INVALID_ARG for a negative count, drop_p outside [0, 1] or
 * NaN, an unknown act or dtype, a non-finite act_param, NULL or misaligned
 * pointers with count > 0.
 */
NRM_API nrm_status nrm_act_dropout_fwd(const void *x, void *y, int64_t count, nrm_act act,
                               float act_param, float drop_p, uint32_t seed, nrm_dtype dt,
                               nrm_stream_t stream);

/*
 * nrm_act_dropout_bwd -- same article, section "五、反向传播融合同样成立": the mask
 * is rebuilt from the same seed and offsets and the derivative is taken at the
 * saved input,
 *   dx[e] = dy[e] / (1 - drop_p) * act'(x[e])  if kept,  else 0   (ReLU'(0) = 0).
 * dy, x, dx: count elements in dt (dx may equal dy or x).  act, act_param,
 * drop_p, seed: those of the forward.  Errors as nrm_act_dropout_fwd.
 */
NRM_API nrm_status nrm_act_dropout_bwd(const void *dy, const void *x, void *dx, int64_t count,
                               nrm_act act, float act_param, float drop_p, uint32_t seed,
                               nrm_dtype dt, nrm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Helpers                                                                   */
/* ------------------------------------------------------------------------ */

/* Workspace bytes the row-norm backward needs on the current device for
 * [rows, cols] (it depends on the device's SM count).  Returns 0 for bad
 * arguments or when no CUDA device is usable. */
NRM_API size_t nrm_workspace_bytes(nrm_op op, int64_t rows, int64_t cols, nrm_dtype dt);

/* Workspace bytes that suffice for nrm_batchnorm_fwd/bwd on [n, c, l] on the
 * current device (it depends on the device's SM count).  Returns 0 for bad
 * arguments or when no CUDA device is usable. */
NRM_API size_t nrm_batchnorm_workspace_bytes(int64_t n, int64_t c, int64_t l, nrm_dtype dt);

/* Number of uint32 words of a BatchNorm ReLU mask for [n, c, l]. */
NRM_API int64_t nrm_act_mask_words(int64_t n, int64_t c, int64_t l);

/* Synchronises `stream`, then returns NRM_ERR_TIMEOUT if a kernel of this
 * library on the current device reported a timed-out wait since the last call
 * (and clears that report), NRM_ERR_CUDA if the stream reported an error, and
 * NRM_OK otherwise. */
NRM_API nrm_status nrm_sync_status(nrm_stream_t stream);

/* Static string naming a status code. */
NRM_API const char *nrm_status_str(nrm_status status);

/* Human-readable reason for the last non-OK status returned on this thread
 * ("" if none). */
NRM_API const char *nrm_last_error_message(void);

/* Library version, major*10000 + minor*100 + patch. */
NRM_API int nrm_version(void);

/*
 * nrm_test_expire_peer_waits -- a test hook for the failure path of the
 * BatchNorm kernels whose channels span several CTAs.  The articles have no
 * counterpart: it exercises this library's own failure detection.
 * Those kernels wait, bounded, for every CTA of a channel to publish its
 * partial sums; a CTA that gives up records NRM_ERR_TIMEOUT (reported by the
 * next nrm_sync_status), finishes its own part of the call with the partial
 * sums it found and waits for its own copies before it exits.  This call arms,
 * for the next nrm_batchnorm_fwd or nrm_batchnorm_bwd in training mode on the
 * calling thread that runs such a kernel (16-byte aligned tensors, or the
 * scalar path, with a channel cut into more than one slice), a wait for one
 * CTA more than the launch has and a limit of `limit_ns` nanoseconds instead
 * of 2 s: every waiting CTA then gives up after `limit_ns`, and that call's
 * outputs are undefined.  Calls that do not wait for other CTAs leave it armed.
 * limit_ns must be in [1, 10^9] (else NRM_ERR_INVALID_ARG).  No GPU fault is
 * involved: the kernel ends normally and the device stays usable.
 */
NRM_API nrm_status nrm_test_expire_peer_waits(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* LIBNORM_H */
