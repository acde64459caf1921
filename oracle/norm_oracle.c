/*
 * norm_oracle.c -- plain double-precision CPU oracle for LayerNorm, RMSNorm and
 * BatchNorm, forward and backward, and for the activation with fused dropout.
 *
 * TEST INFRASTRUCTURE ONLY.  The parity tests, the smoke check and the bench's
 * CPU-baseline leg call it; the CUDA library never does, and this file shares no
 * code, header, table or helper with the CUDA path.
 *
 * Every function is the textbook definition written out with plain loops, in the
 * order the articles describe the computation, with no blocking, fusion or
 * reordering.  All arithmetic is in double; inputs are double copies of the
 * (already rounded) tensors the GPU sees.
 *
 * Sources (web articles on the attorch normalization kernels):
 *   [NK] "attorch如何实现LayerNorm、BatchNorm与RMSNorm？3种归一化Triton核代码全解析"
 *   [AM] "如何用attorch.math快速开发自定义GPU算子：面向进阶开发者的算子融合实战指南"
 *   [AF] "算子融合实战：attorch激活函数与Dropout融合核的完整实现原理"
 *
 * Readings taken where the articles leave a step open (each is also listed in the
 * design notes):
 *   - LayerNorm variance divides by N (biased), as a drop-in nn.LayerNorm does.
 *   - eps sits inside the root: (var + eps)^(-1/2), (ms + eps)^(-1/2).
 *   - RMSNorm has a weight; its bias (NULL in the articles' formula) is added
 *     after the weight, as LayerNorm's is, and its gradient is db = sum dy.
 *   - BatchNorm normalises with the biased batch variance and feeds the unbiased
 *     one, M/(M-1) times larger, to running_var.
 *   - EMA: new = (1 - momentum) * old + momentum * batch value.
 *   - The residual is added after the affine step and before the activation; its
 *     gradient is the pre-activation gradient itself.
 *   - ReLU'(z) = 1 for z > 0 and 0 otherwise; GELU is the exact erf form.
 *   - The activations with a parameter a (the article encodes it in the name):
 *     leaky_relu(z) = z for z > 0, else a*z (derivative 1, else a);
 *     elu(z) = z for z > 0, else a*(e^z - 1) (derivative 1, else a*e^z);
 *     celu(z) = z for z > 0, else a*(e^(z/a) - 1) (derivative 1, else e^(z/a)).
 *   - sigmoid(z) = 1/(1 + e^-z); selu(z) = L*z for z > 0, else L*A*(e^z - 1),
 *     with the constants L, A of Klambauer et al., "Self-Normalizing Neural
 *     Networks" (2017).
 *   - The clamping activations the activation article names beside ReLU
 *     (section 七): relu6(z) = min(max(z, 0), 6) and hardtanh(z) =
 *     min(max(z, -1), 1); each has derivative 1 strictly inside its range and
 *     0 outside it and at its ends.
 *   - Dropout draws Philox4x32-10 with key (seed, 0) and counter (e / 4, 0, 0) for
 *     element e, which takes output word e % 4 as the uniform (word >> 8) * 2^-24;
 *     the element is dropped when that value is below drop_p (single precision).
 *
 * Parity status: every function here is pinned by the CPU tests (closed forms,
 * invariants, finite differences, independent library routines, hand-worked
 * fixtures).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "norm_oracle.h"

/* ------------------------------------------------------------------------ */
/* LayerNorm                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * [NK] section "LayerNorm：一个程序归一化一批行", forward steps 2-4: the row mean is
 * the row sum over feat_dim; the variance is the sum of squared deviations from
 * that mean; a reciprocal square root gives inv_std; the normalised row is scaled
 * by weight and shifted by bias (both optional).  [AM] function table,
 * calc_mean_and_inv_std and standardize.
 */
void oracle_layernorm_fwd(int64_t rows, int64_t cols, const double *x,
                          const double *w, const double *b, double eps,
                          double *y, double *mean, double *rstd)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            sum += xr[j];
        double mu = sum / (double)cols;

        double ssd = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            ssd += (xr[j] - mu) * (xr[j] - mu);
        double var = ssd / (double)cols;
        double rs = 1.0 / sqrt(var + eps);

        for (int64_t j = 0; j < cols; ++j) {
            double xhat = (xr[j] - mu) * rs;
            double wj = w ? w[j] : 1.0;
            double bj = b ? b[j] : 0.0;
            y[r * cols + j] = xhat * wj + bj;
        }
        if (mean) mean[r] = mu;
        if (rstd) rstd[r] = rs;
    }
}

/*
 * [NK] section "LayerNorm：一个程序归一化一批行", backward paragraph: the input
 * gradient needs two sums along the feature axis ("term1", "term2").  With
 * g = dy * w and xhat = (x - mean) * rstd these are sum(g) and sum(g * xhat):
 *   dx = rstd * (g - sum(g)/N - xhat * sum(g * xhat)/N).
 * [NK] section "三种核共享的工程技巧", blocked gradient aggregation: dw and db are
 * column sums over all rows of dy * xhat and dy.  Statistics are recomputed here
 * from x in double.
 */
void oracle_layernorm_bwd(int64_t rows, int64_t cols, const double *dy,
                          const double *x, const double *w, double eps,
                          double *dx, double *dw, double *db)
{
    if (dw) for (int64_t j = 0; j < cols; ++j) dw[j] = 0.0;
    if (db) for (int64_t j = 0; j < cols; ++j) db[j] = 0.0;

    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        const double *dyr = dy + r * cols;

        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            sum += xr[j];
        double mu = sum / (double)cols;
        double ssd = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            ssd += (xr[j] - mu) * (xr[j] - mu);
        double rs = 1.0 / sqrt(ssd / (double)cols + eps);

        double sum_g = 0.0, sum_gxhat = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double xhat = (xr[j] - mu) * rs;
            double g = dyr[j] * (w ? w[j] : 1.0);
            sum_g += g;
            sum_gxhat += g * xhat;
        }
        for (int64_t j = 0; j < cols; ++j) {
            double xhat = (xr[j] - mu) * rs;
            double g = dyr[j] * (w ? w[j] : 1.0);
            dx[r * cols + j] = rs * (g - sum_g / (double)cols
                                       - xhat * sum_gxhat / (double)cols);
            if (dw) dw[j] += dyr[j] * xhat;
            if (db) db[j] += dyr[j];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * [NK] section "RMSNorm：去掉均值的极简版 LayerNorm": no mean is taken; the output
 * is input * inv_rms * weight, inv_rms = (mean(x^2) + eps)^(-1/2).  An optional
 * bias b (the formula has none) is added last.
 */
void oracle_rmsnorm_fwd(int64_t rows, int64_t cols, const double *x,
                        const double *w, const double *b, double eps, double *y,
                        double *rstd)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        double ss = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            ss += xr[j] * xr[j];
        double rr = 1.0 / sqrt(ss / (double)cols + eps);
        for (int64_t j = 0; j < cols; ++j)
            y[r * cols + j] = xr[j] * rr * (w ? w[j] : 1.0) + (b ? b[j] : 0.0);
        if (rstd) rstd[r] = rr;
    }
}

/*
 * [NK] section "RMSNorm：去掉均值的极简版 LayerNorm", backward sentence: the
 * LayerNorm reduction is reused with the row sum of input * output_grad * weight.
 * With g = dy * w and s = sum(g * x):
 *   dx = inv_rms * g - x * inv_rms^3 * s / N,    dw = sum over rows of dy * x * inv_rms,
 *   db = sum over rows of dy (the optional bias).
 */
void oracle_rmsnorm_bwd(int64_t rows, int64_t cols, const double *dy,
                        const double *x, const double *w, double eps,
                        double *dx, double *dw, double *db)
{
    if (dw) for (int64_t j = 0; j < cols; ++j) dw[j] = 0.0;
    if (db) for (int64_t j = 0; j < cols; ++j) db[j] = 0.0;

    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        const double *dyr = dy + r * cols;
        double ss = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            ss += xr[j] * xr[j];
        double rr = 1.0 / sqrt(ss / (double)cols + eps);

        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += dyr[j] * (w ? w[j] : 1.0) * xr[j];
        for (int64_t j = 0; j < cols; ++j) {
            double g = dyr[j] * (w ? w[j] : 1.0);
            dx[r * cols + j] = rr * g - xr[j] * rr * rr * rr * s / (double)cols;
            if (dw) dw[j] += dyr[j] * xr[j] * rr;
            if (db) db[j] = db[j] + dyr[j];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* LayerNorm over the channels of an NCHW tensor                             */
/* ------------------------------------------------------------------------ */

/*
 * The LayerNorm of [NK] section "LayerNorm：一个程序归一化一批行" (mean, biased
 * variance, reciprocal square root, weight and bias), taken for every sample i
 * and spatial position p over the c channels of x[i, :, p], x of shape
 * [n, c, l] with l = H*W.  [NK] section "三种核共享的工程技巧" (application
 * paragraph) has ConvNeXt use attorch.LayerNorm; ConvNeXt normalises over the
 * channels of each position.  mean and rstd are [n, l].
 */
void oracle_layernorm_cf_fwd(int64_t n, int64_t c, int64_t l, const double *x,
                             const double *w, const double *b, double eps,
                             double *y, double *mean, double *rstd)
{
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t p = 0; p < l; ++p) {
            const double *xp = x + i * c * l + p;
            double sum = 0.0;
            for (int64_t ch = 0; ch < c; ++ch) sum += xp[ch * l];
            double mu = sum / (double)c;
            double ssd = 0.0;
            for (int64_t ch = 0; ch < c; ++ch) {
                double d = xp[ch * l] - mu;
                ssd += d * d;
            }
            double var = ssd / (double)c;
            double inv_std = 1.0 / sqrt(var + eps);
            for (int64_t ch = 0; ch < c; ++ch) {
                double xhat = (xp[ch * l] - mu) * inv_std;
                y[i * c * l + ch * l + p] = xhat * (w ? w[ch] : 1.0) + (b ? b[ch] : 0.0);
            }
            if (mean) mean[i * l + p] = mu;
            if (rstd) rstd[i * l + p] = inv_std;
        }
    }
}

/* Backward of the above: with g = dy*w over the channels of a position,
 * dx = rstd*(g - sum(g)/c - xhat*sum(g*xhat)/c); dw = sum over (i, p) of
 * dy*xhat, db = sum of dy (the row LayerNorm's backward, per position). */
void oracle_layernorm_cf_bwd(int64_t n, int64_t c, int64_t l, const double *dy,
                             const double *x, const double *w, double eps,
                             double *dx, double *dw, double *db)
{
    if (dw) for (int64_t ch = 0; ch < c; ++ch) dw[ch] = 0.0;
    if (db) for (int64_t ch = 0; ch < c; ++ch) db[ch] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t p = 0; p < l; ++p) {
            const int64_t base = i * c * l + p;
            double sum = 0.0;
            for (int64_t ch = 0; ch < c; ++ch) sum += x[base + ch * l];
            double mu = sum / (double)c;
            double ssd = 0.0;
            for (int64_t ch = 0; ch < c; ++ch) {
                double d = x[base + ch * l] - mu;
                ssd += d * d;
            }
            double rs = 1.0 / sqrt(ssd / (double)c + eps);
            double sum_g = 0.0, sum_gxhat = 0.0;
            for (int64_t ch = 0; ch < c; ++ch) {
                double g = dy[base + ch * l] * (w ? w[ch] : 1.0);
                double xhat = (x[base + ch * l] - mu) * rs;
                sum_g += g;
                sum_gxhat += g * xhat;
            }
            for (int64_t ch = 0; ch < c; ++ch) {
                double g = dy[base + ch * l] * (w ? w[ch] : 1.0);
                double xhat = (x[base + ch * l] - mu) * rs;
                dx[base + ch * l] = rs * (g - sum_g / (double)c - xhat * sum_gxhat / (double)c);
                if (dw) dw[ch] += dy[base + ch * l] * xhat;
                if (db) db[ch] += dy[base + ch * l];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* BatchNorm with fused residual add and activation                          */
/* ------------------------------------------------------------------------ */

/* [AF] section "五、反向传播融合同样成立": the activation derivative is taken from
 * the pre-activation input; GELU is the error-function form.  [NK] BatchNorm
 * section names silu and mish among the fused activations; their formulas are
 * the standard ones (the articles give none): silu(z) = z * sigmoid(z),
 * mish(z) = z * tanh(softplus(z)), softplus(z) = log(1 + e^z). */
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
/* SELU's scale and alpha (Klambauer et al. 2017, the fixed point of their
 * self-normalising mapping) */
#define SELU_LAMBDA 1.0507009873554804934193349852946
#define SELU_ALPHA 1.6732632423543772848170429916717
static double softplus(double z) { return z > 0.0 ? z + log1p(exp(-z)) : log1p(exp(z)); }

static double act_forward(int act, double param, double z)
{
    switch (act) {
    case ORACLE_ACT_RELU: return z > 0.0 ? z : 0.0;
    case ORACLE_ACT_LEAKY_RELU: return z > 0.0 ? z : param * z;
    case ORACLE_ACT_ELU: return z > 0.0 ? z : param * expm1(z);
    case ORACLE_ACT_SIGMOID: return sigmoid(z);
    case ORACLE_ACT_CELU: return z > 0.0 ? z : param * expm1(z / param);
    case ORACLE_ACT_SELU: return z > 0.0 ? SELU_LAMBDA * z : SELU_LAMBDA * SELU_ALPHA * expm1(z);
    case ORACLE_ACT_GELU: return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
    case ORACLE_ACT_SILU: return z * sigmoid(z);
    case ORACLE_ACT_MISH: return z * tanh(softplus(z));
    case ORACLE_ACT_RELU6: return z < 0.0 ? 0.0 : (z > 6.0 ? 6.0 : z);
    case ORACLE_ACT_HARDTANH: return z < -1.0 ? -1.0 : (z > 1.0 ? 1.0 : z);
    default:              return z;
    }
}

static double act_derivative(int act, double param, double z)
{
    switch (act) {
    case ORACLE_ACT_RELU: return z > 0.0 ? 1.0 : 0.0;
    case ORACLE_ACT_LEAKY_RELU: return z > 0.0 ? 1.0 : param;
    case ORACLE_ACT_ELU: return z > 0.0 ? 1.0 : param * exp(z);
    case ORACLE_ACT_SIGMOID: {
        double s = sigmoid(z);
        return s * (1.0 - s);
    }
    case ORACLE_ACT_CELU: return z > 0.0 ? 1.0 : exp(z / param);
    case ORACLE_ACT_SELU: return z > 0.0 ? SELU_LAMBDA : SELU_LAMBDA * SELU_ALPHA * exp(z);
    case ORACLE_ACT_GELU: {
        double cdf = 0.5 * (1.0 + erf(z / sqrt(2.0)));
        double pdf = exp(-0.5 * z * z) / sqrt(2.0 * M_PI);
        return cdf + z * pdf;
    }
    case ORACLE_ACT_SILU: {
        /* d/dz z*s(z) = s + z*s*(1 - s) */
        double s = sigmoid(z);
        return s + z * s * (1.0 - s);
    }
    case ORACLE_ACT_MISH: {
        /* d/dz z*tanh(sp(z)) = tanh(sp) + z*(1 - tanh(sp)^2)*sp'(z), sp' = sigmoid */
        double t = tanh(softplus(z));
        return t + z * (1.0 - t * t) * sigmoid(z);
    }
    case ORACLE_ACT_RELU6: return (z > 0.0 && z < 6.0) ? 1.0 : 0.0;
    case ORACLE_ACT_HARDTANH: return (z > -1.0 && z < 1.0) ? 1.0 : 0.0;
    default: return 1.0;
    }
}

static int64_t mask_words_per_segment(int64_t l) { return (l + 31) / 32; }

/*
 * [NK] section "BatchNorm：按特征并行 + 激活融合": statistics per feature channel
 * over batch and spatial positions; training updates running_mean/running_var with
 * momentum and inference reads them directly, with PyTorch semantics; weight and
 * bias, then the optional residual (pre_act_add), then the activation (act_func),
 * all in one pass.  [AM] section "实战二 Welford EMA 组合手写 BatchNorm 融合统计":
 * the EMA is (1 - momentum) * old + momentum * new, and the residual and activation
 * follow the normalisation.
 *
 * Layout: x, res, y, z_out are [n, c, l] (NCHW with l = H*W).  w, b, running_*,
 * save_* are [c].  act_mask (written only for ReLU, may be NULL) holds one bit per
 * element, z > 0, packed per (sample, channel) segment: segment (i, ch) owns
 * ceil(l/32) 32-bit words starting at word (i*c + ch)*ceil(l/32); element j of
 * the segment is bit j%32 of word j/32.  z_out (may be NULL) receives the
 * pre-activation values, for the tests.
 *
 * In eval mode save_mean/save_rstd receive running_mean and (running_var+eps)^-1/2.
 */
void oracle_batchnorm_fwd(int64_t n, int64_t c, int64_t l, const double *x,
                          const double *res, const double *w, const double *b,
                          double eps, double momentum, int training, int act,
                          double act_param, double *running_mean, double *running_var,
                          double *y, double *save_mean, double *save_rstd,
                          uint32_t *act_mask, double *z_out)
{
    const int64_t m = n * l;
    const int64_t words = mask_words_per_segment(l);
    if (act_mask && act == ORACLE_ACT_RELU)
        memset(act_mask, 0, (size_t)(n * c * words) * sizeof(uint32_t));

    for (int64_t ch = 0; ch < c; ++ch) {
        double mu, rs;
        if (training) {
            double sum = 0.0;
            for (int64_t i = 0; i < n; ++i)
                for (int64_t j = 0; j < l; ++j)
                    sum += x[(i * c + ch) * l + j];
            mu = sum / (double)m;
            double ssd = 0.0;
            for (int64_t i = 0; i < n; ++i)
                for (int64_t j = 0; j < l; ++j) {
                    double d = x[(i * c + ch) * l + j] - mu;
                    ssd += d * d;
                }
            double var_biased = ssd / (double)m;
            double var_unbiased = ssd / (double)(m - 1);
            rs = 1.0 / sqrt(var_biased + eps);
            if (running_mean)
                running_mean[ch] = (1.0 - momentum) * running_mean[ch] + momentum * mu;
            if (running_var)
                running_var[ch] = (1.0 - momentum) * running_var[ch] + momentum * var_unbiased;
        } else {
            mu = running_mean[ch];
            rs = 1.0 / sqrt(running_var[ch] + eps);
        }
        if (save_mean) save_mean[ch] = mu;
        if (save_rstd) save_rstd[ch] = rs;

        double wc = w ? w[ch] : 1.0;
        double bc = b ? b[ch] : 0.0;
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = 0; j < l; ++j) {
                int64_t e = (i * c + ch) * l + j;
                double z = (x[e] - mu) * rs * wc + bc;
                if (res) z += res[e];
                if (z_out) z_out[e] = z;
                y[e] = act_forward(act, act_param, z);
                if (act_mask && act == ORACLE_ACT_RELU && z > 0.0)
                    act_mask[(i * c + ch) * words + j / 32] |= (uint32_t)1u << (j % 32);
            }
    }
}

/*
 * [NK] section "BatchNorm：按特征并行 + 激活融合", last sentences: with a fused
 * activation the backward first runs the activation backward to recover the
 * pre-activation gradient dz, then the BatchNorm gradient.  Statistics are
 * recomputed from x (training) or taken from the running buffers (eval).
 *   dz   = dy * act'(z)          (ReLU': the act_mask bit when act_mask != NULL)
 *   dres = dz
 *   db   = sum dz,  dw = sum dz * xhat           (per channel)
 *   dx   = w * rstd * (dz - db/M - xhat * dw/M)   (training)
 *   dx   = w * rstd * dz                          (eval)
 */
void oracle_batchnorm_bwd(int64_t n, int64_t c, int64_t l, const double *dy,
                          const double *x, const double *res, const double *w,
                          const double *b, const double *running_mean,
                          const double *running_var, double eps, int training,
                          int act, double act_param, const uint32_t *act_mask, double *dx,
                          double *dres, double *dw, double *db)
{
    const int64_t m = n * l;
    const int64_t words = mask_words_per_segment(l);

    for (int64_t ch = 0; ch < c; ++ch) {
        double mu, rs;
        if (training) {
            double sum = 0.0;
            for (int64_t i = 0; i < n; ++i)
                for (int64_t j = 0; j < l; ++j)
                    sum += x[(i * c + ch) * l + j];
            mu = sum / (double)m;
            double ssd = 0.0;
            for (int64_t i = 0; i < n; ++i)
                for (int64_t j = 0; j < l; ++j) {
                    double d = x[(i * c + ch) * l + j] - mu;
                    ssd += d * d;
                }
            rs = 1.0 / sqrt(ssd / (double)m + eps);
        } else {
            mu = running_mean[ch];
            rs = 1.0 / sqrt(running_var[ch] + eps);
        }
        double wc = w ? w[ch] : 1.0;
        double bc = b ? b[ch] : 0.0;

        /* activation backward: recover dz from dy */
        double sum_dz = 0.0, sum_dz_xhat = 0.0;
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = 0; j < l; ++j) {
                int64_t e = (i * c + ch) * l + j;
                double xhat = (x[e] - mu) * rs;
                double z = xhat * wc + bc + (res ? res[e] : 0.0);
                double d;
                if (act == ORACLE_ACT_RELU && act_mask)
                    d = (act_mask[(i * c + ch) * words + j / 32] >> (j % 32)) & 1u ? 1.0 : 0.0;
                else
                    d = act_derivative(act, act_param, z);
                double dz = dy[e] * d;
                if (dres) dres[e] = dz;
                sum_dz += dz;
                sum_dz_xhat += dz * xhat;
            }
        if (db) db[ch] = sum_dz;
        if (dw) dw[ch] = sum_dz_xhat;

        /* BatchNorm backward */
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = 0; j < l; ++j) {
                int64_t e = (i * c + ch) * l + j;
                double xhat = (x[e] - mu) * rs;
                double z = xhat * wc + bc + (res ? res[e] : 0.0);
                double d;
                if (act == ORACLE_ACT_RELU && act_mask)
                    d = (act_mask[(i * c + ch) * words + j / 32] >> (j % 32)) & 1u ? 1.0 : 0.0;
                else
                    d = act_derivative(act, act_param, z);
                double dz = dy[e] * d;
                if (training)
                    dx[e] = wc * rs * (dz - sum_dz / (double)m - xhat * sum_dz_xhat / (double)m);
                else
                    dx[e] = wc * rs * dz;
            }
    }
}

/* ------------------------------------------------------------------------ */
/* Activation with fused dropout                                             */
/* ------------------------------------------------------------------------ */

/*
 * The counter-based generator, Philox4x32 with 10 rounds, from its published
 * definition (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
 * 1, 2, 3", SC 2011).  A round forms the 64-bit products of counter words 0 and 2
 * with the multipliers 0xD2511F53 and 0xCD9E8D57 and replaces the counter by
 *   (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
 * between rounds the key is advanced by the Weyl increments 0x9E3779B9 and
 * 0xBB67AE85.  The output is the counter after the tenth round.
 */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/*
 * [AF] section "四、Dropout 融合的关键：可复现的随机掩码": an element's random value is
 * a function of the seed and the element's offset alone, so the backward rebuilds
 * the forward's mask from the seed; an element is dropped when its value is below
 * drop_p and kept elements are divided by (1 - drop_p) (inverted dropout).  The
 * generator and the offset-to-counter mapping are this library's reading (header).
 */
static int dropout_keep(uint32_t seed, int64_t e, double drop_p)
{
    uint32_t ctr[4] = {(uint32_t)((uint64_t)e >> 2), (uint32_t)((uint64_t)e >> 34), 0u, 0u};
    uint32_t key[2] = {seed, 0u};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    float u = (float)(out[e & 3] >> 8) * (1.0f / 16777216.0f);
    return !(u < (float)drop_p);
}

/* Arrays hold elements first .. first + count - 1 of the tensor: the random
 * value belongs to the element's offset in the whole tensor. */
void oracle_dropout_mask(int64_t count, int64_t first, double drop_p, uint32_t seed, uint8_t *keep)
{
    for (int64_t i = 0; i < count; ++i) keep[i] = (uint8_t)dropout_keep(seed, first + i, drop_p);
}

/* [AF] sections "三、融合内核的骨架" and "四": the activation is applied first and its
 * result goes through dropout in the same pass: y = act(x) / (1 - p) where kept,
 * 0 where dropped. */
void oracle_act_dropout_fwd(int64_t count, int64_t first, const double *x, int act,
                            double act_param, double drop_p, uint32_t seed, double *y)
{
    for (int64_t i = 0; i < count; ++i) {
        double a = act_forward(act, act_param, x[i]);
        y[i] = dropout_keep(seed, first + i, drop_p) ? a / (1.0 - drop_p) : 0.0;
    }
}

/* [AF] section "五、反向传播融合同样成立": the output gradient goes through the
 * dropout gradient (the same mask rebuilt from the seed, the same 1/(1 - p)
 * scale) and is multiplied by the activation's derivative at the saved input:
 * dx = dy / (1 - p) * act'(x) where kept, 0 where dropped. */
void oracle_act_dropout_bwd(int64_t count, int64_t first, const double *dy, const double *x,
                            int act, double act_param, double drop_p, uint32_t seed,
                            double *dx)
{
    for (int64_t i = 0; i < count; ++i) {
        if (dropout_keep(seed, first + i, drop_p))
            dx[i] = dy[i] / (1.0 - drop_p) * act_derivative(act, act_param, x[i]);
        else
            dx[i] = 0.0;
    }
}
