// activation.cuh -- the activations that the BatchNorm kernels and the
// activation-dropout kernels fuse, in fp32: ReLU, GELU (erf form), SiLU
// and Mish, with their derivatives at the pre-activation value.
//
// The activation-dropout article ("算子融合实战：attorch激活函数与Dropout融合核的完整
// 实现原理", section "五、反向传播融合同样成立") takes the derivative at the saved
// input and uses the error-function GELU; the normalization article's BatchNorm
// section lists SiLU and Mish among the fusable activations (their formulas
// are the standard ones: silu(z) = z*sigmoid(z), mish(z) = z*tanh(softplus(z))),
// and the activation article's list (section 六) has leaky_relu, elu and celu,
// whose parameter prm (slope, alpha) the article encodes in the name:
// leaky_relu(z) = z > 0 ? z : prm*z, elu(z) = z > 0 ? z : prm*(e^z - 1),
// celu(z) = z > 0 ? z : prm*(e^(z/prm) - 1); it also names sigmoid and SELU
// (section 七), selu(z) = L*z for z > 0, else L*A*(e^z - 1), with the constants
// of Klambauer et al., "Self-Normalizing Neural Networks" (2017).
#pragma once

#include "libnorm.h"

namespace nrm {

constexpr float kSeluLambda = 1.0507009873554805f;
constexpr float kSeluAlpha = 1.6732632423543772f;
// The template value of the kernels that dispatch the less common activations
// (sigmoid, CELU, SELU) at run time, so that each does not cost a set of
// instantiations.
constexpr int kActGeneric = 100;

// softplus(z) = log(1 + e^z), without overflow for large z
__device__ __forceinline__ float softplus_f(float z) {
    return z > 0.f ? z + log1pf(expf(-z)) : log1pf(expf(z));
}

// The standard normal CDF Phi(z) and the Gaussian exp(-z^2/2), branch-free,
// for GELU and its derivative.  erfc(x) for x >= 0 follows Abramowitz and
// Stegun, Handbook of Mathematical Functions, formula 7.1.26 (Hastings'
// rational approximation, |error of erf| <= 1.5e-7):
//   erfc(x) = t*(a1 + t*(a2 + t*(a3 + t*(a4 + t*a5))))*exp(-x^2), t = 1/(1 + p*x),
// with x = |z|/sqrt(2), so Phi(z) = 1 - erfc(x)/2 for z >= 0 and erfc(x)/2
// below; the coefficients are halved (exactly) to give erfc(x)/2 directly,
// p*x is taken as (p/sqrt(2))*|z| and exp(-z^2/2) as 2^(z*(-log2(e)/2)*z).
// In fp32 the GELU built on it is within 5e-7 of the exact value over
// [-12, 12], as close as the exact erf rounded to fp32 (one polynomial, one
// reciprocal and one exponential: the library erf takes two code paths that a
// warp with mixed |z| runs both of).
constexpr float kCdfP = 0.3275911f * 0.70710678118654752f;
constexpr float kCdfA1 = 0.5f * 0.254829592f;
constexpr float kCdfA2 = 0.5f * -0.284496736f;
constexpr float kCdfA3 = 0.5f * 1.421413741f;
constexpr float kCdfA4 = 0.5f * -1.453152027f;
constexpr float kCdfA5 = 0.5f * 1.061405429f;
constexpr float kNegHalfLog2e = -0.72134752044448170f;  // -log2(e)/2
constexpr float kInvSqrt2Pi = 0.39894228040143268f;     // 1/sqrt(2*pi)

// The reciprocal and base-2 exponential as the single approximate hardware
// instructions (PTX rcp.approx, ex2.approx; about 1 and 2 ulp), subnormal
// results flushed to zero.  Here 1 + p*x >= 1, so t is flushed only when it is
// below 2^-126 (Phi is then 0 or 1 exactly in fp32), and exp(-z^2/2) only for
// |z| > 13.2, where GELU and GELU' change by less than 1e-36.
__device__ __forceinline__ float rcp_approx_ftz(float v) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float exp2_approx_ftz(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

struct NormalCdf {
    float cdf;    // Phi(z)
    float gauss;  // exp(-z^2/2)
};
__device__ __forceinline__ NormalCdf normal_cdf(float z) {
    const float t = rcp_approx_ftz(fmaf(fabsf(z), kCdfP, 1.f));
    float y = fmaf(kCdfA5, t, kCdfA4);
    y = fmaf(y, t, kCdfA3);
    y = fmaf(y, t, kCdfA2);
    y = fmaf(y, t, kCdfA1);
    const float gauss = exp2_approx_ftz(z * kNegHalfLog2e * z);
    const float q = t * y * gauss;  // erfc(|z|/sqrt(2))/2 = Phi(-|z|)
    return NormalCdf{z >= 0.f ? 1.f - q : q, gauss};
}

// The same for a pair of z on packed fp32 (FFMA2/FMUL2): the same IEEE
// operations in the same order as normal_cdf, so each lane's result is
// bitwise the scalar one.
__device__ __forceinline__ float2 act_pair(float v) { return make_float2(v, v); }
struct NormalCdf2 {
    float2 cdf;
    float2 gauss;
};
__device__ __forceinline__ NormalCdf2 normal_cdf2(float2 z) {
    const float2 d = __ffma2_rn(make_float2(fabsf(z.x), fabsf(z.y)), act_pair(kCdfP), act_pair(1.f));
    const float2 t = make_float2(rcp_approx_ftz(d.x), rcp_approx_ftz(d.y));
    float2 y = __ffma2_rn(act_pair(kCdfA5), t, act_pair(kCdfA4));
    y = __ffma2_rn(y, t, act_pair(kCdfA3));
    y = __ffma2_rn(y, t, act_pair(kCdfA2));
    y = __ffma2_rn(y, t, act_pair(kCdfA1));
    const float2 e = __fmul2_rn(__fmul2_rn(z, act_pair(kNegHalfLog2e)), z);
    const float2 gauss = make_float2(exp2_approx_ftz(e.x), exp2_approx_ftz(e.y));
    const float2 q = __fmul2_rn(__fmul2_rn(t, y), gauss);
    const float2 c = __fadd2_rn(act_pair(1.f), make_float2(-q.x, -q.y));
    return NormalCdf2{make_float2(z.x >= 0.f ? c.x : q.x, z.y >= 0.f ? c.y : q.y), gauss};
}

// GELU(z) = z*Phi(z) and GELU'(z) = Phi(z) + z*phi(z), phi the normal density.
__device__ __forceinline__ float gelu_f(float z) { return z * normal_cdf(z).cdf; }
__device__ __forceinline__ float gelu_grad_f(float z) {
    const NormalCdf n = normal_cdf(z);
    return fmaf(z * n.gauss, kInvSqrt2Pi, n.cdf);
}
__device__ __forceinline__ float2 gelu2_f(float2 z) { return __fmul2_rn(z, normal_cdf2(z).cdf); }
__device__ __forceinline__ float2 gelu_grad2_f(float2 z) {
    const NormalCdf2 n = normal_cdf2(z);
    return __ffma2_rn(__fmul2_rn(z, n.gauss), act_pair(kInvSqrt2Pi), n.cdf);
}

__device__ __forceinline__ float act_forward(int act, float z, float prm) {
    if (act == NRM_ACT_RELU) return z > 0.f ? z : 0.f;
    if (act == NRM_ACT_LEAKY_RELU) return z > 0.f ? z : prm * z;
    if (act == NRM_ACT_ELU) return z > 0.f ? z : prm * expm1f(z);
    if (act == NRM_ACT_SIGMOID) return 1.f / (1.f + expf(-z));
    if (act == NRM_ACT_CELU) return z > 0.f ? z : prm * expm1f(z / prm);
    if (act == NRM_ACT_SELU) return z > 0.f ? kSeluLambda * z : (kSeluLambda * kSeluAlpha) * expm1f(z);
    if (act == NRM_ACT_RELU6) return z < 0.f ? 0.f : (z > 6.f ? 6.f : z);
    if (act == NRM_ACT_HARDTANH) return z < -1.f ? -1.f : (z > 1.f ? 1.f : z);
    if (act == NRM_ACT_GELU) return gelu_f(z);
    if (act == NRM_ACT_SILU) return z / (1.f + expf(-z));
    if (act == NRM_ACT_MISH) return z * tanhf(softplus_f(z));
    return z;
}

// Derivative at the pre-activation value z (ReLU'(0) = 0).
__device__ __forceinline__ float act_derivative(int act, float z, float prm) {
    if (act == NRM_ACT_RELU) return z > 0.f ? 1.f : 0.f;
    if (act == NRM_ACT_LEAKY_RELU) return z > 0.f ? 1.f : prm;
    if (act == NRM_ACT_ELU) return z > 0.f ? 1.f : prm * expf(z);
    if (act == NRM_ACT_SIGMOID) {
        const float sg = 1.f / (1.f + expf(-z));
        return sg * (1.f - sg);
    }
    if (act == NRM_ACT_CELU) return z > 0.f ? 1.f : expf(z / prm);
    if (act == NRM_ACT_SELU) return z > 0.f ? kSeluLambda : (kSeluLambda * kSeluAlpha) * expf(z);
    if (act == NRM_ACT_RELU6) return (z > 0.f && z < 6.f) ? 1.f : 0.f;
    if (act == NRM_ACT_HARDTANH) return (z > -1.f && z < 1.f) ? 1.f : 0.f;
    if (act == NRM_ACT_GELU) return gelu_grad_f(z);
    if (act == NRM_ACT_SILU) {
        const float sg = 1.f / (1.f + expf(-z));
        return sg * fmaf(z, 1.f - sg, 1.f);
    }
    if (act == NRM_ACT_MISH) {
        const float t = tanhf(softplus_f(z));
        const float sg = 1.f / (1.f + expf(-z));
        return fmaf(z * sg, 1.f - t * t, t);
    }
    return 1.f;
}

// The same for an activation fixed at compile time (the ring and group
// kernels are instantiated per activation, so the hot loops carry one).
template <int ACT>
__device__ __forceinline__ float act_forward_c(float z, float prm, int act_rt) {
    if constexpr (ACT == NRM_ACT_RELU) return z > 0.f ? z : 0.f;
    else if constexpr (ACT == NRM_ACT_NONE) return z;
    else if constexpr (ACT == kActGeneric) return act_forward(act_rt, z, prm);
    else return act_forward(ACT, z, prm);
}
template <int ACT>
__device__ __forceinline__ float act_derivative_c(float z, float prm, int act_rt) {
    if constexpr (ACT == NRM_ACT_RELU) return z > 0.f ? 1.f : 0.f;
    else if constexpr (ACT == NRM_ACT_NONE) return 1.f;
    else if constexpr (ACT == kActGeneric) return act_derivative(act_rt, z, prm);
    else return act_derivative(ACT, z, prm);
}

// Both lanes of a pair: GELU on packed fp32, the others lane by lane.
template <int ACT>
__device__ __forceinline__ float2 act_forward2_c(float2 z, float prm, int act_rt) {
    if constexpr (ACT == NRM_ACT_GELU) return gelu2_f(z);
    else return make_float2(act_forward_c<ACT>(z.x, prm, act_rt), act_forward_c<ACT>(z.y, prm, act_rt));
}
template <int ACT>
__device__ __forceinline__ float2 act_derivative2_c(float2 z, float prm, int act_rt) {
    if constexpr (ACT == NRM_ACT_GELU) return gelu_grad2_f(z);
    else return make_float2(act_derivative_c<ACT>(z.x, prm, act_rt), act_derivative_c<ACT>(z.y, prm, act_rt));
}

// Calls f(std::integral_constant-like tag) with the activation as a compile-time value.
template <int A>
struct ActTag {
    static constexpr int value = A;
};
template <typename F>
auto with_act(int act, F&& f) {
    switch (act) {
    case NRM_ACT_RELU: return f(ActTag<NRM_ACT_RELU>{});
    case NRM_ACT_GELU: return f(ActTag<NRM_ACT_GELU>{});
    case NRM_ACT_SILU: return f(ActTag<NRM_ACT_SILU>{});
    case NRM_ACT_MISH: return f(ActTag<NRM_ACT_MISH>{});
    case NRM_ACT_LEAKY_RELU: return f(ActTag<NRM_ACT_LEAKY_RELU>{});
    case NRM_ACT_ELU: return f(ActTag<NRM_ACT_ELU>{});
    case NRM_ACT_SIGMOID:
    case NRM_ACT_CELU:
    case NRM_ACT_SELU:
    case NRM_ACT_RELU6:
    case NRM_ACT_HARDTANH: return f(ActTag<kActGeneric>{});
    default: return f(ActTag<NRM_ACT_NONE>{});
    }
}

}  // namespace nrm
