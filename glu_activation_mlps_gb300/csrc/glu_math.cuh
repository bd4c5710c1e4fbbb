// fp32 device math of the four gated activations, forward and backward.
//
// Formulas: "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel" (Required
// reasoning process steps 5 and 7; Common failure modes, "GELU variant
// mismatch") and "Kernel Profile: SwiGLU (Tier 1 - Element-wise)" (Backward
// Pass).  Everything is evaluated in fp32 ("Kernel design rules": sigmoid and
// GELU in fp32 for fp16/bf16 inputs), without flush-to-zero.
//
// Rewrites used for accuracy (each an exact identity):
//   sigmoid(x)          = 1/(1+e) for x >= 0, e/(1+e) for x < 0, e = exp(-|x|)
//                         (exp never overflows; "Kernel design rules" ask for a
//                         form that is stable for very negative x)
//   silu'(x)            = sigmoid + x*sigmoid*(1 - sigmoid)
//                       = (1 + e + x e) / (1+e)^2            for x >= 0
//                       = e (1 + x + e) / (1+e)^2            for x < 0
//                         (the only cancellation left is (1 + x) + e near the
//                         root x* = -1.2785, where 1 + x is exact in fp32)
//   0.5 (1 + erf(x/sqrt2)) = Phi(x) = 1 - Phi(-x), with the lower tail Phi(-|x|)
//                         computed directly (no cancellation for x < 0)
//   0.5 (1 + tanh(u))   = sigmoid(2u)           (no cancellation for u < 0)
//
// Near the root x* of act' (silu' at -1.2785, both GELU' near -0.752) the two
// terms of act' cancel, and the absolute error of any fp32 evaluation of them
// (~1e-8) becomes a large relative error of act' itself.  Within |x - x*| <
// 2^-7 act' is therefore taken from its Taylor series about x*, evaluated in
// u = x - x* (exact in fp32 there, by Sterbenz's lemma): the series has no
// cancellation, and its truncation error at degree 4 is ~1e-10 relative.  The
// coefficients are act^(k+1)(x*)/k!, from the closed forms above.
//
// `Exact` selects the variant used when the storage dtype is fp32: there the
// rounding of the scaled arguments (the tanh polynomial, x^2) would be
// amplified by up to 2z^2 in the tails, so those arguments are carried as
// (hi, lo) float pairs and the first-order effect of `lo` is applied
// analytically.  For fp16/bf16 outputs the plain fp32 forms are far below
// half an output ulp and the corrections are skipped; there exp(-t) is taken
// as 2^(-t log2 e) with the hardware base-2 exponential (ex2.approx, relative
// error ~2^-22, subnormal results kept) and 1/(1+e), whose argument lies in
// [1, 2], with the hardware reciprocal (rcp.approx, ~1 ulp).
#pragma once
#include <cuda_runtime.h>
#include <math.h>

namespace glu {

struct SigmoidParts {
    float e;      // exp(-|x|), in (0, 1]
    float r;      // 1 / (1 + e), in [0.5, 1)
    float s;      // sigmoid(x)
    float sm;     // 1 - sigmoid(x) = sigmoid(-x), formed without cancellation
};

// e^(-t) for t >= 0.
template <bool Exact>
__device__ __forceinline__ float exp_neg(float t)
{
    if (Exact) return expf(-t);
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(t * -1.44269504f));   // -t log2(e)
    return y;
}

// 1/d for d in [1, 2] (never subnormal, so flush-to-zero cannot change it).
template <bool Exact>
__device__ __forceinline__ float recip_1_2(float d)
{
    if (Exact) return __frcp_rn(d);
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
    return y;
}

template <bool Exact>
__device__ __forceinline__ SigmoidParts sigmoid_parts(float x)
{
    SigmoidParts p;
    p.e = exp_neg<Exact>(fabsf(x));
    p.r = recip_1_2<Exact>(1.0f + p.e);
    float er = __fmul_rn(p.e, p.r);
    p.s = x >= 0.0f ? p.r : er;
    p.sm = x >= 0.0f ? er : p.r;
    return p;
}

// (hi, lo) splits of constants: hi is the nearest float, lo the nearest float
// to the remainder.
constexpr float kInvSqrt2Pi = 0.398942292f;         // 1/sqrt(2 pi)
// tanh form: w(x) = 2u(x) = C1 x + C3 x^3 with C1 = 2 sqrt(2/pi), C3 = C1 * 0.044715
constexpr float kC1Hi = 1.59576917f;
constexpr float kC1Lo = -4.53406805e-08f;
constexpr float kC3Hi = 0.0713548139f;
constexpr float kC3Lo = 2.39883247e-09f;

// act'(x) = u (c1 + u (c2 + u (c3 + u c4))), u = x - x*, for |u| < kRootRadius.
// x* = hi + lo (hi the nearest float).
constexpr float kRootRadius = 0.0078125f;   // 2^-7
struct RootSeries {
    float hi, lo, c1, c2, c3, c4;
};
__host__ __device__ constexpr RootSeries silu_root()
{
    return {-1.27846456f, 1.29792825e-08f, 2.17811706e-01f,
            1.46648797e-01f, 1.88748142e-02f, -1.52226552e-02f};
}
__host__ __device__ constexpr RootSeries gelu_erf_root()
{
    return {-0.751791537f, 1.21144499e-08f, 4.31493992e-01f,
            3.88284983e-01f, -1.81996764e-02f, -1.14008233e-01f};
}
__host__ __device__ constexpr RootSeries gelu_tanh_root()
{
    return {-0.752461433f, 1.13396279e-08f, 4.30400091e-01f,
            3.87518446e-01f, -1.57828535e-02f, -1.13944483e-01f};
}

// Replaces *dact by the series when x is within kRootRadius of the root.
__device__ __forceinline__ void root_series(float x, const RootSeries r, float *dact)
{
    const float u = __fsub_rn(__fsub_rn(x, r.hi), r.lo);
    if (fabsf(u) < kRootRadius) *dact = u * fmaf(u, fmaf(u, fmaf(u, r.c4, r.c3), r.c2), r.c1);
}

// The cheap test the kernels run on every element; the series itself
// (root_series) is only evaluated for the rare elements that pass it.  The
// test is slightly wider than kRootRadius, so it never misses one.
__device__ __forceinline__ bool near_root(float x, const RootSeries r)
{
    return fabsf(x - r.hi) < 1.0625f * kRootRadius;
}

// Lower tail of the standard normal:
//     Phi(-x) = exp(-x^2/2) * t * P(t),  t = 1/(1 + 0.3 x),  x >= 0,
// with P a polynomial fitted to the exact ratio (Mills' ratio form): degree 7
// for bf16/f16 storage (relative error of P <= 2.7e-6 in float32), degree 10
// for f32 storage (<= 1.4e-7).  The coefficients are produced by
// gen_phi_tail.py next to this file.  The exponential is returned too: it is
// also sqrt(2 pi) phi(x), the density the GeGLU-erf backward needs.  For f32
// storage, x^2 is carried as p + pe (exact) and exp(-x^2/2) =
// exp(-p/2) (1 - pe/2), and 1/(1 + 0.3 x) is rounded correctly.
constexpr float kPhiTailC = 0.3f;
__host__ __device__ constexpr float phi_tail_coef(bool exact, int i)
{
    constexpr float p7[8] = {1.196823716e-01f, 1.197295263e-01f, 1.077751145e-01f,
                             9.759789705e-02f, 1.416620519e-02f, 1.230392978e-01f,
                             -1.036966890e-01f, 2.170499042e-02f};
    constexpr float p10[11] = {1.196826845e-01f, 1.196820512e-01f, 1.089364216e-01f,
                               8.699049801e-02f, 6.073883548e-02f, 1.550978515e-02f,
                               2.356493101e-02f, -3.294012696e-02f, -3.021260537e-02f,
                               3.880830109e-02f, -1.076079253e-02f};
    return exact ? p10[i] : p7[i];
}

struct PhiTail {
    float q;   // Phi(-x)
    float e;   // exp(-x^2 / 2)
};

template <bool Exact>
__device__ __forceinline__ PhiTail phi_tail(float x)   // x = |a| >= 0
{
    PhiTail r;
    float t;
    if (Exact) {
        const float xc = fminf(x, 40.0f);                  // Phi(-40) is 0 in fp32
        const float p = __fmul_rn(xc, xc);
        r.e = expf(-0.5f * p) * (1.0f - 0.5f * fmaf(xc, xc, -p));
        t = __frcp_rn(fmaf(kPhiTailC, x, 1.0f));
    } else {
        r.e = exp_neg<false>(0.5f * x * x);
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(kPhiTailC, x, 1.0f)));   // t in (0, 1]
    }
    constexpr int kDeg = Exact ? 10 : 7;
    float poly = phi_tail_coef(Exact, kDeg);
#pragma unroll
    for (int i = kDeg - 1; i >= 0; --i) poly = fmaf(poly, t, phi_tail_coef(Exact, i));
    r.q = r.e * (t * poly);
    return r;
}

// w(x) = 2 sqrt(2/pi) (x + 0.044715 x^3) as hi (+ lo when Exact).
template <bool Exact>
__device__ __forceinline__ float tanh_arg(float x, float *lo)
{
    float p = __fmul_rn(x, x);
    float inner = fmaf(kC3Hi, p, kC1Hi);     // C1 + C3 x^2
    float w = __fmul_rn(x, inner);
    *lo = 0.0f;
    if (Exact && fabsf(x) < 1.0e4f) {        // beyond, sigmoid(w) is exactly 0 or 1
        float pe = fmaf(x, x, -p);                         // x^2 = p + pe exactly
        float q = __fmul_rn(kC3Hi, p);
        float qe = fmaf(kC3Hi, p, -q);                     // C3hi p = q + qe exactly
        float s = __fadd_rn(kC1Hi, q);                     // two-sum of C1hi + q
        float bb = __fsub_rn(s, kC1Hi);
        float se = __fadd_rn(__fsub_rn(kC1Hi, __fsub_rn(s, bb)), __fsub_rn(q, bb));
        float slo = se + qe + kC3Hi * pe + kC3Lo * p + kC1Lo;
        float wh = __fmul_rn(x, s);
        float we = fmaf(x, s, -wh) + x * slo;
        w = wh;
        *lo = we;
    }
    return w;
}

// --------------------------------------------------------------------------
// Each activation: act(x) for the forward, and (act, act') for the backward.

struct Silu {
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        SigmoidParts p = sigmoid_parts<Exact>(x);
        return x * p.s;
    }
    // act and act' without the root series (see bwd)
    template <bool Exact>
    __device__ __forceinline__ static void bwd_main(float x, float *act, float *dact)
    {
        SigmoidParts p = sigmoid_parts<Exact>(x);
        *act = x * p.s;
        float num;
        if (Exact) {
            num = x >= 0.0f ? fmaf(x, p.e, 1.0f + p.e)          // 1 + e + x e
                            : p.e * ((1.0f + x) + p.e);         // e (1 + x + e)
        } else {
            // the same numerator as (1+e) m + x e, m = 1 (x >= 0) or e (x < 0):
            // one FMA; its cancellation near the root is left to the series
            const float d = 1.0f + p.e;
            num = fmaf(x, p.e, d * (x >= 0.0f ? 1.0f : p.e));
        }
        *dact = num * (p.r * p.r);
    }
    __device__ __forceinline__ static bool near_root(float x) { return glu::near_root(x, silu_root()); }
    __device__ __forceinline__ static void fix_root(float x, float *dact) { root_series(x, silu_root(), dact); }
    template <bool Exact>
    __device__ __forceinline__ static void bwd(float x, float *act, float *dact)
    {
        bwd_main<Exact>(x, act, dact);
        fix_root(x, dact);
    }
};

struct GeluErf {
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        const float q = phi_tail<Exact>(fabsf(x)).q;       // Phi(-|x|)
        return x * (x <= 0.0f ? q : 1.0f - q);              // x Phi(x)
    }
    template <bool Exact>
    __device__ __forceinline__ static void bwd_main(float x, float *act, float *dact)
    {
        const PhiTail t = phi_tail<Exact>(fabsf(x));
        const float cdf = x <= 0.0f ? t.q : 1.0f - t.q;     // Phi(x)
        *act = x * cdf;
        *dact = fmaf(x, kInvSqrt2Pi * t.e, cdf);            // Phi + x phi
    }
    __device__ __forceinline__ static bool near_root(float x) { return glu::near_root(x, gelu_erf_root()); }
    __device__ __forceinline__ static void fix_root(float x, float *dact) { root_series(x, gelu_erf_root(), dact); }
    template <bool Exact>
    __device__ __forceinline__ static void bwd(float x, float *act, float *dact)
    {
        bwd_main<Exact>(x, act, dact);
        fix_root(x, dact);
    }
};

struct GeluTanh {
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        float lo;
        float w = tanh_arg<Exact>(x, &lo);
        SigmoidParts p = sigmoid_parts<Exact>(w);
        float s = p.s;
        if (Exact) s = fmaf(s * p.sm, lo, s);              // sigmoid(w + lo)
        return x * s;
    }
    __device__ __forceinline__ static bool near_root(float x) { return glu::near_root(x, gelu_tanh_root()); }
    __device__ __forceinline__ static void fix_root(float x, float *dact) { root_series(x, gelu_tanh_root(), dact); }
    template <bool Exact>
    __device__ __forceinline__ static void bwd(float x, float *act, float *dact)
    {
        bwd_main<Exact>(x, act, dact);
        fix_root(x, dact);
    }
    template <bool Exact>
    __device__ __forceinline__ static void bwd_main(float x, float *act, float *dact)
    {
        float lo;
        float w = tanh_arg<Exact>(x, &lo);
        SigmoidParts p = sigmoid_parts<Exact>(w);
        float s = p.s;
        if (Exact) s = fmaf(s * p.sm, lo, s);
        // Beyond |x| = 1e4 either 1 - sigmoid(w) or sigmoid(w) is exactly 0, so
        // clamping x inside the bracket leaves act' unchanged and keeps it finite.
        float xc = fminf(fmaxf(x, -1.0e4f), 1.0e4f);
        float dw = fmaf(3.0f * kC3Hi, xc * xc, kC1Hi);      // w'(x) = C1 + 3 C3 x^2
        *act = x * s;
        // d/dx [x sigmoid(w)] = sigmoid(w) (1 + x (1 - sigmoid(w)) w')
        *dact = s * fmaf(xc * p.sm, dw, 1.0f);
    }
};

struct Relu {
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        return x > 0.0f ? x : (x != x ? x : 0.0f);          // NaN propagates
    }
    template <bool Exact>
    __device__ __forceinline__ static void bwd_main(float x, float *act, float *dact)
    {
        *act = x > 0.0f ? x : (x != x ? x : 0.0f);
        *dact = x > 0.0f ? 1.0f : (x != x ? x : 0.0f);      // 0 at x == 0
    }
    __device__ __forceinline__ static bool near_root(float) { return false; }   // act' has no root
    __device__ __forceinline__ static void fix_root(float, float *) {}
    template <bool Exact>
    __device__ __forceinline__ static void bwd(float x, float *act, float *dact)
    {
        bwd_main<Exact>(x, act, dact);
    }
};

}  // namespace glu
