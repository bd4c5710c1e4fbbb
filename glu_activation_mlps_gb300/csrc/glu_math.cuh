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
// analytically.
//
// For fp16/bf16 outputs the plain fp32 forms are far below half an output ulp
// and the corrections are skipped.  That path works on PAIRS of elements (the
// two halves of a 32-bit storage word) with the packed fp32x2 add, multiply
// and fused multiply-add of sm_100 and later (one instruction for both
// elements, IEEE round-to-nearest, subnormals kept), which halves the
// arithmetic instructions a 16-bit element costs; a single element is the
// pair (x, x), so the vector body and the scalar row tails give identical
// bits.  There exp(-t) is the square of 2^(-t log2(e) / 2) from the hardware
// base-2 exponential with flush-to-zero (ex2.approx.ftz, relative error
// ~2^-22): the half exponent stays a normal number wherever the result
// matters, and the square, an IEEE multiply, reaches the subnormal range
// correctly (silu(-88) in bf16 needs e^-88 = 6e-39).  1/(1+e), whose argument
// lies in [1, 2], is the hardware reciprocal (rcp.approx, ~1 ulp).
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

// The scalar forms below serve f32 storage (Exact == true) only.
template <bool Exact>
__device__ __forceinline__ SigmoidParts sigmoid_parts(float x)
{
    static_assert(Exact, "16-bit storage takes sigmoid_pair");
    SigmoidParts p;
    p.e = expf(-fabsf(x));
    p.r = __frcp_rn(1.0f + p.e);                       // 1 + e in [1, 2]
    float er = __fmul_rn(p.e, p.r);
    p.s = x >= 0.0f ? p.r : er;
    p.sm = x >= 0.0f ? er : p.r;
    return p;
}

// ---------------------------------------------------------------- pairs
// Two fp32 values in one register pair, for the 16-bit storage path.

using f2 = float2;
__device__ __forceinline__ f2 splat(float v) { return make_float2(v, v); }
__device__ __forceinline__ f2 add2(f2 a, f2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ f2 mul2(f2 a, f2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ f2 abs2(f2 x) { return make_float2(fabsf(x.x), fabsf(x.y)); }

__device__ __forceinline__ float ex2_ftz(float h)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(h));
    return y;
}

__device__ __forceinline__ float rcp_ftz(float d)   // d in [1, 2]: never subnormal
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
    return y;
}

// 2^(2h), h <= 0, as the square of the hardware 2^h: 2^h is normal down to
// h = -126, so the result is right down to 2^-252 (0 below), subnormals
// included.
__device__ __forceinline__ f2 exp2_twice(f2 h)
{
    const f2 y = make_float2(ex2_ftz(h.x), ex2_ftz(h.y));
    return mul2(y, y);
}

constexpr float kNegHalfLog2e = -0.721347520f;      // -log2(e) / 2: e^-t = 2^(2 (t kNegHalfLog2e))

// sigmoid(w) = m r and sigmoid(-w) = m' r for a pair, with e = exp(-|w|),
// d = 1 + e, r = 1/d, m = 1 (w >= 0) or e (w < 0), m' the other one.
struct SigmoidPair {
    f2 e, d, r, m;
};

__device__ __forceinline__ SigmoidPair sigmoid_pair(f2 w)
{
    SigmoidPair p;
    p.e = exp2_twice(mul2(abs2(w), splat(kNegHalfLog2e)));
    p.d = add2(p.e, splat(1.0f));
    p.r = make_float2(rcp_ftz(p.d.x), rcp_ftz(p.d.y));
    p.m = make_float2(w.x >= 0.0f ? 1.0f : p.e.x, w.y >= 0.0f ? 1.0f : p.e.y);
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
//     Phi(-x) = exp(-x^2/2) * t * P(t),  t = 1/(1 + C x),  x >= 0,
// with P a polynomial fitted to the exact ratio (Mills' ratio form):
//   - degree 4, C = 0.4, for the forward on bf16/f16 storage (relative error
//     of P <= 9.5e-5: below a quarter of the f16 half-ulp 2^-12, a twentieth
//     of the bf16 one);
//   - degree 7, C = 0.3, for the backward on bf16/f16 storage (<= 2.7e-6:
//     next to the root of act' the terms Phi and x phi cancel and magnify the
//     error of Phi up to ~130 times before the root series takes over);
//   - degree 10, C = 0.3, for f32 storage (<= 1.4e-7).
// The coefficients are produced by gen_phi_tail.py next to this file.  The
// exponential is returned too: it is also sqrt(2 pi) phi(x), the density the
// GeGLU-erf backward needs.  For f32 storage, x^2 is carried as p + pe
// (exact) and exp(-x^2/2) = exp(-p/2) (1 - pe/2), and 1/(1 + 0.3 x) is
// rounded correctly.
constexpr float kPhiTailC = 0.3f;
constexpr float kPhiTailC4 = 0.4f;
__host__ __device__ constexpr float phi_tail_coef4(int i)
{
    constexpr float p4[5] = {1.595728099e-01f, 1.605101526e-01f, 1.205828786e-01f, 1.440442950e-01f,
                             -8.475755900e-02f};
    return p4[i];
}
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
    static_assert(Exact, "16-bit storage takes phi_tail_pair");
    PhiTail r;
    const float xc = fminf(x, 40.0f);                  // Phi(-40) is 0 in fp32
    const float p = __fmul_rn(xc, xc);
    r.e = expf(-0.5f * p) * (1.0f - 0.5f * fmaf(xc, xc, -p));
    const float t = __frcp_rn(fmaf(kPhiTailC, x, 1.0f));
    constexpr int kDeg = 10;
    float poly = phi_tail_coef(true, kDeg);
#pragma unroll
    for (int i = kDeg - 1; i >= 0; --i) poly = fmaf(poly, t, phi_tail_coef(true, i));
    r.q = r.e * (t * poly);
    return r;
}

template <int DEG>
__host__ __device__ constexpr float tail_coef(int i)
{
    if constexpr (DEG == 4) return phi_tail_coef4(i);
    else return phi_tail_coef(false, i);
}

struct PhiTailPair {
    f2 q;   // Phi(-x)
    f2 e;   // exp(-x^2 / 2)
};

// phi_tail for a pair, 16-bit storage: DEG = 4 (forward) or 7 (backward).
template <int DEG>
__device__ __forceinline__ PhiTailPair phi_tail_pair(f2 x)   // x = |a| >= 0
{
    static_assert(DEG == 4 || DEG == 7, "fitted degrees");
    constexpr float C = DEG == 4 ? kPhiTailC4 : kPhiTailC;
    PhiTailPair r;
    r.e = exp2_twice(mul2(mul2(x, x), splat(0.5f * kNegHalfLog2e)));   // e^(-x^2/2)
    const f2 d = fma2(x, splat(C), splat(1.0f));
    const f2 t = make_float2(rcp_ftz(d.x), rcp_ftz(d.y));                // (0, 1]
    f2 poly = splat(tail_coef<DEG>(DEG));
#pragma unroll
    for (int i = DEG - 1; i >= 0; --i) poly = fma2(poly, t, splat(tail_coef<DEG>(i)));
    r.q = mul2(r.e, mul2(t, poly));
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

// For 16-bit storage (Exact == false) every activation works on pairs
// (fwd2, bwd2); its scalar form is the pair (x, x), so that one element gets
// the same bits wherever it sits.

struct Silu {
    __device__ __forceinline__ static f2 fwd2(f2 x)
    {
        const SigmoidPair p = sigmoid_pair(x);
        return mul2(x, mul2(p.m, p.r));                     // x sigmoid(x)
    }
    // act and act' without the root series (see bwd)
    __device__ __forceinline__ static void bwd2(f2 x, f2 *act, f2 *dact)
    {
        const SigmoidPair p = sigmoid_pair(x);
        *act = mul2(x, mul2(p.m, p.r));
        // silu' = ((1+e) m + x e) / (1+e)^2, the numerator as one FMA; its
        // cancellation near the root is left to the series
        const f2 num = fma2(x, p.e, mul2(p.d, p.m));
        *dact = mul2(num, mul2(p.r, p.r));
    }
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        if (!Exact) return fwd2(splat(x)).x;
        SigmoidParts p = sigmoid_parts<true>(x);
        return x * p.s;
    }
    template <bool Exact>
    __device__ __forceinline__ static void bwd_main(float x, float *act, float *dact)
    {
        if (!Exact) {
            f2 a, d;
            bwd2(splat(x), &a, &d);
            *act = a.x;
            *dact = d.x;
            return;
        }
        SigmoidParts p = sigmoid_parts<true>(x);
        *act = x * p.s;
        const float num = x >= 0.0f ? fmaf(x, p.e, 1.0f + p.e)      // 1 + e + x e
                                    : p.e * ((1.0f + x) + p.e);     // e (1 + x + e)
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
    __device__ __forceinline__ static f2 cdf2(f2 x, f2 q)     // Phi(x) from q = Phi(-|x|)
    {
        const f2 upper = fma2(q, splat(-1.0f), splat(1.0f));  // 1 - q
        return make_float2(x.x <= 0.0f ? q.x : upper.x, x.y <= 0.0f ? q.y : upper.y);
    }
    __device__ __forceinline__ static f2 fwd2(f2 x)
    {
        const PhiTailPair t = phi_tail_pair<4>(abs2(x));
        return mul2(x, cdf2(x, t.q));                           // x Phi(x)
    }
    __device__ __forceinline__ static void bwd2(f2 x, f2 *act, f2 *dact)
    {
        const PhiTailPair t = phi_tail_pair<7>(abs2(x));
        const f2 cdf = cdf2(x, t.q);
        *act = mul2(x, cdf);
        *dact = fma2(x, mul2(splat(kInvSqrt2Pi), t.e), cdf);   // Phi + x phi
    }
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        if (!Exact) return fwd2(splat(x)).x;
        const float q = phi_tail<true>(fabsf(x)).q;        // Phi(-|x|)
        return x * (x <= 0.0f ? q : 1.0f - q);              // x Phi(x)
    }
    template <bool Exact>
    __device__ __forceinline__ static void bwd_main(float x, float *act, float *dact)
    {
        if (!Exact) {
            f2 a, d;
            bwd2(splat(x), &a, &d);
            *act = a.x;
            *dact = d.x;
            return;
        }
        const PhiTail t = phi_tail<true>(fabsf(x));
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
    __device__ __forceinline__ static f2 arg2(f2 x)          // w = x (C1 + C3 x^2)
    {
        return mul2(x, fma2(splat(kC3Hi), mul2(x, x), splat(kC1Hi)));
    }
    __device__ __forceinline__ static f2 fwd2(f2 x)
    {
        const SigmoidPair p = sigmoid_pair(arg2(x));
        return mul2(x, mul2(p.m, p.r));                     // x sigmoid(w)
    }
    __device__ __forceinline__ static void bwd2(f2 x, f2 *act, f2 *dact)
    {
        const f2 w = arg2(x);
        const SigmoidPair p = sigmoid_pair(w);
        const f2 s = mul2(p.m, p.r);                        // sigmoid(w)
        const f2 sm = mul2(make_float2(w.x >= 0.0f ? p.e.x : 1.0f, w.y >= 0.0f ? p.e.y : 1.0f), p.r);
        // clamping x leaves act' unchanged (see the scalar form) and finite
        const f2 xc = make_float2(fminf(fmaxf(x.x, -1.0e4f), 1.0e4f), fminf(fmaxf(x.y, -1.0e4f), 1.0e4f));
        const f2 dw = fma2(splat(3.0f * kC3Hi), mul2(xc, xc), splat(kC1Hi));
        *act = mul2(x, s);
        *dact = mul2(s, fma2(mul2(xc, sm), dw, splat(1.0f)));
    }
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        if (!Exact) return fwd2(splat(x)).x;
        float lo;
        float w = tanh_arg<true>(x, &lo);
        SigmoidParts p = sigmoid_parts<true>(w);
        const float s = fmaf(p.s * p.sm, lo, p.s);          // sigmoid(w + lo)
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
        if (!Exact) {
            f2 a, d;
            bwd2(splat(x), &a, &d);
            *act = a.x;
            *dact = d.x;
            return;
        }
        float lo;
        float w = tanh_arg<true>(x, &lo);
        SigmoidParts p = sigmoid_parts<true>(w);
        const float s = fmaf(p.s * p.sm, lo, p.s);
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
    __device__ __forceinline__ static float relu(float x) { return x > 0.0f ? x : (x != x ? x : 0.0f); }
    __device__ __forceinline__ static f2 fwd2(f2 x) { return make_float2(relu(x.x), relu(x.y)); }
    __device__ __forceinline__ static void bwd2(f2 x, f2 *act, f2 *dact)
    {
        *act = fwd2(x);
        *dact = make_float2(x.x > 0.0f ? 1.0f : (x.x != x.x ? x.x : 0.0f),   // 0 at x == 0
                            x.y > 0.0f ? 1.0f : (x.y != x.y ? x.y : 0.0f));
    }
    template <bool Exact>
    __device__ __forceinline__ static float fwd(float x)
    {
        return relu(x);                                     // NaN propagates
    }
    template <bool Exact>
    __device__ __forceinline__ static void bwd_main(float x, float *act, float *dact)
    {
        *act = relu(x);
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
