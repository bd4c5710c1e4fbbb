/*
 * Double-precision CPU oracle for the fused gated activation y = act(a) * b
 * and its backward.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by
 * the smoke check and by the CPU-baseline leg of the benchmark, never by the
 * product path.  It shares no code, header or constant table with the CUDA
 * library.
 *
 * Every value is computed in double from the exact value of the stored input
 * element, and the result is rounded ONCE, to nearest with ties to even, into
 * the storage dtype.  Subnormals are kept (no flush to zero).
 *
 * Sources (page titles and sections):
 *   [SM]  "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel"
 *         - Required reasoning process, steps 5-7 (SiLU, multiply, GeGLU erf form)
 *         - Common failure modes, "GELU variant mismatch" (the tanh form)
 *         - Correctness requirements (silu' forms; activation on a, not b)
 *         - Kernel design rules (fp32 math, stable sigmoid, cast at the store)
 *   [LP]  "Kernel Profile: SwiGLU (Tier 1 - Element-wise)"
 *         - Backward Pass, gradient_formulas (da, db)
 *   The GeGLU and ReGLU backward passes are not printed on the pages; they are
 *   the analytic derivatives of the printed forward formulas.
 *
 * Nothing here is blocked, fused or reordered: each output element is the
 * plain formula applied to the corresponding input elements.
 *
 * Two further operations of the same MLP block, each the plain definition
 * written out: the gate/up projections with the activation applied (dot
 * products in double, k in order) and the fused residual add + RMSNorm of
 * "Skill: Write a Triton Fused Add+RMSNorm Kernel" (row sums of squares in
 * double, compensated).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* enum values are part of the oracle's own calling convention */
enum { ORC_SILU = 0, ORC_GELU_ERF = 1, ORC_GELU_TANH = 2, ORC_RELU = 3 };
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

#define ORC_SQRT1_2 0.70710678118654752440   /* 1/sqrt(2), the [SM] step-7 constant */
#define ORC_SQRT_2_OVER_PI 0.79788456080286535588  /* sqrt(2/pi), [SM] tanh form */
#define ORC_TANH_CUBIC 0.044715                 /* [SM] tanh form cubic coefficient */
#define ORC_INV_SQRT_2PI 0.39894228040143267794   /* 1/sqrt(2*pi), normal density */

/* ------------------------------------------------------------------ */
/* Logistic sigmoid, 1/(1+exp(-x)).  [SM] Kernel design rules ask for a form
 * that is stable for very negative x; exp is only ever taken of a
 * non-positive number, so it never overflows. */
double oracle_sigmoid(double x)
{
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* Forward activations.  [SM] step 5 (SiLU = x*sigmoid(x)), step 7 (GeGLU erf
 * form 0.5*x*(1+erf(x/sqrt(2)))), "GELU variant mismatch" (tanh form
 * 0.5*x*(1+tanh(sqrt(2/pi)*(x+0.044715*x^3)))), and ReLU from the Purpose
 * section (ReGLU = relu(a)*b). */
double oracle_act(int act, double x)
{
    switch (act) {
    case ORC_SILU:
        return x * oracle_sigmoid(x);
    case ORC_GELU_ERF:
        /* 1 + erf(z) == erfc(-z) exactly; the erfc form keeps full relative
         * precision for negative x, where 1 + erf(z) cancels. */
        return 0.5 * x * erfc(-x * ORC_SQRT1_2);
    case ORC_GELU_TANH: {
        /* 0.5*(1 + tanh(u)) == sigmoid(2u) exactly; the sigmoid form keeps
         * full relative precision where tanh(u) rounds to -1. */
        double u = ORC_SQRT_2_OVER_PI * (x + ORC_TANH_CUBIC * x * x * x);
        return x * oracle_sigmoid(2.0 * u);
    }
    case ORC_RELU:
        if (isnan(x)) return x;
        return x > 0.0 ? x : 0.0;
    }
    return NAN;
}

/* The two terms whose sum is act'(x), returned separately so that a test can
 * scale its tolerance by |t1| + |t2| where they cancel (derivative roots).
 *   SiLU:       [LP] da formula, silu(a)*(1-sigmoid(a)) + sigmoid(a)
 *               -> t1 = sigmoid(x), t2 = silu(x) * (1 - sigmoid(x))
 *   GeGLU-erf:  d/dx [x * Phi(x)] = Phi(x) + x*phi(x),
 *               Phi(x) = 0.5*erfc(-x/sqrt 2), phi(x) = exp(-x^2/2)/sqrt(2 pi)
 *   GeGLU-tanh: d/dx [x * sigmoid(w(x))], w = 2u
 *               = sigmoid(w) + x * sigmoid(w)*sigmoid(-w) * w'(x)
 *   ReGLU:      1 for x > 0 and 0 otherwise (subgradient 0 at x = 0). */
void oracle_act_grad_terms(int act, double x, double *t1, double *t2)
{
    switch (act) {
    case ORC_SILU: {
        double s = oracle_sigmoid(x);
        double one_minus_s = oracle_sigmoid(-x);   /* 1 - sigmoid(x), no cancellation */
        *t1 = s;
        *t2 = (x * s) * one_minus_s;
        return;
    }
    case ORC_GELU_ERF:
        *t1 = 0.5 * erfc(-x * ORC_SQRT1_2);
        *t2 = x * exp(-0.5 * x * x) * ORC_INV_SQRT_2PI;
        return;
    case ORC_GELU_TANH: {
        double w = 2.0 * ORC_SQRT_2_OVER_PI * (x + ORC_TANH_CUBIC * x * x * x);
        double dw = 2.0 * ORC_SQRT_2_OVER_PI * (1.0 + 3.0 * ORC_TANH_CUBIC * x * x);
        double s = oracle_sigmoid(w);
        *t1 = s;
        *t2 = x * (s * oracle_sigmoid(-w)) * dw;
        return;
    }
    case ORC_RELU:
        if (isnan(x)) { *t1 = x; *t2 = 0.0; return; }
        *t1 = x > 0.0 ? 1.0 : 0.0;
        *t2 = 0.0;
        return;
    }
    *t1 = NAN;
    *t2 = NAN;
}

double oracle_act_grad(int act, double x)
{
    double t1, t2;
    oracle_act_grad_terms(act, x, &t1, &t2);
    return t1 + t2;
}

/* ------------------------------------------------------------------ */
/* Storage formats.  A binary format is described by p (significand bits,
 * implicit bit included), emin (exponent of the smallest normal) and emax
 * (exponent of the largest finite binade). */
static void fmt_params(int dtype, int *p, int *emin, int *emax)
{
    switch (dtype) {
    case ORC_F32:  *p = 24; *emin = -126; *emax = 127; return;
    case ORC_F16:  *p = 11; *emin = -14;  *emax = 15;  return;
    default:       *p = 8;  *emin = -126; *emax = 127; return;   /* bf16 */
    }
}

/* Round x to the nearest value of the format, ties to even, overflow to inf.
 * The quantum (ulp) is 2^(max(exponent(x), emin) - (p - 1)); dividing by a
 * power of two is exact, and nearbyint() rounds to nearest-even in the default
 * floating-point environment.  Returns the rounded value as a double. */
double oracle_round(double x, int dtype)
{
    int p, emin, emax;
    fmt_params(dtype, &p, &emin, &emax);
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    double ax = fabs(x);
    int e;
    (void)frexp(ax, &e);              /* ax = m * 2^e, m in [0.5, 1) */
    int lead = e - 1;                 /* exponent of the leading bit */
    if (lead < emin) lead = emin;     /* subnormal range: fixed quantum */
    double q = ldexp(1.0, lead - (p - 1));
    double r = nearbyint(ax / q) * q;
    double max_finite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (r > max_finite) r = INFINITY;
    return copysign(r, x);
}

/* Bit patterns <-> values.  f32 bits are the IEEE single encoding, bf16 the top
 * half of it, f16 the IEEE half encoding. */
static double f32_bits_to_double(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static uint32_t f32_value_to_bits(double r)   /* r already representable */
{
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

double oracle_decode(uint32_t bits, int dtype)
{
    switch (dtype) {
    case ORC_F32:
        return f32_bits_to_double(bits);
    case ORC_BF16:
        return f32_bits_to_double((bits & 0xFFFFu) << 16);
    default: {                        /* f16 */
        uint32_t s = (bits >> 15) & 1u, ex = (bits >> 10) & 0x1Fu, m = bits & 0x3FFu;
        double v;
        if (ex == 0) v = ldexp((double)m, -24);                         /* subnormal */
        else if (ex == 31) v = m ? NAN : INFINITY;
        else v = ldexp((double)(m | 0x400u), (int)ex - 25);           /* 1.m * 2^(ex-15) */
        return s ? -v : v;
    }
    }
}

uint32_t oracle_encode(double x, int dtype)   /* rounds, then encodes */
{
    double r = oracle_round(x, dtype);
    switch (dtype) {
    case ORC_F32:
        return f32_value_to_bits(r);
    case ORC_BF16:
        if (isnan(r)) return 0x7FC0u;
        return f32_value_to_bits(r) >> 16;   /* exact: r is a bf16 value */
    default: {                                /* f16 */
        uint32_t s = signbit(r) ? 0x8000u : 0u;
        double ar = fabs(r);
        if (isnan(r)) return 0x7E00u;
        if (isinf(r)) return s | 0x7C00u;
        if (ar == 0.0) return s;
        if (ar < ldexp(1.0, -14))
            return s | (uint32_t)(ar / ldexp(1.0, -24));              /* subnormal */
        int e;
        (void)frexp(ar, &e);
        int lead = e - 1;
        uint32_t m = (uint32_t)((ar / ldexp(1.0, lead) - 1.0) * 1024.0);
        return s | ((uint32_t)(lead + 15) << 10) | m;
    }
    }
}

static uint32_t load_bits(const void *p, int64_t i, int dtype)
{
    if (dtype == ORC_F32) return ((const uint32_t *)p)[i];
    return ((const uint16_t *)p)[i];
}

static void store_bits(void *p, int64_t i, int dtype, uint32_t v)
{
    if (dtype == ORC_F32) ((uint32_t *)p)[i] = v;
    else ((uint16_t *)p)[i] = (uint16_t)v;
}

/* ------------------------------------------------------------------ */
/* Element-wise forward over n elements of flat arrays of bit patterns:
 *   y[i] = round(act(a[i]) * b[i])          ([SM] steps 5-6; [LP] Forward Pass)
 * The activation is applied to a (the gate), never to b ([SM] Correctness). */
void oracle_fwd(int act, int dtype, const void *a, const void *b, void *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double av = oracle_decode(load_bits(a, i, dtype), dtype);
        double bv = oracle_decode(load_bits(b, i, dtype), dtype);
        store_bits(y, i, dtype, oracle_encode(oracle_act(act, av) * bv, dtype));
    }
}

/* Element-wise backward ([LP] Backward Pass, gradient_formulas):
 *   da[i] = round(dc[i] * act'(a[i]) * b[i]),  db[i] = round(dc[i] * act(a[i]))
 * act and act' are recomputed from a ([LP] backward_recompute). */
void oracle_bwd(int act, int dtype, const void *dc, const void *a, const void *b,
                void *da, void *db, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double cv = oracle_decode(load_bits(dc, i, dtype), dtype);
        double av = oracle_decode(load_bits(a, i, dtype), dtype);
        double bv = oracle_decode(load_bits(b, i, dtype), dtype);
        store_bits(da, i, dtype, oracle_encode(cv * oracle_act_grad(act, av) * bv, dtype));
        store_bits(db, i, dtype, oracle_encode(cv * oracle_act(act, av), dtype));
    }
}

/* Magnitude scale of da used by the fp32 tolerance reading:
 *   m[i] = |dc[i] * b[i]| * (|t1(a[i])| + |t2(a[i])|)   (terms as above). */
void oracle_bwd_da_scale(int act, int dtype, const void *dc, const void *a, const void *b,
                         double *m, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double cv = oracle_decode(load_bits(dc, i, dtype), dtype);
        double av = oracle_decode(load_bits(a, i, dtype), dtype);
        double bv = oracle_decode(load_bits(b, i, dtype), dtype);
        double t1, t2;
        oracle_act_grad_terms(act, av, &t1, &t2);
        m[i] = fabs(cv * bv) * (fabs(t1) + fabs(t2));
    }
}

/* Vector helpers over doubles (used by the oracle's own pins). */
void oracle_act_vec(int act, const double *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_act(act, x[i]);
}

void oracle_act_grad_terms_vec(int act, const double *x, double *t1, double *t2, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) oracle_act_grad_terms(act, x[i], &t1[i], &t2[i]);
}

void oracle_round_vec(int dtype, const double *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round(x[i], dtype);
}

void oracle_encode_vec(int dtype, const double *x, void *bits, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) store_bits(bits, i, dtype, oracle_encode(x[i], dtype));
}

void oracle_decode_vec(int dtype, const void *bits, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_decode(load_bits(bits, i, dtype), dtype);
}

/* ------------------------------------------------------------------ */
/* The gated MLP's first half with the activation applied to the projections
 * ("Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel", Purpose: the MLP is
 * down_proj(act(gate_proj(x)) * up_proj(x)); "Fused Kernels", section 4: the
 * gate and up tiles computed as x @ gate^T and x @ up^T):
 *   g[m,i] = sum_k x[m,k] * w_gate[i,k],   u[m,i] = sum_k x[m,k] * w_up[i,k]
 *   y[m,i] = round(act(g[m,i]) * u[m,i])
 * x is M x K, the weights are I x K (row i holds output feature i), all
 * row-major with row strides in elements.  Sums in double, k in order. */
static void gate_up_at(int dtype, const void *x, int64_t sx, const void *wg, const void *wu, int64_t sw,
                       int64_t K, int64_t m, int64_t i, double *g, double *u, double *ag, double *au)
{
    double sg = 0.0, su = 0.0, tg = 0.0, tu = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = oracle_decode(load_bits(x, m * sx + k, dtype), dtype);
        double gv = xv * oracle_decode(load_bits(wg, i * sw + k, dtype), dtype);
        double uv = xv * oracle_decode(load_bits(wu, i * sw + k, dtype), dtype);
        sg += gv;
        su += uv;
        tg += fabs(gv);
        tu += fabs(uv);
    }
    *g = sg;
    *u = su;
    *ag = tg;
    *au = tu;
}

/* y for the listed (m, i) pairs (n of them), plus g, u and the sums of
 * |products| (Sg, Su) that bound the error of any reordered summation.  Any
 * of g, u, sg, su may be NULL. */
void oracle_gemm_glu_at(int act, int dtype, const void *x, int64_t sx, const void *wg, const void *wu,
                        int64_t sw, int64_t K, const int64_t *ms, const int64_t *is, int64_t n, void *y,
                        double *g, double *u, double *sg, double *su)
{
    for (int64_t j = 0; j < n; ++j) {
        double gv, uv, ag, au;
        gate_up_at(dtype, x, sx, wg, wu, sw, K, ms[j], is[j], &gv, &uv, &ag, &au);
        store_bits(y, j, dtype, oracle_encode(oracle_act(act, gv) * uv, dtype));
        if (g) g[j] = gv;
        if (u) u[j] = uv;
        if (sg) sg[j] = ag;
        if (su) su[j] = au;
    }
}

/* The MLP's second half, the down projection ("Skill: Write a Triton SiLU-Mul
 * (SwiGLU) Kernel", Purpose: down_proj of the gated product; "Fused Kernels",
 * section 4, "The fused MLP": the gated tile multiplied by the down weights):
 *   d[m,n] = round(sum_k a[m,k] * b[n,k])
 * a is M x K (the stored y of the first half), b is N x K (row n holds output
 * feature n), row strides in elements.  The sum in double, k in order, and
 * one rounding; the sum of |products| is returned too (it bounds the error of
 * any reordered fp32 summation).  exact and sabs may be NULL. */
void oracle_matmul_nt_at(int dtype, const void *a, int64_t sa, const void *b, int64_t sb, int64_t K,
                         const int64_t *ms, const int64_t *ns, int64_t n, void *d, double *exact, double *sabs)
{
    for (int64_t j = 0; j < n; ++j) {
        double sum = 0.0, tot = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double pv = oracle_decode(load_bits(a, ms[j] * sa + k, dtype), dtype) *
                              oracle_decode(load_bits(b, ns[j] * sb + k, dtype), dtype);
            sum += pv;
            tot += fabs(pv);
        }
        store_bits(d, j, dtype, oracle_encode(sum, dtype));
        if (exact) exact[j] = sum;
        if (sabs) sabs[j] = tot;
    }
}

/* ------------------------------------------------------------------ */
/* Fused residual add + RMSNorm ("Skill: Write a Triton Fused Add+RMSNorm
 * Kernel": Purpose, y = rmsnorm(x + residual) with x + residual written back;
 * Required reasoning process steps 3-7; Kernel design rules, eps inside the
 * square root, gamma indexed by column only, no mean and no bias):
 *   h[j]  = x[j] + res[j]                   exact; the stored h is rounded once
 *   ms    = (1/H) * sum_j h[j]^2            of the exact h, over the whole row
 *   rstd  = 1 / sqrt(ms + eps)
 *   y[j]  = round(h[j] * rstd * gamma[j])
 * All rows contiguous (row r starts at r * H); gamma has H entries in the
 * input dtype.  The sum of squares is compensated (Neumaier), so its relative
 * error stays near 2^-53 for any H.  Outputs: h and y as bit patterns, rstd
 * per row and the unrounded y (both in double; either pointer may be NULL). */
static double row_sum_squares(const double *h, int64_t H)
{
    double s = 0.0, c = 0.0;
    for (int64_t j = 0; j < H; ++j) {
        const double t = h[j] * h[j];
        const double u = s + t;
        if (fabs(s) >= fabs(t))
            c += (s - u) + t;
        else
            c += (t - u) + s;
        s = u;
    }
    return s + c;
}

void oracle_add_rmsnorm(int dtype, const void *x, const void *res, const void *gamma, void *h, void *y,
                        double *rstd, double *y_exact, int64_t n_rows, int64_t H, double eps)
{
    double *hv = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int64_t j = 0; j < H; ++j) {
            const int64_t i = r * H + j;
            hv[j] = oracle_decode(load_bits(x, i, dtype), dtype) + oracle_decode(load_bits(res, i, dtype), dtype);
            store_bits(h, i, dtype, oracle_encode(hv[j], dtype));
        }
        const double ms = row_sum_squares(hv, H) / (double)H;
        const double rs = 1.0 / sqrt(ms + eps);
        if (rstd) rstd[r] = rs;
        for (int64_t j = 0; j < H; ++j) {
            const int64_t i = r * H + j;
            const double v = hv[j] * rs * oracle_decode(load_bits(gamma, j, dtype), dtype);
            store_bits(y, i, dtype, oracle_encode(v, dtype));
            if (y_exact) y_exact[i] = v;
        }
    }
    free(hv);
}

/* Backward of the residual add + RMSNorm ("Skill: Write a Triton Fused
 * Add+RMSNorm Kernel", Required reasoning process steps 9-10: the forward keeps
 * rstd and the summed rows; the gradient of the norm goes to x and to the
 * residual alike).  With y = s * rstd * gamma and rstd = (sum s^2 / H + eps)^(-1/2),
 *   ds[j]  = rstd * gamma[j] * dy[j] - (rstd^3 / H) * s[j] * sum_k gamma[k] dy[k] s[k]
 *            (+ dh[j], the gradient reaching s through the residual stream)
 *   dgamma[j] = sum over rows of dy[j] * s[j] * rstd
 * s is the stored sum h, rstd the stored fp32 value (f32 bit patterns), both
 * taken as given.  dh may be NULL.  Outputs: ds rounded once into the dtype,
 * ds unrounded (may be NULL) and dgamma (H doubles, overwritten).  Contiguous
 * rows. */
void oracle_add_rmsnorm_bwd(int dtype, const void *dy, const void *h, const void *rstd_bits, const void *gamma,
                            const void *dh, void *ds, double *ds_exact, double *dgamma, int64_t n_rows, int64_t H)
{
    for (int64_t j = 0; j < H; ++j) dgamma[j] = 0.0;
    for (int64_t r = 0; r < n_rows; ++r) {
        const double rs = oracle_decode(load_bits(rstd_bits, r, ORC_F32), ORC_F32);
        double dot = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            const int64_t i = r * H + j;
            dot += oracle_decode(load_bits(gamma, j, dtype), dtype) * oracle_decode(load_bits(dy, i, dtype), dtype) *
                   oracle_decode(load_bits(h, i, dtype), dtype);
        }
        const double c = rs * rs * rs / (double)H * dot;
        for (int64_t j = 0; j < H; ++j) {
            const int64_t i = r * H + j;
            const double g = oracle_decode(load_bits(gamma, j, dtype), dtype);
            const double d = oracle_decode(load_bits(dy, i, dtype), dtype);
            const double s = oracle_decode(load_bits(h, i, dtype), dtype);
            double v = rs * g * d - c * s;
            if (dh) v += oracle_decode(load_bits(dh, i, dtype), dtype);
            store_bits(ds, i, dtype, oracle_encode(v, dtype));
            if (ds_exact) ds_exact[i] = v;
            dgamma[j] += d * s * rs;
        }
    }
}
