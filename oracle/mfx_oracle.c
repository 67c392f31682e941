/*
 * mfx_oracle.c -- plain CPU oracle for the fused MLP and residual epilogues.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by tests/, by the smoke check and by the
 * CPU-baseline leg of bench.py, never by the library.  Shares no code with
 * the CUDA path.  Build with -O2 -ffp-contract=off and without fast-math so
 * that every float operation below is one IEEE-754 rounding, in the order
 * written.
 *
 * Source of every formula: the web page "Megatron-LM operator fusion
 * walkthrough" (www.wmrh.cn/news/51426), cited as "fusions page §N".  Where
 * that page is silent the reading taken is stated next to the code.
 *
 * Parity pins (tests/test_oracle_pins.py, tests/test_philox_pins.py) tie each
 * function to something other than itself: the erf form of GeLU, central
 * finite differences, scipy's logistic, torch's bf16 rounding and fp32
 * arithmetic, numpy's Philox4x64-10, cuRAND's host Philox4_32_10 generator
 * (stored known-answer words and a live comparison), the Weyl constants'
 * definitions and the statistics of the mask.
 */
#include "mfx_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 is the top half of an fp32 bit pattern, so widening is exact. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to nearest, ties to even; NaN stays a (quiet) NaN; subnormals kept. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u; /* carries into the exponent correctly, up to infinity */
    return (uint16_t)upper;
}

static float load_elem(int dt, const void* p, int64_t i)
{
    if (dt == 1)
        return orc_bf16_to_f32(((const uint16_t*)p)[i]);
    return ((const float*)p)[i];
}

static void store_elem(int dt, void* p, int64_t i, float v)
{
    if (dt == 1)
        ((uint16_t*)p)[i] = orc_f32_to_bf16(v);
    else
        ((float*)p)[i] = v;
}

/* Bias add: the one statement of each op that materialises a tensor of the
 * input dtype ("x = bias + y", fusions page §4.2).  It is one fp32 addition;
 * with bias absent it adds +0. */
static double bias_add_f32(int dt, const void* y, int64_t i, const void* bias, int64_t c)
{
    float yv = load_elem(dt, y, i);
    float bv = bias ? load_elem(dt, bias, c) : 0.0f;
    float x = yv + bv;
    return (double)x;
}

/* ------------------------------------------------------------------------ */
/* GeLU, tanh approximation (fusions page §4.2)                              */
/* ------------------------------------------------------------------------ */

/* Constants exactly as the page prints them. */
static const double GELU_K0 = 0.79788456;   /* sqrt(2/pi)                  */
static const double GELU_K1 = 0.044715;     /* cubic coefficient           */
static const double GELU_KD = 0.1070322243; /* sqrt(2/pi) * 3 * 0.044715   */

/* 1 + tanh(u).  For u < 0 the printed sum cancels; the identity
 * 1 + tanh(u) = 2 / (1 + e^(-2u)) gives the same number without losing the
 * relative precision. */
static double one_plus_tanh(double u)
{
    if (u >= 0.0)
        return 1.0 + tanh(u);
    return 2.0 / (1.0 + exp(-2.0 * u));
}

/* 1 - tanh(u)^2 written as 1 / cosh(u)^2, the same number without the
 * cancellation of the printed form at large |u|. */
static double one_minus_tanh_sq(double u)
{
    double ch = cosh(u);
    return 1.0 / (ch * ch);
}

/* Forward: x * 0.5 * (1 + tanh(0.79788456 * x * (1 + 0.044715 * x * x))). */
double orc_gelu_tanh(double x)
{
    double u = GELU_K0 * x * (1.0 + GELU_K1 * x * x);
    return x * 0.5 * one_plus_tanh(u);
}

/* Backward factor d/dx of the forward, in the grouping the page's backward
 * uses with its printed constant 0.1070322243:
 *   ff = 0.5 x ((1 - tanh^2 u)(0.79788456 + 0.1070322243 x^2)) + 0.5 (1 + tanh u).
 * The page prints only the constant; this is the exact derivative of the
 * forward (d/dx of u is 0.79788456 + 3 * 0.79788456 * 0.044715 * x^2).
 * The two terms are returned separately: near the root of ff (x ~ -0.75) they
 * cancel, and |t1| + |t2| is the scale of any fp32 evaluation's error. */
static void gelu_grad_terms(double x, double* t1, double* t2)
{
    double u = GELU_K0 * x * (1.0 + GELU_K1 * x * x);
    *t1 = 0.5 * x * (one_minus_tanh_sq(u) * (GELU_K0 + GELU_KD * x * x));
    *t2 = 0.5 * one_plus_tanh(u);
}

double orc_gelu_tanh_grad(double x)
{
    double t1, t2;
    gelu_grad_terms(x, &t1, &t2);
    return t1 + t2;
}

void orc_bias_gelu_fwd(int dt, int64_t rows, int64_t cols, const void* bias,
                       const void* y, double* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            double x = bias_add_f32(dt, y, i, bias, c);
            out[i] = orc_gelu_tanh(x);
        }
}

/* dy = ff(bias + y) * g (fusions page §4.2, bias_gelu_back(g, bias, y)).
 * dy_scale (nullable) receives |g| (|t1| + |t2|), the magnitude of the sum
 * that forms ff. */
void orc_bias_gelu_bwd(int dt, int64_t rows, int64_t cols, const void* g,
                       const void* bias, const void* y, double* dy, double* dy_scale)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            double x = bias_add_f32(dt, y, i, bias, c);
            double gv = (double)load_elem(dt, g, i);
            double t1, t2;
            gelu_grad_terms(x, &t1, &t2);
            dy[i] = (t1 + t2) * gv;
            if (dy_scale)
                dy_scale[i] = (fabs(t1) + fabs(t2)) * fabs(gv);
        }
}

/* ------------------------------------------------------------------------ */
/* Gated linear units (fusions page §2: fused_bias_geglu, fused_bias_swiglu  */
/* and the weighted SwiGLU; §9: the weighted-SwiGLU test).                   */
/* Reading: the page names these ops without printing them.  The input of    */
/* width 2F gets the bias first, then splits into halves; the first half is  */
/* activated and multiplies the second.  GEGLU's activation is the §4.2      */
/* tanh GeLU; SwiGLU's is SiLU.                                              */
/* ------------------------------------------------------------------------ */

double orc_logistic(double z)
{
    if (z >= 0.0)
        return 1.0 / (1.0 + exp(-z));
    double e = exp(z);
    return e / (1.0 + e);
}

double orc_silu(double z) { return z * orc_logistic(z); }

void orc_bias_geglu_fwd(int dt, int64_t rows, int64_t F, const void* x,
                        const void* bias, double* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < F; ++c) {
            double a = bias_add_f32(dt, x, r * 2 * F + c, bias, c);
            double b = bias_add_f32(dt, x, r * 2 * F + F + c, bias, F + c);
            out[r * F + c] = orc_gelu_tanh(a) * b;
        }
}

/* d/da [gelu(a) b] = gelu'(a) b,  d/db = gelu(a); both times the upstream g.
 * dx_scale (nullable): for d/da, |g b| (|t1| + |t2|) (see gelu_grad_terms);
 * for d/db, |d/db| (a product, nothing cancels). */
void orc_bias_geglu_bwd(int dt, int64_t rows, int64_t F, const void* g,
                        const void* x, const void* bias, double* dx, double* dx_scale)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < F; ++c) {
            double a = bias_add_f32(dt, x, r * 2 * F + c, bias, c);
            double b = bias_add_f32(dt, x, r * 2 * F + F + c, bias, F + c);
            double gv = (double)load_elem(dt, g, r * F + c);
            double t1, t2;
            gelu_grad_terms(a, &t1, &t2);
            dx[r * 2 * F + c] = gv * b * (t1 + t2);
            dx[r * 2 * F + F + c] = gv * orc_gelu_tanh(a);
            if (dx_scale) {
                dx_scale[r * 2 * F + c] = fabs(gv * b) * (fabs(t1) + fabs(t2));
                dx_scale[r * 2 * F + F + c] = fabs(dx[r * 2 * F + F + c]);
            }
        }
}

/* out = silu(a) * b, times weight[r] when a per-token weight is given. */
void orc_bias_swiglu_fwd(int dt, int64_t rows, int64_t F, const void* x,
                         const void* bias, const float* weight, double* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < F; ++c) {
            double a = bias_add_f32(dt, x, r * 2 * F + c, bias, c);
            double b = bias_add_f32(dt, x, r * 2 * F + F + c, bias, F + c);
            double v = orc_silu(a) * b;
            if (weight)
                v *= (double)weight[r];
            out[r * F + c] = v;
        }
}

/* With gw = g * weight[r] (or g):
 *   d/da = gw * b * sigma(a) * (1 + a * (1 - sigma(a)))
 *   d/db = gw * silu(a)
 *   d/dweight[r] = sum_c g * silu(a) * b
 * dx_scale (nullable): for d/da, |gw b sigma(a)| (1 + |a (1 - sigma(a))|), the
 * magnitude of the sum that vanishes at the minimum of silu (a ~ -1.278);
 * for d/db, |d/db|. */
void orc_bias_swiglu_bwd(int dt, int64_t rows, int64_t F, const void* g,
                         const void* x, const void* bias, const float* weight,
                         double* dx, double* dweight, double* dweight_abs, double* dx_scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t c = 0; c < F; ++c) {
            double a = bias_add_f32(dt, x, r * 2 * F + c, bias, c);
            double b = bias_add_f32(dt, x, r * 2 * F + F + c, bias, F + c);
            double gv = (double)load_elem(dt, g, r * F + c);
            double gw = weight ? gv * (double)weight[r] : gv;
            double sig = orc_logistic(a);
            double one_minus_sig = orc_logistic(-a);
            dx[r * 2 * F + c] = gw * b * sig * (1.0 + a * one_minus_sig);
            dx[r * 2 * F + F + c] = gw * orc_silu(a);
            if (dx_scale) {
                dx_scale[r * 2 * F + c] = fabs(gw * b * sig) * (1.0 + fabs(a * one_minus_sig));
                dx_scale[r * 2 * F + F + c] = fabs(dx[r * 2 * F + F + c]);
            }
            if (weight) {
                double term = gv * orc_silu(a) * b;
                acc += term;
                acc_abs += fabs(term);
            }
        }
        if (weight) {
            dweight[r] = acc;
            if (dweight_abs)
                dweight_abs[r] = acc_abs;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Philox-4xW-10 (Salmon et al., SC'11)                                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    unsigned width;      /* word width W in bits: 32 or 64           */
    uint64_t mul0, mul1; /* round multipliers                        */
    uint64_t weyl0, weyl1; /* key increments between rounds          */
} philox_params;

/* Philox4x32 multipliers from the paper; key increments are the golden
 * ratio's fraction and sqrt(3) - 1, each times 2^W. */
static const philox_params PHILOX_4x32 = {
    32, 0xD2511F53u, 0xCD9E8D57u, 0x9E3779B9u, 0xBB67AE85u};
static const philox_params PHILOX_4x64 = {
    64, 0xD2E7470EE14C6C93ull, 0xCA5A826395121157ull,
    0x9E3779B97F4A7C15ull, 0xBB67AE8584CAA73Bull};

/* One S-box/permutation round on the four-word counter:
 *   (hi0, lo0) = mul0 * c0,  (hi1, lo1) = mul1 * c2
 *   c' = (hi1 ^ c1 ^ k0,  lo1,  hi0 ^ c3 ^ k1,  lo0)
 * and the key is bumped by the Weyl increments between rounds. */
static void philox_generic(const philox_params* P, int rounds, uint64_t c[4], uint64_t k[2])
{
    const uint64_t mask = P->width == 64 ? ~(uint64_t)0 : (((uint64_t)1 << P->width) - 1);
    for (int r = 0; r < rounds; ++r) {
        if (r > 0) {
            k[0] = (k[0] + P->weyl0) & mask;
            k[1] = (k[1] + P->weyl1) & mask;
        }
        unsigned __int128 p0 = (unsigned __int128)P->mul0 * c[0];
        unsigned __int128 p1 = (unsigned __int128)P->mul1 * c[2];
        uint64_t hi0 = (uint64_t)(p0 >> P->width) & mask, lo0 = (uint64_t)p0 & mask;
        uint64_t hi1 = (uint64_t)(p1 >> P->width) & mask, lo1 = (uint64_t)p1 & mask;
        uint64_t n0 = hi1 ^ c[1] ^ k[0];
        uint64_t n2 = hi0 ^ c[3] ^ k[1];
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

void orc_philox4x32_rounds(int rounds, const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint64_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint64_t k[2] = {key[0], key[1]};
    philox_generic(&PHILOX_4x32, rounds, c, k);
    for (int i = 0; i < 4; ++i)
        out[i] = (uint32_t)c[i];
}

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    orc_philox4x32_rounds(10, ctr, key, out);
}

void orc_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    uint64_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint64_t k[2] = {key[0], key[1]};
    philox_generic(&PHILOX_4x64, 10, c, k);
    for (int i = 0; i < 4; ++i)
        out[i] = c[i];
}

/* ------------------------------------------------------------------------ */
/* Dropout mask.  The page names no generator (fusions page §3.2 only says   */
/* the unfused and fused versions run under one seed).  Reading taken:      */
/* element e (global flat index) uses Philox4x32-10 block j = e / 8 with     */
/* counter (lo32 j, hi32 j, lo32 offset, hi32 offset) and key (lo32 seed,    */
/* hi32 seed); lane e % 8 takes 16-bit word (e % 8) of the 128-bit output,   */
/* i.e. bits [16 (lane % 2), +16) of 32-bit output word lane / 2.            */
/* The element is kept iff that word >= ceil(p * 65536) (clamped to 65535). */
/* ------------------------------------------------------------------------ */

uint32_t orc_dropout_threshold(float p)
{
    double t = ceil((double)p * 65536.0);
    if (t < 0.0)
        t = 0.0;
    if (t > 65535.0)
        t = 65535.0;
    return (uint32_t)t;
}

uint32_t orc_uniform16(uint64_t seed, uint64_t offset, uint64_t e)
{
    uint64_t j = e >> 3;
    unsigned lane = (unsigned)(e & 7u);
    uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return (out[lane >> 1] >> (16u * (lane & 1u))) & 0xFFFFu;
}

void orc_keep_mask(uint64_t seed, uint64_t offset, uint64_t elem_base, int64_t n,
                   float p, uint8_t* keep)
{
    uint32_t T = orc_dropout_threshold(p);
    for (int64_t i = 0; i < n; ++i)
        keep[i] = orc_uniform16(seed, offset, elem_base + (uint64_t)i) >= T ? 1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Bias + dropout + residual add (fusions page §3.2-§3.3)                    */
/*   out = residual + dropout(x + bias, p, training)                         */
/* The residual is first cast to x's dtype ("residual.to(x.dtype)", §3.2).   */
/* Readings: inverted dropout, kept values scaled by 1 / (1 - p) computed    */
/* once in fp32; a dropped element contributes +0; the arithmetic is fp32.   */
/* ------------------------------------------------------------------------ */

/* residual cast to x's dtype, then widened to fp32 */
static float residual_as_x(int x_dt, int r_dt, const void* residual, int64_t i)
{
    float rv = load_elem(r_dt, residual, i);
    if (x_dt == 1 && r_dt == 0)
        rv = orc_bf16_to_f32(orc_f32_to_bf16(rv));
    return rv;
}

void orc_bias_dropout_add_train(int x_dt, int r_dt, int64_t rows, int64_t cols,
                                const void* x, const void* bias, const void* residual,
                                float p, uint64_t seed, uint64_t offset,
                                uint64_t elem_base, void* out, uint8_t* keep)
{
    const uint32_t T = orc_dropout_threshold(p);
    const float scale = 1.0f / (1.0f - p);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            float v = load_elem(x_dt, x, i) + (bias ? load_elem(x_dt, bias, c) : 0.0f);
            int k = orc_uniform16(seed, offset, elem_base + (uint64_t)i) >= T;
            v = k ? v * scale : 0.0f;
            float o = v + residual_as_x(x_dt, r_dt, residual, i);
            store_elem(x_dt, out, i, o);
            keep[i] = (uint8_t)k;
        }
}

/* Inference: no dropout, written in place into x (fusions page §3.2). */
void orc_bias_dropout_add_inference(int x_dt, int r_dt, int64_t rows, int64_t cols,
                                    void* x, const void* bias, const void* residual)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            float v = load_elem(x_dt, x, i) + (bias ? load_elem(x_dt, bias, c) : 0.0f);
            float o = v + residual_as_x(x_dt, r_dt, residual, i);
            store_elem(x_dt, x, i, o);
        }
}

/* ------------------------------------------------------------------------ */
/* Backward of bias-dropout-add (fusions page §3.4: the unit test compares   */
/* the fused and unfused gradients).  With out = r~ + dropout(x + b):        */
/*   d(x + b) = keep ? g * scale : 0   (fp32, rounded to x's dtype = dx)     */
/*   d(residual) = g, through the cast: g in the residual's dtype            */
/* keep: the forward's mask, or NULL to regenerate it from                   */
/* (seed, offset, elem_base, p) exactly as the forward drew it.              */
/* ------------------------------------------------------------------------ */
void orc_bias_dropout_add_bwd(int x_dt, int r_dt, int64_t rows, int64_t cols, const void* g,
                              const uint8_t* keep, float p, uint64_t seed, uint64_t offset,
                              uint64_t elem_base, void* dx, void* dres)
{
    const uint32_t T = orc_dropout_threshold(p);
    const float scale = 1.0f / (1.0f - p);
    for (int64_t i = 0; i < rows * cols; ++i) {
        float gv = load_elem(x_dt, g, i);
        int k = keep ? keep[i] != 0 : orc_uniform16(seed, offset, elem_base + (uint64_t)i) >= T;
        store_elem(x_dt, dx, i, k ? gv * scale : 0.0f);
        if (dres)
            store_elem(r_dt, dres, i, gv);
    }
}

/* Bias gradient: the column sums of a gradient tensor as it is stored.  The
 * page's backward hands the same gradient tensor to the input and to the
 * broadcast bias (§4.3), and autograd sums it over the broadcast rows; the
 * values summed are the stored ones, i.e. v rounded to dtype dt.  sum and
 * abs_sum are exact-ish fp64 sums of round_dt(v) and |round_dt(v)|. */
void orc_column_sums(int dt, int64_t rows, int64_t cols, const double* v, double* sum, double* abs_sum)
{
    for (int64_t c = 0; c < cols; ++c) {
        sum[c] = 0.0;
        if (abs_sum)
            abs_sum[c] = 0.0;
    }
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float f = (float)v[r * cols + c];
            if (dt == 1)
                f = orc_bf16_to_f32(orc_f32_to_bf16(f));
            sum[c] += (double)f;
            if (abs_sum)
                abs_sum[c] += fabs((double)f);
        }
}

/* ------------------------------------------------------------------------ */
/* Weighted squared ReLU (fusions page §2, fused_weighted_squared_relu: the  */
/* MoE activation weighted per token, named next to the weighted SwiGLU).    */
/* The page only names it; reading: out = relu(x)^2 * weight[r], no bias.    */
/*   d/dx = g * weight[r] * 2 relu(x);  d/dweight[r] = sum_c g * relu(x)^2  */
/* ------------------------------------------------------------------------ */
static double relu(double v) { return v > 0.0 ? v : 0.0; }

void orc_weighted_squared_relu_fwd(int dt, int64_t rows, int64_t cols, const void* x,
                                   const float* weight, double* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            double a = relu((double)load_elem(dt, x, r * cols + c));
            out[r * cols + c] = a * a * (double)weight[r];
        }
}

void orc_weighted_squared_relu_bwd(int dt, int64_t rows, int64_t cols, const void* g, const void* x,
                                   const float* weight, double* dx, double* dweight, double* dweight_abs)
{
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            double a = relu((double)load_elem(dt, x, i));
            double gv = (double)load_elem(dt, g, i);
            dx[i] = gv * (double)weight[r] * 2.0 * a;
            acc += gv * a * a;
            acc_abs += fabs(gv * a * a);
        }
        dweight[r] = acc;
        if (dweight_abs)
            dweight_abs[r] = acc_abs;
    }
}

/* ------------------------------------------------------------------------ */
/* Scale-mask-softmax, fusions page §6.2 (ScaledSoftmax: scale then softmax; */
/* ScaledMaskedSoftmax: scale, then the given mask, then softmax, input      */
/* [b, np, sq, sk]; ScaledUpperTriangMaskedSoftmax: scale, then the causal   */
/* upper-triangle mask, then softmax, input [attn_batches, sq, sk]) and the  */
/* backward all three share (softmax results and scale only).               */
/*                                                                           */
/* Readings where the page leaves a step open:                               */
/*  - the mask is additive (§6.2 calls it a broadcastable additive mask): it */
/*    is added to the scaled scores; -inf excludes a position.  It has the   */
/*    input's dtype and shape [mb, mnp, msq, sk], each of mb, mnp, msq either */
/*    1 (broadcast) or the input's size;                                     */
/*  - the causal mask excludes key k from query row q when k > q (upper     */
/*    triangle), with sq == sk (§6.4: the causal path asserts sq == sk);     */
/*  - a row with no finite score left (every position excluded) has no      */
/*    softmax; its output is all zeros, and so is its gradient;             */
/*  - all arithmetic in fp32 or wider (§6.3: with a scale the softmax runs   */
/*    in fp32); the oracle evaluates in double.                              */
/* ------------------------------------------------------------------------ */
void orc_scaled_masked_softmax_fwd(int dt, int64_t b, int64_t np, int64_t sq, int64_t sk,
                                   const void* x, const void* mask, int64_t mb, int64_t mnp,
                                   int64_t msq, int causal, float scale, double* y)
{
    for (int64_t i = 0; i < b; ++i)
        for (int64_t h = 0; h < np; ++h)
            for (int64_t q = 0; q < sq; ++q) {
                const int64_t row = (i * np + h) * sq + q;
                const int64_t mrow = ((mb == 1 ? 0 : i) * mnp + (mnp == 1 ? 0 : h)) * msq + (msq == 1 ? 0 : q);
                double* out = y + row * sk;
                /* scores z_k, with excluded positions at -inf */
                for (int64_t k = 0; k < sk; ++k) {
                    double z = (double)load_elem(dt, x, row * sk + k) * (double)scale;
                    if (mask)
                        z += (double)load_elem(dt, mask, mrow * sk + k);
                    if (causal && k > q)
                        z = -INFINITY;
                    out[k] = z;
                }
                double m = -INFINITY;
                for (int64_t k = 0; k < sk; ++k)
                    if (out[k] > m)
                        m = out[k];
                if (m == -INFINITY) {
                    for (int64_t k = 0; k < sk; ++k)
                        out[k] = 0.0;
                    continue;
                }
                double sum = 0.0;
                for (int64_t k = 0; k < sk; ++k) {
                    out[k] = exp(out[k] - m);
                    sum += out[k];
                }
                for (int64_t k = 0; k < sk; ++k)
                    out[k] /= sum;
            }
}

void orc_scaled_softmax_bwd(int dt, int64_t rows, int64_t sk, const void* dy, const void* y, int causal,
                            float scale, double* dx, double* dx_scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t q = r % sk; /* query index when causal (sq == sk) */
        double s = 0.0;
        for (int64_t k = 0; k < sk; ++k) {
            if (causal && k > q)
                continue;
            s += (double)load_elem(dt, dy, r * sk + k) * (double)load_elem(dt, y, r * sk + k);
        }
        for (int64_t k = 0; k < sk; ++k) {
            const int64_t i = r * sk + k;
            if (causal && k > q) {
                dx[i] = 0.0;
                if (dx_scale)
                    dx_scale[i] = 0.0;
                continue;
            }
            const double yk = (double)load_elem(dt, y, i), gk = (double)load_elem(dt, dy, i);
            dx[i] = (double)scale * yk * (gk - s);
            if (dx_scale)
                dx_scale[i] = fabs((double)scale * yk) * (fabs(gk) + fabs(s));
        }
    }
}
