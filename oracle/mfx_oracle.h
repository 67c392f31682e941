/*
 * mfx_oracle.h -- declarations of the CPU oracle for the fused MLP and
 * residual epilogues.
 *
 * TEST INFRASTRUCTURE ONLY.  The oracle is a plain, slow, single-threaded C
 * restatement of what the fused ops compute.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load it.  It shares no
 * code, header, table or helper with the CUDA library: this header is the
 * oracle's own and is never included by the library.
 *
 * Citations name the web page "Megatron-LM operator fusion walkthrough"
 * (www.wmrh.cn/news/51426), which explains megatron/core/fusions/, and its
 * numbered sections (for example "fusions page §4.2").
 *
 * Precision: the activations (GeLU, GEGLU, SwiGLU and their gradients) are
 * evaluated in double precision from the pages' formulas.  Only the bias add
 * is rounded to fp32, because it is the one statement that materialises a
 * tensor of the input dtype.  The bias-dropout-add ops follow the fp32 op
 * sequence exactly: (x + b), then the keep/scale step, then + residual, each
 * rounded to fp32, with one rounding to the output dtype at the store.
 * Dtype codes: 0 = fp32, 1 = bf16 (stored as raw uint16 bit patterns).
 */
#ifndef MFX_ORACLE_H
#define MFX_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar pieces (exported so the pins can probe them) ---------------- */
float    orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);
double   orc_gelu_tanh(double x);       /* fusions page §4.2, forward            */
double   orc_gelu_tanh_grad(double x);  /* fusions page §4.2, backward factor    */
double   orc_logistic(double z);        /* sigma(z) = 1 / (1 + e^-z)             */
double   orc_silu(double z);            /* z * sigma(z), the SwiGLU activation   */

/* Philox-4xW-10 block functions (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11).  Both widths run through one generic
 * round function so that the 64-bit instance, which numpy also implements,
 * checks the round structure shared with the 32-bit instance. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void orc_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);
void orc_philox4x32_rounds(int rounds, const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Dropout mask mapping (16-bit uniform per element; 8 elements per block). */
uint32_t orc_dropout_threshold(float p);
uint32_t orc_uniform16(uint64_t seed, uint64_t offset, uint64_t e);
void     orc_keep_mask(uint64_t seed, uint64_t offset, uint64_t elem_base, int64_t n,
                       float p, uint8_t* keep);

/* ---- tensor ops ----------------------------------------------------------- */
/* All tensors contiguous row-major.  bias may be NULL (treated as +0). */
void orc_bias_gelu_fwd(int dt, int64_t rows, int64_t cols, const void* bias,
                       const void* y, double* out);
/* *_scale outputs (nullable) give, per element, the magnitude of the terms
 * of the sum that forms the derivative, times the other factors: the scale
 * against which an fp32 evaluation's rounding error is measured where the
 * derivative crosses zero and the sum cancels. */
void orc_bias_gelu_bwd(int dt, int64_t rows, int64_t cols, const void* g,
                       const void* bias, const void* y, double* dy, double* dy_scale);

/* x is [rows, 2F]; the first F columns are the activated half, the last F the
 * linear half; bias is [2F] and is added before the split. */
void orc_bias_geglu_fwd(int dt, int64_t rows, int64_t F, const void* x,
                        const void* bias, double* out);
void orc_bias_geglu_bwd(int dt, int64_t rows, int64_t F, const void* g,
                        const void* x, const void* bias, double* dx, double* dx_scale);
/* weight: [rows] fp32 or NULL.  dweight, dweight_abs: [rows], used iff weight
 * is given; dweight_abs receives sum |term|, the condition scale of the sum. */
void orc_bias_swiglu_fwd(int dt, int64_t rows, int64_t F, const void* x,
                         const void* bias, const float* weight, double* out);
void orc_bias_swiglu_bwd(int dt, int64_t rows, int64_t F, const void* g,
                         const void* x, const void* bias, const float* weight,
                         double* dx, double* dweight, double* dweight_abs, double* dx_scale);

/* out and x share x_dt; residual has r_dt (cast to x_dt first). */
void orc_bias_dropout_add_train(int x_dt, int r_dt, int64_t rows, int64_t cols,
                                const void* x, const void* bias, const void* residual,
                                float p, uint64_t seed, uint64_t offset,
                                uint64_t elem_base, void* out, uint8_t* keep);
void orc_bias_dropout_add_inference(int x_dt, int r_dt, int64_t rows, int64_t cols,
                                    void* x, const void* bias, const void* residual);

/* Backward of bias-dropout-add: dx = keep ? g * scale : 0 (x_dt), dres = g
 * in r_dt (nullable).  keep NULL regenerates the forward's mask. */
void orc_bias_dropout_add_bwd(int x_dt, int r_dt, int64_t rows, int64_t cols, const void* g,
                              const uint8_t* keep, float p, uint64_t seed, uint64_t offset,
                              uint64_t elem_base, void* dx, void* dres);

/* Column sums of v rounded to dtype dt (the bias gradient of a stored
 * gradient tensor); abs_sum (nullable) gets the sums of magnitudes. */
void orc_column_sums(int dt, int64_t rows, int64_t cols, const double* v, double* sum, double* abs_sum);

/* Weighted squared ReLU: out = relu(x)^2 * weight[r]; backward dx, dweight
 * (and dweight_abs = sum |term|, nullable). */
void orc_weighted_squared_relu_fwd(int dt, int64_t rows, int64_t cols, const void* x,
                                   const float* weight, double* out);
void orc_weighted_squared_relu_bwd(int dt, int64_t rows, int64_t cols, const void* g, const void* x,
                                   const float* weight, double* dx, double* dweight, double* dweight_abs);

/* Scale-mask-softmax along the last dim of x [b, np, sq, sk] (fusions page
 * §6.2): z = x * scale (+ mask, additive, [mb, mnp, msq, sk] broadcast where a
 * size is 1; mask NULL = none), causal != 0 excludes k > q (sq == sk); rows
 * with every position excluded give zeros.  y: float64 [b, np, sq, sk]. */
void orc_scaled_masked_softmax_fwd(int dt, int64_t b, int64_t np, int64_t sq, int64_t sk,
                                   const void* x, const void* mask, int64_t mb, int64_t mnp,
                                   int64_t msq, int causal, float scale, double* y);
/* Backward from the softmax results: dx = scale * y * (dy - sum_k dy_k y_k)
 * per row; with causal != 0 (rows of [.., sk, sk]) the excluded positions
 * are exactly 0.  dx_scale (nullable): |scale y| (|dy| + |sum|), the scale of
 * the terms that cancel in the difference. */
void orc_scaled_softmax_bwd(int dt, int64_t rows, int64_t sk, const void* dy, const void* y, int causal,
                            float scale, double* dx, double* dx_scale);

#ifdef __cplusplus
}
#endif
#endif /* MFX_ORACLE_H */
