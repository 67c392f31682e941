/*
 * mfx.h -- C ABI of libmfx, fused transformer MLP and residual epilogues for
 * NVIDIA GB300 (sm_103a).
 *
 * Each entry point is one fused, bandwidth-bound pass written as a CUDA
 * kernel.  The operations are those of Megatron-LM's megatron/core/fusions/
 * as the web page "Megatron-LM operator fusion walkthrough"
 * (www.wmrh.cn/news/51426) describes them; each declaration cites the
 * section of that page ("fusions page §N") that defines it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are dense, contiguous, row-major.  `rows` is the token count
 *    (sequence x batch flattened), `cols` the hidden width.  The GLU ops take
 *    an input of width 2F whose first F columns are the activated ("gate")
 *    half and whose last F columns are the linear ("up") half.
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *    never allocates, frees or synchronises.  Any alignment is accepted; a
 *    16-byte aligned pointer with a width that is a multiple of 8 takes the
 *    fastest path, other cases take a slower path with the same results.
 *  - dtype codes: MFX_F32 or MFX_BF16.  Outputs take the dtype of the main
 *    input (y or x); the bias has that dtype too; the SwiGLU weight and its
 *    gradient are always fp32.  All arithmetic is fp32 inside the kernels,
 *    with one rounding at each output store.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous: they enqueue one kernel and return.
 *  - An empty tensor (rows == 0 or a zero width) is a no-op returning MFX_OK
 *    without reading any pointer.  Negative sizes, and sizes whose element
 *    count or byte count overflows int64, return MFX_ERR_SHAPE.
 *  - Return value: an mfx_status.  Arguments are validated on the host before
 *    anything is launched, so an error status means nothing was enqueued.
 *    MFX_ERR_CUDA reports a failed launch; mfx_last_cuda_error() then gives
 *    the cudaError_t (thread-local).  Besides that and the device error word
 *    described at mfx_device_error(), the library has no global state.
 *  - Thread safety: calls from several host threads are safe; calls that
 *    overlap on the GPU and write the same buffers race, as with any kernel.
 */
#ifndef MFX_H
#define MFX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { MFX_F32 = 0, MFX_BF16 = 1 } mfx_dtype;

typedef enum {
    MFX_OK = 0,
    MFX_ERR_NULL = 1,  /* a required pointer is NULL                          */
    MFX_ERR_SHAPE = 2, /* negative or overflowing sizes                        */
    MFX_ERR_DTYPE = 3, /* unknown dtype code                                   */
    MFX_ERR_PROB = 4,  /* dropout probability outside [0, 1) or NaN           */
    MFX_ERR_ALIAS = 5, /* buffers overlap in a way the op does not allow       */
    MFX_ERR_CUDA = 6,  /* the kernel launch failed (see mfx_last_cuda_error)   */
    MFX_ERR_DEVICE = 7, /* a kernel gave up a bounded wait (mfx_device_error)  */
    MFX_ERR_WORKSPACE = 8 /* workspace too small or not 16-byte aligned        */
} mfx_status;

/* ------------------------------------------------------------------------ */
/* Bias + GeLU (tanh approximation), fusions page §4.2 bias_gelu(bias, y) and */
/* §4.2 bias_gelu_back(g, bias, y).                                           */
/* ------------------------------------------------------------------------ */

/* out[r,c] = gelu(x), x = y[r,c] + bias[c],
 *   gelu(x) = x * 0.5 * (1 + tanh(0.79788456 * x * (1 + 0.044715 * x * x))).
 * y, out: [rows, cols] of dtype dt.  bias: [cols] of dtype dt, or NULL (no
 * bias).  out may equal y (in place); any other overlap -> MFX_ERR_ALIAS. */
int mfx_bias_gelu_fwd(int dt, int64_t rows, int64_t cols,
                      const void* bias, const void* y, void* out, void* stream);

/* dy[r,c] = g[r,c] * gelu'(x), x = y[r,c] + bias[c], with the page's
 * derivative of the tanh form (its constant 0.1070322243 = 3 * 0.79788456 *
 * 0.044715):  gelu'(x) = 0.5 x (1 - t^2)(0.79788456 + 0.1070322243 x^2)
 *                        + 0.5 (1 + t),  t = tanh(0.79788456 x (1 + 0.044715 x^2)).
 * g, y, dy: [rows, cols] of dtype dt; bias: [cols] or NULL.  The bias
 * gradient is the column sum of dy (the page's backward returns the same
 * tensor for input and bias); this call does not form it.  dy may equal g or
 * y; any other overlap -> MFX_ERR_ALIAS. */
int mfx_bias_gelu_bwd(int dt, int64_t rows, int64_t cols,
                      const void* g, const void* bias, const void* y, void* dy,
                      void* stream);

/* ------------------------------------------------------------------------ */
/* Bias + gated linear units, fusions page §2 (fused_bias_geglu,              */
/* fused_bias_swiglu with its weighted variant) and §9 (the weighted-SwiGLU   */
/* test).  The page names these ops; the split is: z = x + bias over the full */
/* width 2F, a = z[:, :F] is activated, b = z[:, F:] is linear.               */
/* ------------------------------------------------------------------------ */

/* out[r,c] = gelu(a) * b with the §4.2 tanh GeLU.
 * x: [rows, 2F]; bias: [2F] or NULL; out: [rows, F]; all dtype dt.
 * out must not overlap x -> MFX_ERR_ALIAS. */
int mfx_bias_geglu_fwd(int dt, int64_t rows, int64_t F,
                       const void* x, const void* bias, void* out, void* stream);

/* dx[r, c]   = g[r,c] * b * gelu'(a)
 * dx[r, F+c] = g[r,c] * gelu(a)
 * g: [rows, F]; x: [rows, 2F]; bias: [2F] or NULL; dx: [rows, 2F].
 * dx may equal x (in place); other overlaps -> MFX_ERR_ALIAS. */
int mfx_bias_geglu_bwd(int dt, int64_t rows, int64_t F,
                       const void* g, const void* x, const void* bias, void* dx,
                       void* stream);

/* out[r,c] = silu(a) * b * weight[r], silu(a) = a / (1 + exp(-a)).
 * weight: [rows] fp32 per-token weight, or NULL for the plain SwiGLU.
 * x: [rows, 2F]; bias: [2F] or NULL; out: [rows, F]; dtype dt.
 * out must not overlap x or weight -> MFX_ERR_ALIAS. */
int mfx_bias_swiglu_fwd(int dt, int64_t rows, int64_t F,
                        const void* x, const void* bias, const float* weight,
                        void* out, void* stream);

/* With gw = g[r,c] * weight[r] (or g[r,c] without weight), s = sigma(a):
 *   dx[r, c]    = gw * b * s * (1 + a * (1 - s))
 *   dx[r, F+c]  = gw * silu(a)
 *   dweight[r]  = sum_c g[r,c] * silu(a) * b        (fp32)
 * dweight: [rows] fp32, required iff weight != NULL (else MFX_ERR_NULL); the
 * row sum runs in a fixed order inside one thread block, so it is bitwise
 * reproducible run to run and GPU to GPU.  dx may equal x; other overlaps
 * -> MFX_ERR_ALIAS. */
int mfx_bias_swiglu_bwd(int dt, int64_t rows, int64_t F,
                        const void* g, const void* x, const void* bias,
                        const float* weight, void* dx, float* dweight, void* stream);

/* ------------------------------------------------------------------------ */
/* Weighted squared ReLU, fusions page §2 (fused_weighted_squared_relu, the  */
/* per-token weighted MoE activation named beside the weighted SwiGLU).  The */
/* page names the fusion without its formula; the reading here is the        */
/* squared ReLU scaled by the token's fp32 router weight, with no bias.      */
/* ------------------------------------------------------------------------ */

/* out[r,c] = relu(x[r,c])^2 * weight[r], relu(v) = max(v, 0) (NaN -> 0).
 * x, out: [rows, cols] of dtype dt; weight: [rows] fp32 (required).
 * out may equal x (in place); any other overlap of out with x or weight
 * -> MFX_ERR_ALIAS. */
int mfx_weighted_squared_relu_fwd(int dt, int64_t rows, int64_t cols,
                                  const void* x, const float* weight, void* out, void* stream);

/* dx[r,c]    = g[r,c] * weight[r] * 2 relu(x[r,c])           (dtype dt)
 * dweight[r] = sum_c g[r,c] * relu(x[r,c])^2                  (fp32)
 * g, x, dx: [rows, cols] of dtype dt; weight, dweight: [rows] fp32 (both
 * required).  One thread block owns each row's sum and adds it in a fixed
 * order, so dweight is bitwise reproducible.  dx may equal g or x; other
 * overlaps (dweight with anything, dx with weight) -> MFX_ERR_ALIAS. */
int mfx_weighted_squared_relu_bwd(int dt, int64_t rows, int64_t cols,
                                  const void* g, const void* x, const float* weight,
                                  void* dx, float* dweight, void* stream);

/* ------------------------------------------------------------------------ */
/* Scale-mask-softmax, fusions page §6.2-§6.3: ScaledSoftmax,                */
/* ScaledMaskedSoftmax and ScaledUpperTriangMaskedSoftmax, the three         */
/* autograd functions fused_softmax wraps around CUDA kernels, and the one   */
/* backward they share.  Softmax along the last dimension; fp32 arithmetic;  */
/* inputs and outputs in the dtype dt.  Unlike the page's kernels these take */
/* any row length, any sizes and any alignment (the page's kernels require   */
/* 16 < sk <= 4096 and sizes divisible by 4 and fall back to PyTorch         */
/* otherwise, §6.3).                                                         */
/* ------------------------------------------------------------------------ */

/* y = softmax(x * scale + mask) over the last dimension, x and y: [b, np,
 * sq, sk].  mask: NULL (ScaledSoftmax) or an ADDITIVE mask of dtype dt
 * (§6.2 describes it as a broadcastable additive mask) of shape [mask_b,
 * mask_np, mask_sq, sk], where each of mask_b, mask_np, mask_sq is 1
 * (broadcast) or equal to b, np, sq (else MFX_ERR_SHAPE); -inf excludes a
 * position (a boolean padding mask is the additive mask 0 / -inf).  A row
 * whose every score is -inf (nothing left) is all zeros.  Scores whose fp32
 * product x * scale overflows make their row NaN.  y may equal x (in place);
 * any other overlap of y with x or the mask -> MFX_ERR_ALIAS. */
int mfx_scaled_masked_softmax_fwd(int dt, int64_t b, int64_t np, int64_t sq, int64_t sk,
                                  const void* x, const void* mask,
                                  int64_t mask_b, int64_t mask_np, int64_t mask_sq,
                                  float scale, void* y, void* stream);

/* Causal: y = softmax over k of x * scale with k > q excluded, x and y:
 * [attn_batches, sq, sq] (the page's upper-triangle mask for GPT's causal
 * self-attention; sq == sk as §6.4's causal check demands).  Excluded
 * positions are written as exact zeros and are never read.  y may equal x;
 * other overlaps -> MFX_ERR_ALIAS. */
int mfx_scaled_upper_triang_masked_softmax_fwd(int dt, int64_t attn_batches, int64_t sq,
                                               const void* x, float scale, void* y, void* stream);

/* Backward of mfx_scaled_masked_softmax_fwd (with or without a mask): from
 * the forward's output y and the upstream gradient dy, both [rows, sk]
 * (rows = b * np * sq),
 *   dx[r, k] = scale * y[r, k] * (dy[r, k] - sum_j dy[r, j] * y[r, j]).
 * The row sum is accumulated with compensated (error-free) arithmetic.  dx
 * may equal dy or y (in place); other overlaps -> MFX_ERR_ALIAS. */
int mfx_scaled_masked_softmax_bwd(int dt, int64_t rows, int64_t sk,
                                  const void* dy, const void* y, float scale, void* dx, void* stream);

/* Backward of the causal forward, on [attn_batches, sq, sq]: the same
 * formula, with positions k > q written as exact zeros without reading dy
 * or y there. */
int mfx_scaled_upper_triang_masked_softmax_bwd(int dt, int64_t attn_batches, int64_t sq,
                                               const void* dy, const void* y, float scale,
                                               void* dx, void* stream);

/* ------------------------------------------------------------------------ */
/* Bias + dropout + residual add, fusions page §3.2-§3.3                     */
/* (_bias_dropout_add_func(x_with_bias, residual, prob, training) and its    */
/* two entry points bias_dropout_add_fused_train / _inference).              */
/* ------------------------------------------------------------------------ */

/* Training:  out = r~ + dropout(x + bias, p), where r~ is the residual cast
 * to x's dtype ("residual.to(x.dtype)", §3.2) and dropout keeps an element
 * with probability 1 - p and scales it by 1 / (1 - p) (computed in fp32).
 * x: [rows, cols] dtype x_dt; bias: [cols] x_dt or NULL; residual: [rows,
 * cols] dtype res_dt (either code); out: [rows, cols] x_dt; keep_mask:
 * [rows, cols] uint8, 1 = kept, 0 = dropped (a dropped element contributes
 * exactly +0, so out == r~ there).
 * Randomness: element (r, c) has global index e = elem_base + r * cols + c;
 * Philox4x32-10 (Salmon et al., SC'11) with key (lo32 seed, hi32 seed) and
 * counter (lo32 e/8, hi32 e/8, lo32 offset, hi32 offset) gives 128 bits, of
 * which 16-bit word e % 8 (little-endian) is the element's uniform u; the
 * element is kept iff u >= min(65535, ceil(p * 65536)).  The mask is thus a
 * pure function of (seed, offset, e): shards of one tensor processed with
 * their own elem_base reproduce the unsharded mask.
 * p must lie in [0, 1) (else MFX_ERR_PROB); p = 0 keeps everything.
 * out may equal x; out must not overlap residual or keep_mask, keep_mask
 * must not overlap any input -> MFX_ERR_ALIAS. */
int mfx_bias_dropout_add_train(int x_dt, int res_dt, int64_t rows, int64_t cols,
                               const void* x, const void* bias, const void* residual,
                               float p, uint64_t seed, uint64_t offset, uint64_t elem_base,
                               void* out, uint8_t* keep_mask, void* stream);

/* mfx_bias_dropout_add_train with the keep mask as bits instead of bytes:
 * bit (i mod 8) of keep_bits[i / 8] (least significant bit first) is the keep
 * flag of element i = r * cols + c of this call, so the mask takes
 * ceil(rows * cols / 8) bytes (the last byte's unused high bits are 0).  The
 * same elements are kept and out is the same bits as with the byte mask;
 * the mask traffic drops from 1 to 1/8 byte per element (bf16 x with an
 * fp32 residual: 8.125 instead of 9 bytes per element).  Fastest when x,
 * out and the residual are 16-byte aligned.  keep_bits must not overlap any
 * other buffer -> MFX_ERR_ALIAS; the other rules are the training call's. */
int mfx_bias_dropout_add_train_packed(int x_dt, int res_dt, int64_t rows, int64_t cols,
                                      const void* x, const void* bias, const void* residual,
                                      float p, uint64_t seed, uint64_t offset, uint64_t elem_base,
                                      void* out, uint8_t* keep_bits, void* stream);

/* Inference: x = (x + bias) + r~, IN PLACE in x (§3.2: when not training the
 * bias add, dropout and residual add all run in place).  p, seed and offset
 * are accepted for symmetry with the training call and ignored (p is still
 * validated).  x must not overlap residual or bias -> MFX_ERR_ALIAS. */
int mfx_bias_dropout_add_inference(int x_dt, int res_dt, int64_t rows, int64_t cols,
                                   void* x, const void* bias, const void* residual,
                                   float p, uint64_t seed, uint64_t offset, void* stream);

/* Backward of the training call (the gradients the fusions page's §3.4 unit
 * test compares between fused and unfused versions), given the upstream
 * gradient g = dL/dout [rows, cols] of dtype x_dt:
 *   dx[i]        = keep[i] ? g[i] * (1 / (1 - p)) : 0      (x_dt)
 *                  -- also the bias gradient before its column sum
 *   dresidual[i] = g[i] in the residual's dtype res_dt      (the cast's backward)
 * keep_mask: the forward's mask, or NULL to regenerate it from (seed, offset,
 * elem_base, p), which must then be the forward's values (no mask read: two
 * bytes per element less traffic in bf16).  dresidual may be NULL (not
 * written), or equal g when res_dt == x_dt (nothing to write).  dx may equal
 * g (in place); other overlaps -> MFX_ERR_ALIAS.  Bit-exact: fp32 multiply,
 * one rounding. */
int mfx_bias_dropout_add_bwd(int x_dt, int res_dt, int64_t rows, int64_t cols,
                             const void* g, const uint8_t* keep_mask,
                             float p, uint64_t seed, uint64_t offset, uint64_t elem_base,
                             void* dx, void* dresidual, void* stream);

/* mfx_bias_dropout_add_bwd reading the bit mask of
 * mfx_bias_dropout_add_train_packed (keep_bits, required): dx and dresidual
 * are the same bits as with the byte mask.  Fastest when g, dx, dresidual
 * and keep_bits are 16-byte aligned and rows * cols is a multiple of 8. */
int mfx_bias_dropout_add_bwd_packed(int x_dt, int res_dt, int64_t rows, int64_t cols,
                                    const void* g, const uint8_t* keep_bits, float p,
                                    void* dx, void* dresidual, void* stream);

/* ------------------------------------------------------------------------ */
/* Fused bias gradients.  The fusions page's backward hands one gradient      */
/* tensor to the input and to the broadcast bias (§4.3, "both return tmp"),  */
/* and autograd sums it over the rows.  These variants of the backward calls */
/* also write that column sum, dbias[c] = sum_r grad[r, c] of the gradient as */
/* stored (rounded to its dtype), without reading the gradient back: each    */
/* thread adds the values it stores for its columns into a partial sum, the  */
/* partials land in a caller-provided fp32 workspace, and a second small     */
/* kernel adds them per column in a fixed order (same bits run to run on a   */
/* given GPU model) and rounds once to the bias dtype.                       */
/*                                                                           */
/* Workspace protocol: call with workspace == NULL to get the required size  */
/* in *workspace_bytes (nothing is launched; sizes and dtype must be the     */
/* real ones, the current device is assumed); then call with a 16-byte       */
/* aligned device buffer of at least that size and its size in               */
/* *workspace_bytes (else MFX_ERR_WORKSPACE).  The buffer is scratch: its    */
/* contents on entry do not matter.  dbias has the gradient's dtype; with    */
/* rows == 0 it is set to zero.                                              */
/* ------------------------------------------------------------------------ */

/* mfx_bias_gelu_bwd, plus dbias[c] = sum_r dy[r, c] (dbias: [cols]). */
int mfx_bias_gelu_bwd_dbias(int dt, int64_t rows, int64_t cols,
                            const void* g, const void* bias, const void* y, void* dy,
                            void* dbias, void* workspace, size_t* workspace_bytes, void* stream);

/* The same as mfx_bias_gelu_bwd_dbias, for callers that cannot hand the
 * library a workspace: code whose device memory is all owned by a pool that
 * does not give library calls scratch buffers, code on a path where a device
 * allocation (which can synchronise the device) is not acceptable, and C
 * callers with no device allocator of their own.  The fusions page has no
 * counterpart; this is a calling convention, not another operation.
 *   - It allocates nothing.  The partial sums go to a fixed 4 MiB array
 *     inside the library, which every GPU that loads the library holds until
 *     the process exits.
 *   - When the size mfx_bias_gelu_bwd_dbias would ask for fits in the array
 *     (on a GB300 its pipelined partials take about 2.5 MB whatever the
 *     shape), the call runs exactly what that entry point runs: dy and dbias
 *     are the same bits.  Otherwise (a device with more resident threads)
 *     it runs the plain backward and the row-interleaved partial layout,
 *     min(rows, 64) partial sums per column, which needs
 *     min(rows, 64) x cols x 4 bytes: dy is still the same bits, dbias is
 *     the same sum in another fixed order (it may differ in the last bits).
 *     Every width up to 16384 columns is therefore accepted.  A problem that
 *     fits neither way returns MFX_ERR_WORKSPACE and launches nothing; use
 *     mfx_bias_gelu_bwd_dbias then.
 *   - The first call on each device looks up that device's array address
 *     (with that device current) and keeps it for later calls.
 *   - Every call uses the same array, so calls whose kernels overlap on the
 *     GPU (different streams, different host threads) race and give wrong
 *     results; serialise them.  Nothing from an earlier call needs clearing:
 *     each call writes every slot it reads. */
int mfx_bias_gelu_bwd_dbias_noalloc(int dt, int64_t rows, int64_t cols,
                                    const void* g, const void* bias, const void* y, void* dy,
                                    void* dbias, void* stream);

/* mfx_bias_geglu_bwd, plus dbias[c] = sum_r dx[r, c] over the full width 2F
 * (dbias: [2F], the gradient of the bias added before the split). */
int mfx_bias_geglu_bwd_dbias(int dt, int64_t rows, int64_t F,
                             const void* g, const void* x, const void* bias, void* dx,
                             void* dbias, void* workspace, size_t* workspace_bytes, void* stream);

/* mfx_bias_swiglu_bwd, plus dbias[c] = sum_r dx[r, c] (dbias: [2F]).  With a
 * weight the backward owns rows, so the partial sums come from one extra
 * read of dx. */
int mfx_bias_swiglu_bwd_dbias(int dt, int64_t rows, int64_t F,
                              const void* g, const void* x, const void* bias,
                              const float* weight, void* dx, float* dweight,
                              void* dbias, void* workspace, size_t* workspace_bytes, void* stream);

/* mfx_bias_dropout_add_bwd, plus dbias[c] = sum_r dx[r, c] (dbias: [cols]). */
int mfx_bias_dropout_add_bwd_dbias(int x_dt, int res_dt, int64_t rows, int64_t cols,
                                   const void* g, const uint8_t* keep_mask,
                                   float p, uint64_t seed, uint64_t offset, uint64_t elem_base,
                                   void* dx, void* dresidual, void* dbias,
                                   void* workspace, size_t* workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Status helpers                                                            */
/* ------------------------------------------------------------------------ */

/* Static English description of a status code (never NULL). */
const char* mfx_status_string(int status);

/* cudaError_t of the last MFX_ERR_CUDA returned on this host thread (0 if
 * none). */
int mfx_last_cuda_error(void);

/* Kernels that stream through shared memory wait on barriers for their own
 * bulk copies; every such wait is bounded (a few seconds), and a kernel whose
 * wait runs out stops early, leaving its outputs unfinished, and records a
 * nonzero code in a per-device error word.  This call synchronises the
 * current device, copies the word into *code (if code is not NULL), clears it
 * and returns MFX_ERR_DEVICE if it was nonzero, else MFX_OK.  A correct
 * program never sees a nonzero word; the word is the library's only device
 * state besides the kernels. */
int mfx_device_error(unsigned* code);

/* Library ABI version, (major << 16) | minor. */
int mfx_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MFX_H */
