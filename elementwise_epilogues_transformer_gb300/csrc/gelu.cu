// gelu.cu -- fused bias + tanh-GeLU forward and backward.
//
// Megatron-LM operator fusion walkthrough (www.wmrh.cn/news/51426), §4.2:
// bias_gelu(bias, y) adds the bias and applies
//     x * 0.5 * (1 + tanh(0.79788456 * x * (1 + 0.044715 * x * x)));
// bias_gelu_back(g, bias, y) re-adds the bias and multiplies g by the
// hand-derived derivative that uses 0.1070322243.  One pass over memory each:
// the forward reads y and writes out (2 x elem bytes per element), the
// backward reads g and y and writes dy (3 x elem bytes per element).
#include "mfx_device.cuh"
#include "mfx_host.h"

namespace mfx {
namespace {

constexpr int kUnroll = MFX_UNROLL_GELU;

// ---------------------------------------------------------------------------
// Fixed-column kernels: rows*cols is a multiple of 8, every pointer is
// 16-byte aligned and the thread count is a multiple of cols/8, so thread t
// always works on columns [8 (t mod cols/8), +8) and keeps their bias in
// registers.  Unit u = elements [8u, 8u + 8).
// ---------------------------------------------------------------------------
template <typename T, bool GRAD>
__global__ void __launch_bounds__(kThreads, MFX_MINB_GELU)
gelu_fixed(const T* g, const T* y, const T* __restrict__ bias, T* out, int64_t units, int64_t cols)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    float b[8];
    bias8(bias, (u * 8) % cols, b);
    // warp k (< kUnroll) prefetches the block's k-th slice of the next iteration
    const int wk = threadIdx.x >> 5;
    const bool pf_warp = wk < kUnroll;
    const int64_t pf_off = (int64_t)(kUnroll + wk) * S - threadIdx.x;

    for (; u + (kUnroll - 1) * S < units; u += kUnroll * S) {
        prefetch_block_span<MFX_PREFETCH_GELU != 0>(y, u + pf_off, units, 8 * sizeof(T), pf_warp);
        if (GRAD)
            prefetch_block_span<MFX_PREFETCH_GELU != 0>(g, u + pf_off, units, 8 * sizeof(T), pf_warp);
        Raw8<T> ry[kUnroll], rg[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            ld8(y + (u + k * S) * 8, ry[k]);
            if (GRAD)
                ld8(g + (u + k * S) * 8, rg[k]);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            float f[8], gf[8];
            widen8(ry[k], f);
            if (GRAD)
                widen8(rg[k], gf);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = f[j] + b[j];
                if (GRAD) {
                    float d;
                    gelu_sigma<kPrecise, true>(x, &d);
                    f[j] = d * gf[j];
                } else {
                    f[j] = x * gelu_sigma<kPrecise, false>(x, nullptr);
                }
            }
            narrow8(f, ry[k]);
            st8(out + (u + k * S) * 8, ry[k]);
        }
    }
    for (; u < units; u += S) {
        Raw8<T> ry, rg;
        ld8(y + u * 8, ry);
        if (GRAD)
            ld8(g + u * 8, rg);
        float f[8], gf[8];
        widen8(ry, f);
        if (GRAD)
            widen8(rg, gf);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float x = f[j] + b[j];
            if (GRAD) {
                float d;
                gelu_sigma<kPrecise, true>(x, &d);
                f[j] = d * gf[j];
            } else {
                f[j] = x * gelu_sigma<kPrecise, false>(x, nullptr);
            }
        }
        narrow8(f, ry);
        st8(out + u * 8, ry);
    }
}

// ---------------------------------------------------------------------------
// Generic kernels: any width (including widths that are not multiples of 8,
// whose rows straddle units), any alignment.  The unit's first column is
// tracked incrementally (dcol = 8 S mod cols); the bias is gathered per
// element; `vec` selects 16-byte accesses when every pointer is aligned; the
// last unit may hold fewer than 8 elements.
// ---------------------------------------------------------------------------
template <typename T, bool GRAD>
__global__ void __launch_bounds__(kThreads)
gelu_generic(const T* g, const T* y, const T* __restrict__ bias, T* out, int64_t n, int64_t cols,
             int64_t dcol, bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t units = (n + 7) / 8;
    int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    int64_t c = (u * 8) % cols;
    for (; u < units; u += S) {
        const int64_t i0 = u * 8;
        const int cnt = n - i0 < 8 ? (int)(n - i0) : 8;
        float f[8], gf[8];
        load8f(y + i0, vec, cnt, f);
        if (GRAD)
            load8f(g + i0, vec, cnt, gf);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int64_t col = c + j;
            while (col >= cols)
                col -= cols;
            const float x = f[j] + bias1(bias, col);
            if (GRAD) {
                float d;
                gelu_sigma<kPrecise, true>(x, &d);
                f[j] = d * gf[j];
            } else {
                f[j] = x * gelu_sigma<kPrecise, false>(x, nullptr);
            }
        }
        store8f(out + i0, vec, cnt, f);
        c += dcol;
        if (c >= cols)
            c -= cols;
    }
}

template <typename T, bool GRAD>
int launch(const void* g, const void* bias, const void* y, void* out, int64_t n, int64_t cols,
           cudaStream_t stream)
{
    const T* gp = static_cast<const T*>(g);
    const T* yp = static_cast<const T*>(y);
    const T* bp = static_cast<const T*>(bias);
    T* op = static_cast<T*>(out);
    const bool vec = aligned16(y) && aligned16(out) && (!GRAD || aligned16(g));
    const bool fixed_ok = vec && cols % 8 == 0 && (!bias || aligned16(bias));
    if (fixed_ok) {
        const Grid grid = plan_grid((const void*)gelu_fixed<T, GRAD>, n / 8, cols / 8, true);
        if (grid.fixed) {
            gelu_fixed<T, GRAD><<<(unsigned)grid.blocks, kThreads, 0, stream>>>(gp, yp, bp, op, n / 8, cols);
            return launch_status();
        }
    }
    const Grid grid = plan_grid((const void*)gelu_generic<T, GRAD>, (n + 7) / 8, 0, false);
    const int64_t dcol = (grid.blocks * kThreads * 8) % cols;
    gelu_generic<T, GRAD><<<(unsigned)grid.blocks, kThreads, 0, stream>>>(gp, yp, bp, op, n, cols, dcol, vec);
    return launch_status();
}

// Shared validation of the two entry points; returns MFX_OK and sets *n, or
// the error status.  `n_out` == 0 means nothing to do.
int check(int dt, int64_t rows, int64_t cols, int64_t* n_out)
{
    *n_out = 0;
    if (!valid_dtype(dt))
        return MFX_ERR_DTYPE;
    if (rows < 0 || cols < 0)
        return MFX_ERR_SHAPE;
    int64_t n = 0, bytes = 0;
    if (!mul_ok(rows, cols, &n) || !mul_ok(n, 16, &bytes))
        return MFX_ERR_SHAPE;
    *n_out = n;
    return MFX_OK;
}

}  // namespace
}  // namespace mfx

extern "C" int mfx_bias_gelu_fwd(int dt, int64_t rows, int64_t cols, const void* bias,
                                 const void* y, void* out, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(dt, rows, cols, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!y || !out)
        return MFX_ERR_NULL;
    const int64_t es = dtype_bytes(dt), bytes = n * es;
    if (partial_overlap(y, bytes, out, bytes) || overlaps(bias, cols * es, out, bytes))
        return MFX_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == MFX_BF16 ? launch<bf16, false>(nullptr, bias, y, out, n, cols, s)
                          : launch<float, false>(nullptr, bias, y, out, n, cols, s);
}

extern "C" int mfx_bias_gelu_bwd(int dt, int64_t rows, int64_t cols, const void* g,
                                 const void* bias, const void* y, void* dy, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(dt, rows, cols, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!g || !y || !dy)
        return MFX_ERR_NULL;
    const int64_t es = dtype_bytes(dt), bytes = n * es;
    if (partial_overlap(g, bytes, dy, bytes) || partial_overlap(y, bytes, dy, bytes) ||
        overlaps(bias, cols * es, dy, bytes))
        return MFX_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == MFX_BF16 ? launch<bf16, true>(g, bias, y, dy, n, cols, s)
                          : launch<float, true>(g, bias, y, dy, n, cols, s);
}
