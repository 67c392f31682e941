// gelu.cu -- fused bias + tanh-GeLU forward and backward.
//
// Megatron-LM operator fusion walkthrough (www.wmrh.cn/news/51426), §4.2:
// bias_gelu(bias, y) adds the bias and applies
//     x * 0.5 * (1 + tanh(0.79788456 * x * (1 + 0.044715 * x * x)));
// bias_gelu_back(g, bias, y) re-adds the bias and multiplies g by the
// hand-derived derivative that uses 0.1070322243.  One pass over memory each:
// the forward reads y and writes out (2 x elem bytes per element), the
// backward reads g and y and writes dy (3 x elem bytes per element).
#include <mutex>

#include "mfx_device.cuh"
#include "mfx_host.h"
#include "mfx_pipe.cuh"

namespace mfx {
namespace {

constexpr int kUnroll = MFX_UNROLL_GELU;

// Timed-out waits of this file's pipelined kernel (see mfx_device_error).
__device__ unsigned g_device_error;

// The forward of one element x = y + bias: the precise tier for fp32
// outputs; for bf16 the fast tier, as the fixed step sequence of
// gelu_fwd_fast (the same bits as its paired form) when the pipeline runs
// pairs, else as written in gelu_sigma (the compiler may fuse its steps).
template <bool PRECISE>
__device__ __forceinline__ float gelu_fwd1(float x)
{
    if constexpr (!PRECISE && MFX_GELU_FWD_EXPLICIT)
        return gelu_fwd_fast(x);
    else
        return x * gelu_sigma<PRECISE, false, 1>(x, nullptr);
}

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
                    f[j] = gelu_fwd1<kPrecise>(x);
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
                f[j] = gelu_fwd1<kPrecise>(x);
            }
        }
        narrow8(f, ry);
        st8(out + u * 8, ry);
    }
}

// ---------------------------------------------------------------------------
// Pipelined fixed-column kernel: the unit ownership of gelu_fixed, with the
// block's 256-unit spans of y (and g) arriving in a shared-memory ring from
// the producer warp's bulk copies (see mfx_pipe.cuh).
// ---------------------------------------------------------------------------
// Spans per stage, and copies of the unit code in the span loop (the
// forward's loop stays rolled: its code is long, and measured faster with a
// small instruction footprint and many spans per stage; its span count is
// given for bf16 and halved for fp32, so that a stage keeps its bytes).
constexpr int kGeluFwdU = MFX_UNROLL_GELU_FWD_PIPE, kGeluBwdU = MFX_UNROLL_GELU_PIPE;
constexpr int kGeluFwdKUnroll = MFX_GELU_FWD_K_UNROLL;
constexpr int kGeluBwdKUnroll = MFX_GELU_BWD_K_UNROLL;

template <typename T, bool GRAD, bool DB = false>
struct GeluPipe {
    static constexpr uint32_t kSpan = kConsumers * 8 * sizeof(T);
    // spans are given for bf16 and halved for fp32, so a stage keeps its bytes
    // (four fp32 spans of y and g made 64 KB stages: one block per SM)
    static constexpr int kU0 = GRAD ? (DB ? MFX_UNROLL_GELU_DB_PIPE : kGeluBwdU) : kGeluFwdU;
    static constexpr int kU = kU0 * 2 / (int)sizeof(T) > 0 ? kU0 * 2 / (int)sizeof(T) : 1;
    static constexpr uint32_t kStage = kU * kSpan * (GRAD ? 2 : 1);
    static constexpr int kStages =
        ring_stages((GRAD ? (DB ? MFX_RING_KB_GELU_DB : MFX_RING_KB_GELU) : MFX_RING_KB_GELU_FWD) * 1024, kStage);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kStage;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

// Elements [i0, i0 + cnt) one at a time (the first in column c), with the
// per-element arithmetic of the unit code: the head and tail of a pipelined
// call, whose elements are not whole 16-byte units.
template <typename T, bool GRAD>
__device__ __forceinline__ void gelu_elems(const T* g, const T* y, const T* __restrict__ bias, T* out, int64_t i0,
                                           int cnt, int64_t c, int64_t cols)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    for (int j = 0; j < cnt; ++j) {
        const float x = load1(y + i0 + j) + bias1(bias, c);
        float r;
        if (GRAD) {
            float d;
            gelu_sigma<kPrecise, true>(x, &d);
            r = d * load1(g + i0 + j);
        } else {
            r = gelu_fwd1<kPrecise>(x);
        }
        store1(out + i0 + j, r);
        if (++c == cols)
            c = 0;
    }
}

// Any width and any common misalignment: g, y and out point at the first
// element of the 16-byte aligned body, whose unit u (elements [8u, 8u + 8))
// starts in column (c_off + 8u) mod cols; S (a multiple of cols / gcd(cols,
// 8)) is the unit stride, so consumer thread g = blockIdx * 256 + t < S
// keeps one column phase and its bias in registers, and threads from S on
// own no units.  The `head` elements before the body and the `tail` after
// its `units` units are done one by one by thread 0 of block 0.
// With DB (cols % 8 == 0, no head or tail), each consumer also adds the
// values it stores into 8 partial column sums and writes them to
// ws[lane][columns], lane = first unit / (cols/8).
template <typename T, bool GRAD, bool DB = false>
__global__ void __launch_bounds__(kPipeThreads, GRAD ? MFX_PIPE_MINB_GELU : MFX_PIPE_MINB_GELU_FWD)
gelu_pipe(const T* g, const T* y, const T* __restrict__ bias, T* out, int64_t units, int64_t cols, int64_t S,
          int head, int tail, int64_t c_off, float* __restrict__ ws = nullptr)
{
    using P = GeluPipe<T, GRAD, DB>;
    constexpr int U = P::kU, NS = P::kStages;
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int64_t ub0 = (int64_t)blockIdx.x * kConsumers;
    const int64_t iters = units > ub0 ? (units - ub0 + U * S - 1) / (U * S) : 0;
    const uint32_t active = S - ub0 < kConsumers ? (uint32_t)(S - ub0) : (uint32_t)kConsumers;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) == 0) {
            if (GRAD) {
                const void* const base[2] = {y, g};
                const uint32_t ub[2] = {8u * (uint32_t)sizeof(T), 8u * (uint32_t)sizeof(T)};
                const uint32_t off[2] = {0u, U * P::kSpan};
                flat_producer<NS, U, 2>(ring, data, P::kStage, base, ub, off, ub0, S, units, iters, &g_device_error,
                                        active);
            } else {
                const void* const base[1] = {y};
                const uint32_t ub[1] = {8u * (uint32_t)sizeof(T)};
                const uint32_t off[1] = {0u};
                flat_producer<NS, U, 1>(ring, data, P::kStage, base, ub, off, ub0, S, units, iters, &g_device_error,
                                        active);
            }
        }
        return;
    }

    const int t = threadIdx.x;
    const int64_t u0 = ub0 + t;
    const bool on = u0 < S;
    float b[8], acc[8];
    bias8_at(bias, (c_off + (u0 % cols) * 8) % cols, cols, b);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc[j] = 0.0f;
    // this thread's units are u0 + j S, j < nj; its output advances S units per j
    const int64_t nj = on && units > u0 ? (units - u0 + S - 1) / S : 0;
    T* po = out + u0 * 8;
    const int64_t pstep = S * 8;
    for (int64_t it = 0; it < iters; ++it) {
        if (!consumer_acquire<NS>(ring, it, &g_device_error))
            return;
        const unsigned char* st = data + (size_t)(it % NS) * P::kStage + t * 8 * sizeof(T);
        const int jl = (int)(nj - it * U < U ? nj - it * U : U);  // spans of this stage in range
#pragma unroll(GRAD ? (DB ? U : kGeluBwdKUnroll) : kGeluFwdKUnroll)
        for (int k = 0; k < U; ++k) {
            T* const dst = po + k * pstep;
            if ((GRAD ? MFX_GELU_SPAN_COUNT_BWD : MFX_GELU_SPAN_COUNT_FWD) ? k < jl
                                                                          : on && u0 + (it * U + k) * S < units) {
                Raw8<T> ry, rg;
                lds8(st + k * P::kSpan, ry);
                if (GRAD)
                    lds8(st + (U + k) * P::kSpan, rg);
                float f[8], gf[8];
                if constexpr (!GRAD && !kPrecise && MFX_GELU_FWD_PAIRED) {
                    // bf16 forward on packed pairs (the same bits as gelu_fwd1)
                    uint32_t w[4] = {ry.v.x, ry.v.y, ry.v.z, ry.v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 v = gelu_fwd_fast2(add2(widen2(w[i]), make_float2(b[2 * i], b[2 * i + 1])));
                        w[i] = pack_bf16x2(v.x, v.y);
                    }
                    ry.v = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
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
                            f[j] = gelu_fwd1<kPrecise>(x);
                        }
                    }
                    narrow8(f, ry);
                }
                st8(dst, ry);
                if (DB) {
                    widen8(ry, f);  // the stored values
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[j] += f[j];
                }
            }
        }
        consumer_release<NS>(ring, it);
        po += U * pstep;
    }
    if (blockIdx.x == 0 && t == 0) {
        gelu_elems<T, GRAD>(g, y, bias, out, -head, head, 0, cols);
        gelu_elems<T, GRAD>(g, y, bias, out, units * 8, tail, (c_off + (units % cols) * 8) % cols, cols);
    }
    if (DB && on) {
        pdl_launch_dependents();
        const int64_t gpr = cols / 8;
        float4* w4 = reinterpret_cast<float4*>(ws + (u0 / gpr) * cols + (u0 % gpr) * 8);
        w4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        w4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
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
                f[j] = gelu_fwd1<kPrecise>(x);
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
    // the pipeline takes any width when every pointer sits the same whole
    // number of elements below a 16-byte boundary (those elements are its head)
    const uintptr_t mis = reinterpret_cast<uintptr_t>(y) & 15u;
    const bool same = (reinterpret_cast<uintptr_t>(out) & 15u) == mis &&
                      (!GRAD || (reinterpret_cast<uintptr_t>(g) & 15u) == mis) && mis % sizeof(T) == 0;
    const int head = (int)(((16u - mis) & 15u) / sizeof(T));
    if (same && MFX_PIPE_GELU && n - head >= 8) {
        const void* k = (const void*)gelu_pipe<T, GRAD>;
        constexpr size_t smem = GeluPipe<T, GRAD>::kSmem;
        const int64_t units = (n - head) / 8;
        const Grid grid = plan_fixed_any(k, kPipeThreads, smem, units, cols);
        if (grid.fixed) {
            gelu_pipe<T, GRAD><<<(unsigned)grid.blocks, kPipeThreads, smem, stream>>>(
                GRAD ? gp + head : gp, yp + head, bp, op + head, units, cols, grid.S, head, (int)((n - head) % 8),
                head % cols);
            return launch_status();
        }
    }
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

// bias-GeLU backward plus the fused bias gradient.  Without `allow_pipe`
// the pipelined kernel is not planned: dy comes from the plain backward and
// the partials from the row-interleaved column pass (min(rows, 64) lanes),
// whose workspace does not grow with the pipeline's grid.
template <typename T>
int launch_dbias(const void* g, const void* bias, const void* y, void* dy, void* dbias, int64_t n, int64_t cols,
                 int64_t rows, void* workspace, size_t* ws_bytes, cudaStream_t stream, bool allow_pipe = true)
{
    const void* k = (const void*)gelu_pipe<T, true, true>;
    constexpr size_t smem = GeluPipe<T, true, true>::kSmem;
    int64_t J_pipe = 0;
    Grid grid;
    if (MFX_PIPE_GELU && allow_pipe && cols % 8 == 0) {
        grid = plan_fixed_any(k, kPipeThreads, smem, n / 8, cols);
        if (grid.fixed)
            J_pipe = grid.S / (cols / 8);
    }
    const int64_t J_gen = dbias_generic_lanes(rows);
    bool query = false;
    int st = dbias_workspace(J_pipe > J_gen ? J_pipe : J_gen, cols, workspace, ws_bytes, &query);
    if (st != MFX_OK || query)
        return st;
    float* ws = static_cast<float*>(workspace);
    const bool pipe_ok = J_pipe > 0 && aligned16(g) && aligned16(y) && aligned16(dy) && (!bias || aligned16(bias));
    if (pipe_ok) {
        gelu_pipe<T, true, true><<<(unsigned)grid.blocks, kPipeThreads, smem, stream>>>(
            static_cast<const T*>(g), static_cast<const T*>(y), static_cast<const T*>(bias), static_cast<T*>(dy),
            n / 8, cols, grid.S, 0, 0, 0, ws);
        st = launch_status();
        return st != MFX_OK ? st : launch_dbias_finish(dtype_code<T>(), ws, J_pipe, cols, dbias, stream);
    }
    st = launch<T, true>(g, bias, y, dy, n, cols, stream);
    if (st == MFX_OK)
        st = launch_column_partials(dtype_code<T>(), dy, rows, cols, J_gen, ws, stream);
    return st != MFX_OK ? st : launch_dbias_finish(dtype_code<T>(), ws, J_gen, cols, dbias, stream);
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

unsigned take_device_error_gelu()
{
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess)
        return 0xFFu;
    if (v)
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    return v;
}

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

namespace mfx {
namespace {

// The workspace entry point's body; `allow_pipe` = false restricts it to the
// row-interleaved partial layout (used by the allocation-free variant).
int gelu_bwd_dbias(int dt, int64_t rows, int64_t cols, const void* g, const void* bias, const void* y, void* dy,
                   void* dbias, void* workspace, size_t* workspace_bytes, void* stream, bool allow_pipe)
{
    int64_t n = 0;
    int st = check(dt, rows, cols, &n);
    if (st != MFX_OK)
        return st;
    if (!workspace_bytes)
        return MFX_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t es = dtype_bytes(dt);
    if (n == 0) {
        if (!workspace) {
            *workspace_bytes = 0;
            return MFX_OK;
        }
        if (cols == 0)
            return MFX_OK;
        if (!dbias)
            return MFX_ERR_NULL;
        return cudaMemsetAsync(dbias, 0, (size_t)(cols * es), s) == cudaSuccess ? MFX_OK
                                                                               : cuda_failure(cudaGetLastError());
    }
    if (workspace && (!g || !y || !dy || !dbias))
        return MFX_ERR_NULL;
    const int64_t bytes = n * es;
    if (workspace && (partial_overlap(g, bytes, dy, bytes) || partial_overlap(y, bytes, dy, bytes) ||
                      overlaps(bias, cols * es, dy, bytes) || overlaps(dbias, cols * es, dy, bytes) ||
                      overlaps(dbias, cols * es, g, bytes) || overlaps(dbias, cols * es, y, bytes) ||
                      overlaps(dbias, cols * es, bias, cols * es) ||
                      overlaps(workspace, (int64_t)*workspace_bytes, dy, bytes) ||
                      overlaps(workspace, (int64_t)*workspace_bytes, dbias, cols * es) ||
                      overlaps(workspace, (int64_t)*workspace_bytes, g, bytes) ||
                      overlaps(workspace, (int64_t)*workspace_bytes, y, bytes)))
        return MFX_ERR_ALIAS;
    return dt == MFX_BF16
               ? launch_dbias<bf16>(g, bias, y, dy, dbias, n, cols, rows, workspace, workspace_bytes, s, allow_pipe)
               : launch_dbias<float>(g, bias, y, dy, dbias, n, cols, rows, workspace, workspace_bytes, s, allow_pipe);
}

}  // namespace
}  // namespace mfx

extern "C" int mfx_bias_gelu_bwd_dbias(int dt, int64_t rows, int64_t cols, const void* g, const void* bias,
                                       const void* y, void* dy, void* dbias, void* workspace,
                                       size_t* workspace_bytes, void* stream)
{
    return mfx::gelu_bwd_dbias(dt, rows, cols, g, bias, y, dy, dbias, workspace, workspace_bytes, stream, true);
}

// ---------------------------------------------------------------------------
// Allocation-free bias-GeLU backward with the bias gradient.
//
// The partial column sums live in one fixed array inside the library
// instead of a caller's workspace.  The array is a device symbol: in host
// code its name is only a stand-in, so its device address is looked up with
// cudaGetSymbolAddress, once per device with that device current, on the
// first call on that device, and passed to the kernels.  Every call shares
// the array; nothing in it needs to start at zero, because each call writes
// every slot it later reads.  A problem whose pipelined partials do not fit
// (they take about 32 bytes per resident consumer thread: 2.5 MB on a GB300,
// more on a device with more resident threads) runs the row-interleaved
// layout instead, min(rows, 64) partials per column.
// ---------------------------------------------------------------------------
namespace mfx {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kNoAllocDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_address[kNoAllocDevices] = {};

int noalloc_scratch(void** address)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_failure(e);
    if (dev < 0 || dev >= kNoAllocDevices)
        return cuda_failure(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_address[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return cuda_failure(e);
        g_noalloc_address[dev] = p;
    }
    *address = g_noalloc_address[dev];
    return MFX_OK;
}

}  // namespace
}  // namespace mfx

extern "C" int mfx_bias_gelu_bwd_dbias_noalloc(int dt, int64_t rows, int64_t cols, const void* g,
                                               const void* bias, const void* y, void* dy, void* dbias,
                                               void* stream)
{
    using namespace mfx;
    // how much scratch this problem needs (nothing is launched by a query):
    // the workspace entry point's own plan if it fits, else the
    // row-interleaved layout if that fits, else a refusal
    bool allow_pipe = true;
    size_t need = 0;
    int st = gelu_bwd_dbias(dt, rows, cols, g, bias, y, dy, dbias, nullptr, &need, stream, true);
    if (st != MFX_OK)
        return st;
    if (need > kNoAllocScratchBytes) {
        allow_pipe = false;
        st = gelu_bwd_dbias(dt, rows, cols, g, bias, y, dy, dbias, nullptr, &need, stream, false);
        if (st != MFX_OK)
            return st;
        if (need > kNoAllocScratchBytes)
            return MFX_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != MFX_OK)
        return st;
    size_t have = kNoAllocScratchBytes;
    return gelu_bwd_dbias(dt, rows, cols, g, bias, y, dy, dbias, scratch, &have, stream, allow_pipe);
}
