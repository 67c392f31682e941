// sqrelu.cu -- weighted squared ReLU, forward and backward.
//
// Megatron-LM operator fusion walkthrough (www.wmrh.cn/news/51426), §2:
// fused_weighted_squared_relu, the MoE activation weighted per token, named
// beside the weighted SwiGLU.  The page only names it; the library reads it
// as out = relu(x)^2 * weight[r] (fp32 per-token weight, no bias), with
//   dx = 2 relu(x) * g * weight[r],   dweight[r] = sum_c g * relu(x)^2.
//
// Memory per element: forward reads x, writes out (2 x elem bytes); backward
// reads g, x, writes dx (3 x elem bytes); 4 bytes per row for the weight and
// 4 more for its gradient.
#include "mfx_device.cuh"
#include "mfx_host.h"
#include "mfx_pipe.cuh"

namespace mfx {
namespace {

__device__ unsigned g_device_error;

// The weight (a router probability, at most 1 in practice) multiplies first:
// (a w) a overflows only when the result does, where a a w would overflow
// for a large a and a small weight.  relu(NaN) is 0, as in the comparison
// form max(x, 0) evaluates to for an unordered x.
template <bool PRECISE>
__device__ __forceinline__ float sqrelu_fwd1(float x, float w)
{
    const float a = x > 0.0f ? x : 0.0f;
    return mul3<PRECISE>(a, w, a);
}

// dx for one element; *term = g * relu(x)^2, the weight-gradient term.  The
// factor 2 comes last (exact unless the result overflows), so 2 relu(x)
// cannot overflow on its own.
template <bool PRECISE>
__device__ __forceinline__ float sqrelu_bwd1(float x, float g, float w, float* term)
{
    const float a = x > 0.0f ? x : 0.0f;
    *term = g * a * a;
    return 2.0f * mul3<PRECISE>(g, w, a);
}

// ---------------------------------------------------------------------------
// Forward, pipelined: thread count a multiple of cols/8, so a thread's rows
// advance by S/(cols/8) with no division; x streams through the ring.
// ---------------------------------------------------------------------------
template <typename T>
struct FwdPipe {
    static constexpr int kU = 2;
    static constexpr uint32_t kSpan = kConsumers * 8 * sizeof(T);
    static constexpr uint32_t kStage = kU * kSpan;
    static constexpr int kStages = ring_stages(MFX_RING_KB_SQRELU_FWD * 1024, kStage);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kStage;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

template <typename T>
__global__ void __launch_bounds__(kPipeThreads, MFX_PIPE_MINB_GELU)
sqrelu_fwd_pipe(const T* x, const float* __restrict__ w, T* out, int64_t units, int64_t gpr)
{
    using P = FwdPipe<T>;
    constexpr int U = P::kU, NS = P::kStages;
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int64_t S = (int64_t)gridDim.x * kConsumers;
    const int64_t ub0 = (int64_t)blockIdx.x * kConsumers;
    const int64_t iters = units > ub0 ? (units - ub0 + U * S - 1) / (U * S) : 0;
    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) == 0) {
            const void* const base[1] = {x};
            const uint32_t ub[1] = {8u * (uint32_t)sizeof(T)};
            const uint32_t off[1] = {0u};
            flat_producer<NS, U, 1>(ring, data, P::kStage, base, ub, off, ub0, S, units, iters, &g_device_error);
        }
        return;
    }
    const int t = threadIdx.x;
    const int64_t u0 = ub0 + t;
    const int64_t row0 = u0 / gpr, drow = S / gpr;
    for (int64_t it = 0; it < iters; ++it) {
        float wk[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t u = u0 + (it * U + k) * S;
            wk[k] = u < units ? w[row0 + (it * U + k) * drow] : 0.0f;
        }
        if (!consumer_acquire<NS>(ring, it, &g_device_error))
            return;
        const unsigned char* st = data + (size_t)(it % NS) * P::kStage + t * 8 * sizeof(T);
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t u = u0 + (it * U + k) * S;
            if (u < units) {
                Raw8<T> rx;
                lds8(st + k * P::kSpan, rx);
                float f[8];
                widen8(rx, f);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    f[j] = sqrelu_fwd1<kPrecise>(f[j], wk[k]);
                narrow8(f, rx);
                st8(out + u * 8, rx);
            }
        }
        consumer_release<NS>(ring, it);
    }
}

// Generic forward: any width and alignment; element (r, c) of unit u is
// tracked incrementally.
template <typename T>
__global__ void __launch_bounds__(kThreads)
sqrelu_fwd_generic(const T* x, const float* __restrict__ w, T* out, int64_t n, int64_t cols, int64_t dcol,
                   int64_t drow)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t units = (n + 7) / 8;
    int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    int64_t r = (u * 8) / cols, c = (u * 8) % cols;
    for (; u < units; u += S) {
        const int64_t i0 = u * 8;
        const int cnt = n - i0 < 8 ? (int)(n - i0) : 8;
        float f[8];
        load8f(x + i0, false, cnt, f);
        int64_t rj = r, cj = c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < cnt)
                f[j] = sqrelu_fwd1<kPrecise>(f[j], w[rj]);
            if (++cj == cols) {
                cj = 0;
                ++rj;
            }
        }
        store8f(out + i0, false, cnt, f);
        c += dcol;
        r += drow;
        if (c >= cols) {
            c -= cols;
            ++r;
        }
    }
}

// ---------------------------------------------------------------------------
// Backward: blocks own rows (the weight gradient is one fixed-order sum per
// row, as in the weighted SwiGLU backward).  The pipelined form streams each
// row in chunks of 256 units of g and x; the generic form loads directly.
// ---------------------------------------------------------------------------
constexpr int kSqreluBwdKUnroll = MFX_SQRELU_BWD_K_UNROLL;  // copies of the unit code in the chunk loop

template <typename T>
struct BwdPipe {
    // units per consumer per stage: given for bf16, halved for fp32 so that a
    // stage keeps its bytes (two 64 KB stages at the default)
    static constexpr int kU = MFX_UNROLL_SQRELU_BWD * 2 / (int)sizeof(T) > 0 ? MFX_UNROLL_SQRELU_BWD * 2 / (int)sizeof(T) : 1;
    static constexpr uint32_t kSpan = kU * kConsumers * 8 * sizeof(T);
    static constexpr uint32_t kStage = 2 * kSpan;
    static constexpr int kStages = ring_stages(MFX_RING_KB_SQRELU * 1024, kStage);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kStage;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

// Fixed-order block sum of one value per consumer thread (xor tree per warp,
// then the warp sums in order); returns the sum in thread 0.
__device__ __forceinline__ float consumer_block_sum(float acc, float (&warp_sums)[2][kConsumerWarps], int parity,
                                                    int t)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if ((t & 31) == 0)
        warp_sums[parity][t >> 5] = acc;
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
    float s = 0.0f;
    if (t == 0)
#pragma unroll
        for (int i = 0; i < kConsumerWarps; ++i)
            s += warp_sums[parity][i];
    return s;
}

template <typename T>
__global__ void __launch_bounds__(kPipeThreads, MFX_PIPE_MINB_SQRELU)
sqrelu_bwd_pipe(const T* g, const T* x, const float* __restrict__ w, T* dx, float* __restrict__ dw, int64_t rows,
                int64_t cols)
{
    using P = BwdPipe<T>;
    constexpr int NS = P::kStages, U = P::kU;
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float warp_sums[2][kConsumerWarps];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int64_t gpr = cols / 8;
    const int64_t nchunk = (gpr + U * kConsumers - 1) / (U * kConsumers);
    const int64_t my_rows = rows > blockIdx.x ? (rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t iters = my_rows * nchunk;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) != 0)
            return;
        int64_t r = blockIdx.x, chunk = 0;  // advanced incrementally (no division)
        for (int64_t it = 0; it < iters; ++it) {
            const int s = (int)(it % NS);
            const int64_t n = it / NS;
            if (n > 0 && !mbar_wait(ring.empty(s), (uint32_t)((n - 1) & 1))) {
                atomicOr(&g_device_error, 2u);
                for (int64_t j = it - 1; j >= 0 && j > it - NS; --j)
                    if (!mbar_wait(ring.full((int)(j % NS)), (uint32_t)((j / NS) & 1)))
                        atomicOr(&g_device_error, 4u);
                return;
            }
            const int64_t c0 = chunk * U * kConsumers;
            const int64_t cnt = gpr - c0 < U * kConsumers ? gpr - c0 : U * kConsumers;
            const uint32_t bytes = (uint32_t)cnt * 8u * sizeof(T);
            mbar_arrive_expect_tx(ring.full(s), 2u * bytes);
            const uint32_t st = smem_addr(data + (size_t)s * P::kStage);
            bulk_g2s(st, x + r * cols + c0 * 8, bytes, ring.full(s));
            bulk_g2s(st + P::kSpan, g + r * cols + c0 * 8, bytes, ring.full(s));
            if (++chunk == nchunk) {
                chunk = 0;
                r += gridDim.x;
            }
        }
        return;
    }

    const int t = threadIdx.x;
    float acc = 0.0f;
    int parity = 0;
    bool dead = false;  // a consumer whose wait ran out still meets the row barrier
    int64_t r = blockIdx.x, chunk = 0;
    float wr = iters > 0 ? w[r] : 0.0f;  // the row's weight, reloaded when the row changes
    for (int64_t it = 0; it < iters; ++it) {
        if (!dead && !consumer_acquire<NS>(ring, it, &g_device_error))
            dead = true;
#pragma unroll(kSqreluBwdKUnroll)
        for (int k = 0; k < U; ++k) {
            const int64_t cu = k * kConsumers + t;           // unit within the chunk
            const int64_t cg = chunk * U * kConsumers + cu;  // unit within the row
            if (!dead && cg < gpr) {
                const unsigned char* st = data + (size_t)(it % NS) * P::kStage + cu * 8 * sizeof(T);
                Raw8<T> rx, rg;
                lds8(st, rx);
                lds8(st + P::kSpan, rg);
                float fx[8], fg[8];
                widen8(rx, fx);
                widen8(rg, fg);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float term;
                    fx[j] = sqrelu_bwd1<kPrecise>(fx[j], fg[j], wr, &term);
                    acc += term;
                }
                narrow8(fx, rx);
                st8(dx + r * cols + cg * 8, rx);
            }
        }
        if (!dead)
            consumer_release<NS>(ring, it);
        if (chunk == nchunk - 1) {
            const float s = consumer_block_sum(acc, warp_sums, parity, t);
            if (t == 0)
                dw[r] = s;
            acc = 0.0f;
            parity ^= 1;
            chunk = 0;
            r += gridDim.x;
            if (it + 1 < iters)
                wr = w[r];
        } else {
            ++chunk;
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
sqrelu_bwd_rows(const T* g, const T* x, const float* __restrict__ w, T* dx, float* __restrict__ dw, int64_t rows,
                int64_t cols)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    __shared__ float warp_sums[2][kThreads / 32];
    const int64_t gpr = (cols + 7) / 8;
    int parity = 0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, parity ^= 1) {
        const float wr = w[r];
        float acc = 0.0f;
        for (int64_t cg = threadIdx.x; cg < gpr; cg += kThreads) {
            const int64_t c0 = cg * 8;
            const int cnt = cols - c0 < 8 ? (int)(cols - c0) : 8;
            float fx[8], fg[8];
            load8f(x + r * cols + c0, false, cnt, fx);
            load8f(g + r * cols + c0, false, cnt, fg);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j < cnt) {
                    float term;
                    fx[j] = sqrelu_bwd1<kPrecise>(fx[j], fg[j], wr, &term);
                    acc += term;
                }
            }
            store8f(dx + r * cols + c0, false, cnt, fx);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if ((threadIdx.x & 31) == 0)
            warp_sums[parity][threadIdx.x >> 5] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < kThreads / 32; ++i)
                s += warp_sums[parity][i];
            dw[r] = s;
        }
    }
}

template <typename T>
int launch_fwd(const void* x, const float* w, void* out, int64_t rows, int64_t cols, cudaStream_t s)
{
    const T* xp = static_cast<const T*>(x);
    T* op = static_cast<T*>(out);
    const int64_t n = rows * cols;
    if (MFX_PIPE_GELU && cols % 8 == 0 && aligned16(x) && aligned16(out)) {
        const void* k = (const void*)sqrelu_fwd_pipe<T>;
        constexpr size_t smem = FwdPipe<T>::kSmem;
        const Grid grid = plan_grid_ex(k, kPipeThreads, smem, n / 8, cols / 8, true);
        if (grid.fixed) {
            sqrelu_fwd_pipe<T><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(xp, w, op, n / 8, cols / 8);
            return launch_status();
        }
    }
    const Grid grid = plan_grid((const void*)sqrelu_fwd_generic<T>, (n + 7) / 8, 0, false);
    const int64_t S8 = grid.blocks * kThreads * 8;
    sqrelu_fwd_generic<T><<<(unsigned)grid.blocks, kThreads, 0, s>>>(xp, w, op, n, cols, S8 % cols, S8 / cols);
    return launch_status();
}

template <typename T>
int launch_bwd(const void* g, const void* x, const float* w, void* dx, float* dw, int64_t rows, int64_t cols,
               cudaStream_t s)
{
    const T* gp = static_cast<const T*>(g);
    const T* xp = static_cast<const T*>(x);
    T* dxp = static_cast<T*>(dx);
    if (MFX_PIPE_WBWD && cols % 8 == 0 && aligned16(g) && aligned16(x) && aligned16(dx)) {
        const void* k = (const void*)sqrelu_bwd_pipe<T>;
        constexpr size_t smem = BwdPipe<T>::kSmem;
        const Grid grid = plan_grid_ex(k, kPipeThreads, smem, rows * kThreads, 0, false);
        sqrelu_bwd_pipe<T><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(gp, xp, w, dxp, dw, rows, cols);
        return launch_status();
    }
    const int64_t cap = (int64_t)sm_count() * blocks_per_sm((const void*)sqrelu_bwd_rows<T>);
    const unsigned blocks = (unsigned)(rows < cap ? rows : cap);
    sqrelu_bwd_rows<T><<<blocks, kThreads, 0, s>>>(gp, xp, w, dxp, dw, rows, cols);
    return launch_status();
}

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

unsigned take_device_error_sqrelu()
{
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess)
        return 0xFFu;
    if (v)
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    return v;
}

}  // namespace mfx

extern "C" int mfx_weighted_squared_relu_fwd(int dt, int64_t rows, int64_t cols, const void* x,
                                             const float* weight, void* out, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(dt, rows, cols, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!x || !weight || !out)
        return MFX_ERR_NULL;
    const int64_t b = n * dtype_bytes(dt);
    if (partial_overlap(x, b, out, b) || overlaps(weight, rows * 4, out, b))
        return MFX_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == MFX_BF16 ? launch_fwd<bf16>(x, weight, out, rows, cols, s)
                          : launch_fwd<float>(x, weight, out, rows, cols, s);
}

extern "C" int mfx_weighted_squared_relu_bwd(int dt, int64_t rows, int64_t cols, const void* g, const void* x,
                                             const float* weight, void* dx, float* dweight, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(dt, rows, cols, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!g || !x || !weight || !dx || !dweight)
        return MFX_ERR_NULL;
    const int64_t b = n * dtype_bytes(dt);
    if (partial_overlap(x, b, dx, b) || partial_overlap(g, b, dx, b) || overlaps(weight, rows * 4, dx, b) ||
        overlaps(dweight, rows * 4, dx, b) || overlaps(dweight, rows * 4, x, b) ||
        overlaps(dweight, rows * 4, g, b) || overlaps(dweight, rows * 4, weight, rows * 4))
        return MFX_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == MFX_BF16 ? launch_bwd<bf16>(g, x, weight, dx, dweight, rows, cols, s)
                          : launch_bwd<float>(g, x, weight, dx, dweight, rows, cols, s);
}
