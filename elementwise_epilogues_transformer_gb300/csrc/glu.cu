// glu.cu -- fused bias + gated linear units: GEGLU and SwiGLU (with the
// optional per-token weight), forward and backward.
//
// Megatron-LM operator fusion walkthrough (www.wmrh.cn/news/51426): §2 lists
// fused_bias_geglu and fused_bias_swiglu (with its weighted variant) as the
// sister fusions of §4's bias-GeLU; §9 describes the weighted-SwiGLU test,
// weighted(x, w) == swiglu(x) * w, with input and weight gradients.  The page
// does not print these ops; the library reads them as: z = x + bias over the
// full width 2F, a = z[:, :F] goes through the activation (the §4.2 tanh GeLU
// for GEGLU, SiLU for SwiGLU) and multiplies b = z[:, F:].
//
// Memory per output element: the forward reads a and b and writes out
// (3 x elem bytes); the backward reads g, a, b and writes da, db (5 x elem
// bytes).  The weight adds 4 bytes per row, its gradient 4 more.
#include "mfx_device.cuh"
#include "mfx_host.h"
#include "mfx_pipe.cuh"

namespace mfx {
namespace {

enum Kind { GEGLU = 0, SWIGLU = 1 };

// Timed-out waits of this file's pipelined kernels (see mfx_device_error).
__device__ unsigned g_device_error;

// Forward of one element: act(a) * b, times the row weight when weighted.
template <int KIND, bool PRECISE, bool WEIGHTED>
__device__ __forceinline__ float glu_fwd1(float a, float b, float w)
{
    float s;
    if (KIND == GEGLU) {
        s = gelu_sigma<PRECISE, false, MFX_RCP_GEGLU>(a, nullptr);  // gelu(a) = a s
    } else {
        float oms;
        constexpr int steps = WEIGHTED ? MFX_RCP_SWIGLU_W : MFX_RCP_SWIGLU;
        silu_sigma<PRECISE, steps>(a, &s, &oms);  // silu(a) = a s
    }
    // the bounded factor (s in [0, 1]) multiplies first, so a huge a whose
    // activation vanishes gives 0, not inf * 0
    return WEIGHTED ? mul4<PRECISE>(s, a, b, w) : mul3<PRECISE>(s, a, b);
}

// Backward of one element with upstream g and row weight w (1 when not
// weighted): writes da, db; returns act(a) * b, the weight-gradient term
// before the factor g.
template <int KIND, bool PRECISE, bool WEIGHTED>
__device__ __forceinline__ float glu_bwd1(float a, float b, float g, float w, float* da, float* db)
{
    if (KIND == GEGLU) {
        float d;
        const float s = gelu_sigma<PRECISE, true>(a, &d);
        *da = mul3<PRECISE>(d, g, b);   // bounded factors first (see glu_fwd1)
        *db = mul3<PRECISE>(s, g, a);
        return s * a * b;
    } else {
        float s, oms;
        constexpr bool hw = WEIGHTED ? MFX_HWRCP_WBWD != 0 : MFX_HWRCP_SWIGLU_BWD != 0;
        silu_sigma<PRECISE, hw ? 0 : 2>(a, &s, &oms);
        const float dsilu = fmaf(a, s * oms, s);      // sigma(a) (1 + a (1 - sigma(a)))
        if (WEIGHTED) {
            *da = mul4<PRECISE>(dsilu, g, b, w);
            *db = mul4<PRECISE>(s, g, a, w);
        } else {
            *da = mul3<PRECISE>(dsilu, g, b);
            *db = mul3<PRECISE>(s, g, a);
        }
        return s * a * b;
    }
}

constexpr int kUnrollFwd = MFX_UNROLL_GLU_FWD;
constexpr int kUnrollBwd = MFX_UNROLL_GLU_BWD;

// ---------------------------------------------------------------------------
// Fixed-column forward: F % 8 == 0, every pointer 16-byte aligned, thread
// count S a multiple of F/8.  Thread t owns output columns [8 cg, 8 cg + 8),
// cg = t mod (F/8), in rows r = t div (F/8) + k S/(F/8); it keeps both halves'
// bias for those columns in registers.
// ---------------------------------------------------------------------------
template <typename T, int KIND, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads, MFX_MINB_GLU)
glu_fwd_fixed(const T* x, const T* __restrict__ bias, const float* __restrict__ w, T* out,
              int64_t rows, int64_t F)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t gpr = F / 8;
    const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t cg = t % gpr, dr = S / gpr;
    int64_t r = t / gpr;
    float ba[8], bb[8];
    bias8(bias, cg * 8, ba);
    bias8(bias, F + cg * 8, bb);
    // warp k (< kUnroll) prefetches the block's column units of the k-th row
    // of the next iteration, both halves (a block that wraps a row fetches a
    // little of the neighbouring half: in bounds, unused)
    const int wk = threadIdx.x >> 5;
    const bool pf_warp = wk < kUnrollFwd;
    const int64_t pf_rows = (int64_t)(kUnrollFwd + wk) * dr;
    const int64_t pf_c0 = cg - (int64_t)threadIdx.x < 0 ? 0 : cg - (int64_t)threadIdx.x;

    for (; r + (kUnrollFwd - 1) * dr < rows; r += kUnrollFwd * dr) {
        {
            const int64_t rn = r + pf_rows;
            const bool on = pf_warp && rn < rows;
            const T* xn = x + (on ? rn : 0) * 2 * F;
            prefetch_block_span<MFX_PREFETCH_GLU_FWD != 0>(xn, pf_c0, 2 * gpr, 8 * sizeof(T), on);
            prefetch_block_span<MFX_PREFETCH_GLU_FWD != 0>(xn + F, pf_c0, gpr, 8 * sizeof(T), on);
        }
        Raw8<T> ra[kUnrollFwd], rb[kUnrollFwd];
        float wk[kUnrollFwd];
#pragma unroll
        for (int k = 0; k < kUnrollFwd; ++k) {
            const T* xr = x + (r + k * dr) * 2 * F + cg * 8;
            ld8(xr, ra[k]);
            ld8(xr + F, rb[k]);
            wk[k] = WEIGHTED ? w[r + k * dr] : 1.0f;
        }
#pragma unroll
        for (int k = 0; k < kUnrollFwd; ++k) {
            float fa[8], fb[8];
            widen8(ra[k], fa);
            widen8(rb[k], fb);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                fa[j] = glu_fwd1<KIND, kPrecise, WEIGHTED>(fa[j] + ba[j], fb[j] + bb[j], wk[k]);
            narrow8(fa, ra[k]);
            st8(out + (r + k * dr) * F + cg * 8, ra[k]);
        }
    }
    for (; r < rows; r += dr) {
        Raw8<T> ra, rb;
        const T* xr = x + r * 2 * F + cg * 8;
        ld8(xr, ra);
        ld8(xr + F, rb);
        const float wr = WEIGHTED ? w[r] : 1.0f;
        float fa[8], fb[8];
        widen8(ra, fa);
        widen8(rb, fb);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            fa[j] = glu_fwd1<KIND, kPrecise, WEIGHTED>(fa[j] + ba[j], fb[j] + bb[j], wr);
        narrow8(fa, ra);
        st8(out + r * F + cg * 8, ra);
    }
}

// Fixed-column backward (no weight), same ownership as the forward.
template <typename T, int KIND>
__global__ void __launch_bounds__(kThreads, MFX_MINB_GLU)
glu_bwd_fixed(const T* g, const T* x, const T* __restrict__ bias, T* dx, int64_t rows, int64_t F)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t gpr = F / 8;
    const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t cg = t % gpr, dr = S / gpr;
    int64_t r = t / gpr;
    float ba[8], bb[8];
    bias8(bias, cg * 8, ba);
    bias8(bias, F + cg * 8, bb);
    const int wk = threadIdx.x >> 5;
    const bool pf_warp = wk < kUnrollBwd;
    const int64_t pf_rows = (int64_t)(kUnrollBwd + wk) * dr;
    const int64_t pf_c0 = cg - (int64_t)threadIdx.x < 0 ? 0 : cg - (int64_t)threadIdx.x;

    for (; r < rows;) {
        const int nk = r + (kUnrollBwd - 1) * dr < rows ? kUnrollBwd : 1;
        {
            const int64_t rn = r + pf_rows;
            const bool on = pf_warp && rn < rows;
            const int64_t rc = on ? rn : 0;
            prefetch_block_span<MFX_PREFETCH_GLU_BWD != 0>(g + rc * F, pf_c0, gpr, 8 * sizeof(T), on);
            prefetch_block_span<MFX_PREFETCH_GLU_BWD != 0>(x + rc * 2 * F, pf_c0, 2 * gpr, 8 * sizeof(T), on);
            prefetch_block_span<MFX_PREFETCH_GLU_BWD != 0>(x + rc * 2 * F + F, pf_c0, gpr, 8 * sizeof(T), on);
        }
        Raw8<T> rg[kUnrollBwd], ra[kUnrollBwd], rb[kUnrollBwd];
#pragma unroll
        for (int k = 0; k < kUnrollBwd; ++k) {
            if (k < nk) {
                const T* xr = x + (r + k * dr) * 2 * F + cg * 8;
                ld8(g + (r + k * dr) * F + cg * 8, rg[k]);
                ld8(xr, ra[k]);
                ld8(xr + F, rb[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kUnrollBwd; ++k) {
            if (k < nk) {
                float fg[8], fa[8], fb[8];
                widen8(rg[k], fg);
                widen8(ra[k], fa);
                widen8(rb[k], fb);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float da, db;
                    glu_bwd1<KIND, kPrecise, false>(fa[j] + ba[j], fb[j] + bb[j], fg[j], 1.0f, &da, &db);
                    fa[j] = da;
                    fb[j] = db;
                }
                narrow8(fa, ra[k]);
                narrow8(fb, rb[k]);
                T* dr_ = dx + (r + k * dr) * 2 * F + cg * 8;
                st8(dr_, ra[k]);
                st8(dr_ + F, rb[k]);
            }
        }
        r += nk * dr;
    }
}

// ---------------------------------------------------------------------------
// Pipelined fixed-column forward and (unweighted) backward.  The flat unit
// f in [0, rows * gpr) is (row f / gpr, column unit f % gpr); thread t of
// block b takes f = b*256 + t + it*S with S a multiple of gpr, so its column
// unit (and bias) is fixed and its row advances by S / gpr.  Per iteration
// the producer warp copies the block's 256 flat units of each input stream
// (the activated half a, the linear half b and, backward, g) into one ring
// stage; a span that crosses a row end is copied in per-row pieces, laid out
// back to back, so consumer t always finds its unit at byte t * 8 * s.
// ---------------------------------------------------------------------------
// Spans per stage: measured per op (the GEGLU backward, the heaviest in
// arithmetic, gains from two; the others are fastest with one).
template <typename T, int KIND, bool BWD>
struct GluPipe {
    static constexpr int kStreams = BWD ? 3 : 2;
    static constexpr int kU = !BWD ? MFX_UNROLL_GLU_PIPE : KIND == GEGLU ? MFX_UNROLL_GEGLU_BWD_PIPE
                                                                        : MFX_UNROLL_SWIGLU_BWD_PIPE;
    static constexpr uint32_t kUnitBytes = 8 * sizeof(T);
    static constexpr uint32_t kSpan = kU * kConsumers * kUnitBytes;  // one stream's part of a stage
    static constexpr uint32_t kStage = kStreams * kSpan;
    static constexpr bool kSwigluBwd = KIND == SWIGLU && BWD;
    static constexpr int kKUnroll = kSwigluBwd             ? MFX_SWIGLU_BWD_K_UNROLL
                                    : (BWD && KIND == GEGLU) ? MFX_GEGLU_BWD_K_UNROLL
                                                             : kU;  // copies of the unit code
    static constexpr int kStages =
        ring_stages((kSwigluBwd ? MFX_RING_KB_SWIGLU_BWD
                     : BWD        ? MFX_RING_KB_GEGLU_BWD
                     : KIND == SWIGLU ? MFX_RING_KB_SWIGLU_FWD
                                      : MFX_RING_KB_GLU_FWD) * 1024,
                    kStage);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kStage;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

// With DB (backward only), each consumer also adds the da and db values it
// stores into partial column sums, written to ws[lane][0:2F] at its columns,
// lane = first flat unit / (F/8).
template <typename T, int KIND, bool WEIGHTED, bool BWD, bool DB = false>
__global__ void __launch_bounds__(kPipeThreads,
                                  KIND == SWIGLU && BWD ? MFX_PIPE_MINB_SWIGLU_BWD : MFX_PIPE_MINB_GLU)
glu_pipe(const T* g, const T* x, const T* __restrict__ bias, const float* __restrict__ w, T* out,
         int64_t rows, int64_t F, float* __restrict__ ws = nullptr)
{
    using P = GluPipe<T, KIND, BWD>;
    constexpr int NS = P::kStages, U = P::kU;
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int64_t gpr = F / 8, units = rows * gpr;
    const int64_t S = (int64_t)gridDim.x * kConsumers;
    const int64_t fb = (int64_t)blockIdx.x * kConsumers;
    // stage `it` holds the block's spans it*U .. it*U + U - 1: span k covers
    // flat units [fb + k S, + 256), one per consumer, all in the consumer's column
    const int64_t iters = units > fb ? (units - fb + U * S - 1) / (U * S) : 0;
    // stream order inside a stage: a, b, then g
    constexpr uint32_t kA = 0, kB = P::kSpan, kG = 2 * P::kSpan;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) != 0)
            return;
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
            uint32_t total = 0;
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int64_t f = fb + (it * U + k) * S;
                const int64_t left = units - f < kConsumers ? units - f : kConsumers;
                total += left > 0 ? (uint32_t)left * P::kUnitBytes * P::kStreams : 0u;
            }
            mbar_arrive_expect_tx(ring.full(s), total);
            const uint32_t st = smem_addr(data + (size_t)s * P::kStage);
#pragma unroll
            for (int k = 0; k < U; ++k) {
                // (the division per span measured faster than advancing the
                // span's row incrementally, 0.97 against 0.86 of the copy
                // peak for the plain GLU kernels; the cause is not known)
                const int64_t f = fb + (it * U + k) * S;
                int64_t left = units - f < kConsumers ? units - f : kConsumers;
                int64_t r = f / gpr, c = f - r * gpr;
                uint32_t off = (uint32_t)k * kConsumers * P::kUnitBytes;
                while (left > 0) {
                    const int64_t len = left < gpr - c ? left : gpr - c;
                    const uint32_t bytes = (uint32_t)len * P::kUnitBytes;
                    const T* xa = x + r * 2 * F + c * 8;
                    bulk_g2s(st + kA + off, xa, bytes, ring.full(s));
                    bulk_g2s(st + kB + off, xa + F, bytes, ring.full(s));
                    if (BWD)
                        bulk_g2s(st + kG + off, g + r * F + c * 8, bytes, ring.full(s));
                    left -= len;
                    off += bytes;
                    ++r;
                    c = 0;
                }
            }
        }
        return;
    }

    const int t = threadIdx.x;
    const int64_t ft = fb + t;
    const int64_t row0 = ft / gpr, cg = ft - row0 * gpr, drow = S / gpr;
    float ba[8], bb[8], acc_a[8], acc_b[8];
    bias8(bias, cg * 8, ba);
    bias8(bias, F + cg * 8, bb);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc_a[j] = acc_b[j] = 0.0f;
    // output row pointer (and weight) advancing drow rows per span
    const int64_t ow = BWD ? 2 * F : F;  // output row width
    T* po = out + row0 * ow + cg * 8;
    const int64_t pstep = drow * ow;
    for (int64_t it = 0; it < iters; ++it) {
        const int s = (int)(it % NS);
        if (!mbar_wait(ring.full(s), (uint32_t)((it / NS) & 1))) {
            atomicOr(&g_device_error, 1u);
            return;
        }
#pragma unroll(DB ? U : P::kKUnroll)  // (the fused bias gradient measured faster unrolled)
        for (int k = 0; k < U; ++k) {
            if (ft + (it * U + k) * S < units) {
                const int64_t row = row0 + (it * U + k) * drow;
                // (measured per kernel: the advanced pointer is faster for the
                // SwiGLU forwards, the recomputed one for the other three)
                T* const dst = (MFX_GLU_PTR_INC && KIND == SWIGLU && !BWD) ? po + k * pstep
                                                                          : out + row * ow + cg * 8;
                const unsigned char* st =
                    data + (size_t)s * P::kStage + ((uint32_t)k * kConsumers + t) * P::kUnitBytes;
                Raw8<T> ra, rb, rg;
                const uint4* pa = reinterpret_cast<const uint4*>(st + kA);
                const uint4* pb = reinterpret_cast<const uint4*>(st + kB);
                const uint4* pg = reinterpret_cast<const uint4*>(st + kG);
                if constexpr (DTypeInfo<T>::kBf16) {
                    ra.v = pa[0];
                    rb.v = pb[0];
                    if (BWD)
                        rg.v = pg[0];
                } else {
                    ra.v[0] = pa[0], ra.v[1] = pa[1];
                    rb.v[0] = pb[0], rb.v[1] = pb[1];
                    if (BWD)
                        rg.v[0] = pg[0], rg.v[1] = pg[1];
                }
                float fa[8], fb8[8];
                widen8(ra, fa);
                widen8(rb, fb8);
                if (!BWD) {
                    const float wr = WEIGHTED ? w[row] : 1.0f;
    #pragma unroll
                    for (int j = 0; j < 8; ++j)
                        fa[j] = glu_fwd1<KIND, kPrecise, WEIGHTED>(fa[j] + ba[j], fb8[j] + bb[j], wr);
                    narrow8(fa, ra);
                    st8(dst, ra);
                } else {
                    float fg[8];
                    widen8(rg, fg);
    #pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float da, db;
                        glu_bwd1<KIND, kPrecise, false>(fa[j] + ba[j], fb8[j] + bb[j], fg[j], 1.0f, &da, &db);
                        fa[j] = da;
                        fb8[j] = db;
                    }
                    narrow8(fa, ra);
                    narrow8(fb8, rb);
                    st8(dst, ra);
                    st8(dst + F, rb);
                    if (DB) {
                        widen8(ra, fa);  // the stored values
                        widen8(rb, fb8);
    #pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            acc_a[j] += fa[j];
                            acc_b[j] += fb8[j];
                        }
                    }
                }
            }
        }
        __syncwarp();
        if ((t & 31) == 0)
            mbar_arrive(ring.empty(s));
        po += U * pstep;
    }
    if (DB) {
        pdl_launch_dependents();
        float4* wa = reinterpret_cast<float4*>(ws + row0 * 2 * F + cg * 8);
        float4* wb = reinterpret_cast<float4*>(ws + row0 * 2 * F + F + cg * 8);
        wa[0] = make_float4(acc_a[0], acc_a[1], acc_a[2], acc_a[3]);
        wa[1] = make_float4(acc_a[4], acc_a[5], acc_a[6], acc_a[7]);
        wb[0] = make_float4(acc_b[0], acc_b[1], acc_b[2], acc_b[3]);
        wb[1] = make_float4(acc_b[4], acc_b[5], acc_b[6], acc_b[7]);
    }
}

// ---------------------------------------------------------------------------
// Generic forward/backward: any F and alignment.  Unit u is up to 8 output
// columns of one row: row u div gpr, columns [8 (u mod gpr), +8) with
// gpr = ceil(F / 8); (row, column-unit) advance incrementally by S.  `vec`
// (all pointers aligned and F % 8 == 0) selects 16-byte accesses.
// ---------------------------------------------------------------------------
template <typename T, int KIND, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads)
glu_fwd_generic(const T* x, const T* __restrict__ bias, const float* __restrict__ w, T* out,
                int64_t rows, int64_t F, int64_t gpr, int64_t dcg, int64_t drow, bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t units = rows * gpr;
    int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    int64_t r = u / gpr, cg = u % gpr;
    for (; u < units; u += S) {
        const int64_t c0 = cg * 8;
        const int cnt = F - c0 < 8 ? (int)(F - c0) : 8;
        const T* xr = x + r * 2 * F + c0;
        float fa[8], fb[8];
        load8f(xr, vec, cnt, fa);
        load8f(xr + F, vec, cnt, fb);
        const float wr = WEIGHTED ? w[r] : 1.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < cnt)
                fa[j] = glu_fwd1<KIND, kPrecise, WEIGHTED>(fa[j] + bias1(bias, c0 + j),
                                                           fb[j] + bias1(bias, F + c0 + j), wr);
        store8f(out + r * F + c0, vec, cnt, fa);
        cg += dcg;
        r += drow;
        if (cg >= gpr) {
            cg -= gpr;
            ++r;
        }
    }
}

template <typename T, int KIND>
__global__ void __launch_bounds__(kThreads)
glu_bwd_generic(const T* g, const T* x, const T* __restrict__ bias, T* dx, int64_t rows, int64_t F,
                int64_t gpr, int64_t dcg, int64_t drow, bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t units = rows * gpr;
    int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    int64_t r = u / gpr, cg = u % gpr;
    for (; u < units; u += S) {
        const int64_t c0 = cg * 8;
        const int cnt = F - c0 < 8 ? (int)(F - c0) : 8;
        const T* xr = x + r * 2 * F + c0;
        float fg[8], fa[8], fb[8];
        load8f(g + r * F + c0, vec, cnt, fg);
        load8f(xr, vec, cnt, fa);
        load8f(xr + F, vec, cnt, fb);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < cnt) {
                float da, db;
                glu_bwd1<KIND, kPrecise, false>(fa[j] + bias1(bias, c0 + j),
                                                fb[j] + bias1(bias, F + c0 + j), fg[j], 1.0f, &da, &db);
                fa[j] = da;
                fb[j] = db;
            }
        }
        T* dxr = dx + r * 2 * F + c0;
        store8f(dxr, vec, cnt, fa);
        store8f(dxr + F, vec, cnt, fb);
        cg += dcg;
        r += drow;
        if (cg >= gpr) {
            cg -= gpr;
            ++r;
        }
    }
}

// ---------------------------------------------------------------------------
// Any F and any alignment (the fixed forms above need F % 8 == 0 and aligned
// pointers).  Units are 8 consecutive elements of the flat [rows, F] grid of
// the forward output (backward: of g), starting at its first 16-byte aligned
// element (`head` elements before it, `tail` after the last unit, are done
// one by one by thread 0 of block 0), so those accesses stay aligned.  The
// unit stride S is a multiple of F / gcd(F, 8): each thread keeps one column
// phase, its bias in registers, the same input alignments and the same
// row-straddling case for its whole run.  The a and b runs (and the
// backward's outputs) sit at any alignment: loads take the aligned vectors
// around them (ld8_any), stores are assembled across the warp
// (st8_any_warp); a unit that straddles two rows goes element by element.
// The unit code is the other forms', so all forms give the same bits.
// ---------------------------------------------------------------------------

// Element k of a unit's raw storage.
template <typename T>
__device__ __forceinline__ uint32_t raw_elem(const Raw8<T>& r, int k)
{
    if constexpr (DTypeInfo<T>::kBf16) {
        const uint32_t w = k < 2 ? r.v.x : k < 4 ? r.v.y : k < 6 ? r.v.z : r.v.w;
        return (k & 1) ? w >> 16 : w & 0xFFFFu;
    } else {
        const uint4 v = r.v[k >> 2];
        const int i = k & 3;
        return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
    }
}
template <typename T>
__device__ __forceinline__ void store_raw(T* p, uint32_t bits)
{
    if constexpr (DTypeInfo<T>::kBf16)
        reinterpret_cast<bf16*>(p)->bits = (uint16_t)bits;
    else
        *reinterpret_cast<uint32_t*>(p) = bits;
}

// Each lane's run of 8 elements at p (`own`: the lane has a run).  A lane
// writes the aligned vectors that start inside its run; the first of them
// is combined with the previous lane's tail (through a shuffle) when that
// lane's run ends where this one starts, else the lane writes its leading
// part element by element; its trailing part (inside the vector the next
// run starts) goes element by element unless the next lane's run follows
// on.  All 32 lanes must call.
template <typename T>
__device__ __forceinline__ void st8_any_warp(T* p, const Raw8<T>& r, bool own)
{
    constexpr int NW = 2 * (int)sizeof(T);  // words per run
    constexpr uint32_t NB = 4u * NW;        // bytes per run
    uint32_t o[NW];
    if constexpr (DTypeInfo<T>::kBf16) {
        o[0] = r.v.x, o[1] = r.v.y, o[2] = r.v.z, o[3] = r.v.w;
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
            o[4 * h] = r.v[h].x, o[4 * h + 1] = r.v[h].y, o[4 * h + 2] = r.v[h].z, o[4 * h + 3] = r.v[h].w;
    }
    const int lane = threadIdx.x & 31;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uintptr_t ap = __shfl_up_sync(0xFFFFFFFFu, own ? a : 0, 1);
    const uintptr_t an = __shfl_down_sync(0xFFFFFFFFu, own ? a : 0, 1);
    const bool prev_ok = lane > 0 && ap != 0 && ap + NB == a;
    const bool next_ok = lane < 31 && an != 0 && a + NB == an;
    uint32_t po[2 * NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        po[i] = __shfl_up_sync(0xFFFFFFFFu, o[i], 1);
        po[NW + i] = o[i];
    }
    if (!own)
        return;
    const uint32_t phi = (uint32_t)(a & 15u);
    if (phi == 0) {
        st8(p, r);
        return;
    }
    char* v0 = reinterpret_cast<char*>(a - phi);
#pragma unroll
    for (int k = 0; k < (int)(NB / 16); ++k)
        if (k > 0 || prev_ok)
            st16(v0 + 16 * k, extract16(po, NB - phi + 16u * k));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t b = (uint32_t)j * sizeof(T);
        if ((!prev_ok && b < 16u - phi) || (!next_ok && b >= NB - phi))
            store_raw(p + j, raw_elem(r, j));
    }
}

// A run of 8 elements at p (a multiple of the element size) written with
// the widest stores its alignment allows: 16-byte vectors, 8-byte pairs,
// 4-byte words, or (bf16 at 2 mod 4) a half-word, three realigned words and
// a half-word.  Neighbouring runs fill each other's sectors; L2 merges them.
template <typename T>
__device__ __forceinline__ void st8_words(T* p, const Raw8<T>& r)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    uint32_t w[2 * sizeof(T)];
    if constexpr (DTypeInfo<T>::kBf16) {
        w[0] = r.v.x, w[1] = r.v.y, w[2] = r.v.z, w[3] = r.v.w;
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
            w[4 * h] = r.v[h].x, w[4 * h + 1] = r.v[h].y, w[4 * h + 2] = r.v[h].z, w[4 * h + 3] = r.v[h].w;
    }
    constexpr int NW = 2 * (int)sizeof(T);
    if ((a & 15u) == 0) {
        st8(p, r);
    } else if ((a & 7u) == 0) {
#pragma unroll
        for (int i = 0; i < NW; i += 2)
            st8(reinterpret_cast<char*>(p) + 4 * i, make_uint2(w[i], w[i + 1]));
    } else if ((a & 3u) == 0) {
#pragma unroll
        for (int i = 0; i < NW; ++i)
            asm volatile(MFX_ST_OP ".u32 [%0], %1;" ::"l"(reinterpret_cast<char*>(p) + 4 * i), "r"(w[i]) : "memory");
    } else if constexpr (DTypeInfo<T>::kBf16) {
        char* q = reinterpret_cast<char*>(p);
        asm volatile(MFX_ST_OP ".u16 [%0], %1;" ::"l"(q), "h"((unsigned short)(w[0] & 0xFFFFu)) : "memory");
#pragma unroll
        for (int i = 0; i < 3; ++i)
            asm volatile(MFX_ST_OP ".u32 [%0], %1;" ::"l"(q + 2 + 4 * i), "r"(__byte_perm(w[i], w[i + 1], 0x5432))
                         : "memory");
        asm volatile(MFX_ST_OP ".u16 [%0], %1;" ::"l"(q + 14), "h"((unsigned short)(w[3] >> 16)) : "memory");
    }
}

template <typename T, int KIND, bool WEIGHTED, bool BWD>
__device__ __forceinline__ void glu_elem(const T* g, const T* x, const T* __restrict__ bias,
                                         const float* __restrict__ w, T* out, int64_t F, int64_t e)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int64_t r = e / F, c = e % F;
    const float a = load1(x + r * 2 * F + c) + bias1(bias, c);
    const float b = load1(x + r * 2 * F + F + c) + bias1(bias, F + c);
    const float wr = WEIGHTED ? w[r] : 1.0f;
    if (BWD) {
        float da, db;
        glu_bwd1<KIND, kPrecise, WEIGHTED>(a, b, load1(g + e), wr, &da, &db);
        store1(out + r * 2 * F + c, da);
        store1(out + r * 2 * F + F + c, db);
    } else {
        store1(out + e, glu_fwd1<KIND, kPrecise, WEIGHTED>(a, b, wr));
    }
}

template <typename T, int KIND, bool WEIGHTED, bool BWD>
__global__ void __launch_bounds__(kThreads)
glu_realign(const T* g, const T* x, const T* __restrict__ bias, const float* __restrict__ w, T* out,
            int64_t rows, int64_t F, int64_t units, int64_t S, int head, int tail, uintptr_t x_lo, uintptr_t x_hi)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    constexpr int U = MFX_UNROLL_GLU_ANY;
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const bool on = gt < S;
    const int64_t e0 = head + 8 * gt;                 // this thread's first unit's first element
    const int64_t r0 = e0 / F, c0 = e0 % F;
    const bool straddle = c0 + 8 > F;
    const int64_t dr = 8 * S / F;                     // rows between this thread's units
    float ba[8], bb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t c = c0 + j < F ? c0 + j : c0 + j - F;
        ba[j] = bias1(bias, c);
        bb[j] = bias1(bias, F + c);
    }
    const int64_t nj = on && gt < units ? (units - gt + S - 1) / S : 0;
    const int64_t nw = __shfl_sync(0xFFFFFFFFu, nj, 0);  // lane 0 has the most units of its warp
    for (int64_t j0 = 0; j0 < nw; j0 += U) {
        Raw8<T> ra[U], rb[U], rg[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t j = j0 + k;
            if (j < nj && !straddle) {
                const T* pa = x + (r0 + j * dr) * 2 * F + c0;
                if (in_vectors(pa, x_lo, x_hi) && in_vectors(pa + F, x_lo, x_hi)) {
                    ld8_any(pa, ra[k]);
                    ld8_any(pa + F, rb[k]);
                } else {  // a run at either end of x: element by element (exact round trip)
                    float fa[8], fb[8];
                    load8f(pa, false, 8, fa);
                    load8f(pa + F, false, 8, fb);
                    narrow8(fa, ra[k]);
                    narrow8(fb, rb[k]);
                }
                if (BWD)
                    ld8(g + e0 + 8 * j * S, rg[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t j = j0 + k;
            const bool act = j < nj;
            const int64_t e = e0 + 8 * j * S;
            const int64_t r = r0 + j * dr;
            const bool mine = act && !straddle;  // a straddling unit waits for the last pass
            float fa[8], fb[8], fg[8];
            Raw8<T> oa, ob;
            if (mine) {
                widen8(ra[k], fa);
                widen8(rb[k], fb);
                if (BWD)
                    widen8(rg[k], fg);
                const float wr = WEIGHTED ? w[r] : 1.0f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (BWD) {
                        glu_bwd1<KIND, kPrecise, WEIGHTED>(fa[q] + ba[q], fb[q] + bb[q], fg[q], wr, &fa[q], &fb[q]);
                    } else {
                        fa[q] = glu_fwd1<KIND, kPrecise, WEIGHTED>(fa[q] + ba[q], fb[q] + bb[q], wr);
                    }
                }
                narrow8(fa, oa);
                if (BWD)
                    narrow8(fb, ob);
            }
            if (!BWD) {
                if (mine)
                    st8(out + e, oa);
            } else {
                T* pa = out + r * 2 * F + c0;
                st8_any_warp(pa, oa, mine);
                st8_any_warp(pa + F, ob, mine);
            }
        }
    }
    // the units that straddle a row boundary (row r's end inside one unit),
    // spread over every thread of the grid, element by element
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    for (int64_t rb = (int64_t)blockIdx.x * kThreads + threadIdx.x; rb + 1 < rows; rb += nthreads) {
        const int64_t eb = (rb + 1) * F - head;  // the boundary, counted from the first unit
        if (eb % 8 != 0 && eb / 8 < units) {
            const int64_t eu = head + (eb / 8) * 8;
            for (int q = 0; q < 8; ++q)
                glu_elem<T, KIND, WEIGHTED, BWD>(g, x, bias, w, out, F, eu + q);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int q = 0; q < head; ++q)
            glu_elem<T, KIND, WEIGHTED, BWD>(g, x, bias, w, out, F, q);
        for (int q = 0; q < tail; ++q)
            glu_elem<T, KIND, WEIGHTED, BWD>(g, x, bias, w, out, F, head + 8 * units + q);
    }
}

// ---------------------------------------------------------------------------
// The same any-width, any-alignment GLU through the bulk-copy ring (F >=
// 2048, so a block's 256-unit span of the output grid meets at most two
// rows).  Per span the producer copies, for each row the span meets, the a
// piece and the b piece (the columns the span's units need) as the aligned
// vectors covering them, clipped to the vectors inside x, into fixed-size
// piece images, the g span (backward; aligned like the units), and a header
// with the span's first row and column.  A consumer keeps its column phase
// and row stride (as in glu_realign), finds its run in its row's piece
// image at the byte distance from the piece's first aligned vector, and
// reads it with aligned shared loads; runs whose vectors were clipped (at
// either end of x) go element by element from global memory, straddling
// units and the head and tail as in glu_realign.
// ---------------------------------------------------------------------------
template <typename T, bool BWD>
struct GluRPipe {
    static constexpr uint32_t kCap = kConsumers * 8 * (uint32_t)sizeof(T) + 32;  // a piece image
    static constexpr uint32_t kG = BWD ? kConsumers * 8 * (uint32_t)sizeof(T) : 0;
    static constexpr uint32_t kSpan = 16 + 4 * kCap + kG;  // header, a0, a1, b0, b1 (, g)
    static constexpr int kStages =
        ring_stages((!DTypeInfo<T>::kBf16 ? MFX_RING_KB_GLU_RPIPE
                     : BWD ? MFX_RING_KB_GLU_RPIPE_BWD16 : MFX_RING_KB_GLU_RPIPE_FWD16) * 1024, kSpan);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kSpan;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

// The 8 elements at byte offset off (a multiple of the element size) of a
// piece image, as 4-byte shared loads: plain words when off is a multiple
// of 4, else (bf16 at 2 mod 4) five words and a fixed half-word permute.
template <typename T>
__device__ __forceinline__ void img_ld8(const unsigned char* img, uint32_t off, Raw8<T>& r)
{
    const uint32_t* p = reinterpret_cast<const uint32_t*>(img + (off & ~3u));
    if constexpr (DTypeInfo<T>::kBf16) {
        if (off & 2u) {
            const uint32_t w0 = p[0], w1 = p[1], w2 = p[2], w3 = p[3], w4 = p[4];
            r.v = make_uint4(__byte_perm(w0, w1, 0x5432), __byte_perm(w1, w2, 0x5432), __byte_perm(w2, w3, 0x5432),
                             __byte_perm(w3, w4, 0x5432));
        } else {
            r.v = make_uint4(p[0], p[1], p[2], p[3]);
        }
    } else {
        r.v[0] = make_uint4(p[0], p[1], p[2], p[3]);
        r.v[1] = make_uint4(p[4], p[5], p[6], p[7]);
    }
}

template <typename T, int KIND, bool WEIGHTED, bool BWD>
__global__ void __launch_bounds__(kPipeThreads, !DTypeInfo<T>::kBf16 ? MFX_PIPE_MINB_GLU_RPIPE
                                                : BWD ? MFX_PIPE_MINB_GLU_RPIPE_BWD16 : MFX_PIPE_MINB_GLU_RPIPE_FWD16)
glu_rpipe(const T* g, const T* x, const T* __restrict__ bias, const float* __restrict__ w, T* out, int64_t rows,
          int64_t F, int64_t units, int64_t S, int head, int tail, uintptr_t x_lo, uintptr_t x_hi)
{
    using P = GluRPipe<T, BWD>;
    constexpr int NS = P::kStages;
    constexpr int ES = (int)sizeof(T);
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int64_t ub0 = (int64_t)blockIdx.x * kConsumers;
    const int64_t iters = units > ub0 ? (units - ub0 + S - 1) / S : 0;
    const int64_t active = S - ub0 < kConsumers ? S - ub0 : kConsumers;
    const uintptr_t xlo16 = (x_lo + 15) & ~(uintptr_t)15, xhi16 = x_hi & ~(uintptr_t)15;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) != 0)
            return;
        // spans advance 8 S = (8 S / F) F elements: the first row by dr, the
        // first column never (no division per span)
        const int64_t dr = 8 * S / F;
        const int64_t E00 = head + 8 * ub0;
        const int64_t r_a0 = E00 / F, c_a = E00 - r_a0 * F;
        for (int64_t it = 0; it < iters; ++it) {
            const int st = (int)(it % NS);
            const int64_t n = it / NS;
            if (n > 0 && !mbar_wait(ring.empty(st), (uint32_t)((n - 1) & 1))) {
                atomicOr(&g_device_error, 2u);
                for (int64_t j = it - 1; j >= 0 && j > it - NS; --j)
                    if (!mbar_wait(ring.full((int)(j % NS)), (uint32_t)((j / NS) & 1)))
                        atomicOr(&g_device_error, 4u);
                return;
            }
            unsigned char* sp = data + (size_t)st * P::kSpan;
            const int64_t start = ub0 + it * S;
            const int64_t left = units - start;
            const int64_t cnt = left < active ? left : active;
            // pieces: a0, a1, b0, b1 (row r_a from column c_a, row r_a + 1
            // from column 0), each as its covering vectors inside x
            const int64_t E0 = head + 8 * start, len = 8 * cnt;
            const int64_t r_a = r_a0 + it * dr;
            const int64_t L0 = len < F - c_a ? len : F - c_a, L1 = len - L0;
            reinterpret_cast<int64_t*>(sp)[0] = r_a;
            reinterpret_cast<int64_t*>(sp)[1] = c_a;
            uintptr_t lo[4], hi[4];
            uint32_t total = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t row = r_a + (q & 1), c = (q & 1) ? 0 : c_a, L = (q & 1) ? L1 : L0;
                const uintptr_t s0 = reinterpret_cast<uintptr_t>(x + row * 2 * F + ((q >> 1) ? F : 0) + c);
                const uintptr_t b16 = s0 & ~(uintptr_t)15, e16 = (s0 + (uintptr_t)(L * ES) + 15) & ~(uintptr_t)15;
                lo[q] = b16 > xlo16 ? b16 : xlo16;
                hi[q] = e16 < xhi16 ? e16 : xhi16;
                if (L <= 0 || hi[q] <= lo[q])
                    hi[q] = lo[q] = b16;  // nothing to copy
                total += (uint32_t)(hi[q] - lo[q]);
            }
            if (BWD)
                total += (uint32_t)(cnt * 8 * ES);
            mbar_arrive_expect_tx(ring.full(st), total);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (hi[q] > lo[q]) {
                    const int64_t row = r_a + (q & 1), c = (q & 1) ? 0 : c_a;
                    const uintptr_t s0 = reinterpret_cast<uintptr_t>(x + row * 2 * F + ((q >> 1) ? F : 0) + c);
                    bulk_g2s(smem_addr(sp + 16 + q * P::kCap + (lo[q] - (s0 & ~(uintptr_t)15))),
                             reinterpret_cast<const void*>(lo[q]), (uint32_t)(hi[q] - lo[q]), ring.full(st));
                }
            }
            if (BWD)
                bulk_g2s(smem_addr(sp + 16 + 4 * P::kCap), g + E0, (uint32_t)(cnt * 8 * ES), ring.full(st));
        }
        return;
    }

    const int t = threadIdx.x;
    const int64_t gt = ub0 + t;
    const bool on = gt < S;
    const int64_t e0 = head + 8 * gt;
    const int64_t r0 = e0 / F, c0 = e0 % F;
    const bool straddle = c0 + 8 > F;
    const int64_t dr = 8 * S / F;  // rows advance 16 S ES bytes of x per span: the phases below hold
    // 16-byte phases of the a and b halves of this thread's rows at column 0
    const uint32_t pha = (uint32_t)((reinterpret_cast<uintptr_t>(x) + (uintptr_t)(r0 * 2 * F * ES)) & 15u);
    const uint32_t phb = (pha + (uint32_t)(F * ES)) & 15u;
    float ba[8], bb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t c = c0 + j < F ? c0 + j : c0 + j - F;
        ba[j] = bias1(bias, c);
        bb[j] = bias1(bias, F + c);
    }
    // per iteration the stage, the unit, the row and the row pointers
    // advance by counters (no 64-bit multiply or division in the loop); the
    // fp32 forward measured faster deriving them from the iteration
    // (0.75 against 0.69 of the copy peak; the others gain 2-9% with counters)
    constexpr bool kCnt = BWD || DTypeInfo<T>::kBf16;
    int sc = 0;
    uint32_t phc = 0;
    int64_t uc = gt, rc = r0;
    const int64_t xstep = dr * 2 * F;
    const T* pac = x + r0 * 2 * F + c0;
    T* poc = out + (BWD ? r0 * 2 * F + c0 : e0);
    const int64_t ostep = BWD ? xstep : 8 * S;
    for (int64_t it = 0; it < iters; ++it, uc += S, rc += dr, pac += xstep, poc += ostep) {
        const int s = kCnt ? sc : (int)(it % NS);
        const uint32_t ph = kCnt ? phc : (uint32_t)((it / NS) & 1);
        const int64_t u = kCnt ? uc : gt + it * S;
        const int64_t r = kCnt ? rc : r0 + it * dr;
        const T* pa = kCnt ? pac : x + r * 2 * F + c0;
        T* po = kCnt ? poc : out + (BWD ? r * 2 * F + c0 : e0 + 8 * it * S);
        if (!mbar_wait(ring.full(s), ph)) {
            atomicOr(&g_device_error, 1u);
            return;
        }
        const unsigned char* sp = data + (size_t)s * P::kSpan;
        // the span's first column: units of its first row sit at or after it,
        // units of the next row before it (a span covers less than a row)
        const uint32_t c_a = (uint32_t)reinterpret_cast<const int64_t*>(sp)[1];
        const bool mine = on && !straddle && u < units;
        Raw8<T> oa, ob;
        if (mine) {
            const int seg = (uint32_t)c0 >= c_a ? 0 : 1;
            const uint32_t cs = seg ? 0u : c_a;
            Raw8<T> ra, rb, rg;
            // only the first and last rows can meet the vectors clipped at
            // either end of x
            if ((r != 0 && r != rows - 1) || (in_vectors(pa, x_lo, x_hi) && in_vectors(pa + F, x_lo, x_hi))) {
                const uint32_t d = ((uint32_t)c0 - cs) * ES;
                img_ld8(sp + 16 + seg * P::kCap, ((pha + cs * ES) & 15u) + d, ra);
                img_ld8(sp + 16 + (2 + seg) * P::kCap, ((phb + cs * ES) & 15u) + d, rb);
            } else {
                float fa[8], fb[8];
                load8f(pa, false, 8, fa);
                load8f(pa + F, false, 8, fb);
                narrow8(fa, ra);
                narrow8(fb, rb);
            }
            float fa[8], fb[8], fg[8];
            widen8(ra, fa);
            widen8(rb, fb);
            if (BWD) {
                lds8(sp + 16 + 4 * P::kCap + t * 8 * ES, rg);
                widen8(rg, fg);
            }
            const float wr = WEIGHTED ? w[r] : 1.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (BWD)
                    glu_bwd1<KIND, kPrecise, WEIGHTED>(fa[q] + ba[q], fb[q] + bb[q], fg[q], wr, &fa[q], &fb[q]);
                else
                    fa[q] = glu_fwd1<KIND, kPrecise, WEIGHTED>(fa[q] + ba[q], fb[q] + bb[q], wr);
            }
            narrow8(fa, oa);
            if (BWD)
                narrow8(fb, ob);
        }
        __syncwarp();
        if ((t & 31) == 0)
            mbar_arrive(ring.empty(s));
        if (++sc == NS) {
            sc = 0;
            phc ^= 1u;
        }
        if (!BWD) {
            if (mine)
                st8(po, oa);
        } else if (MFX_GLU_RPIPE_WORD_ST && DTypeInfo<T>::kBf16) {
            if (mine) {
                st8_words(po, oa);
                st8_words(po + F, ob);
            }
        } else {
            st8_any_warp(po, oa, mine);
            st8_any_warp(po + F, ob, mine);
        }
    }
    // straddling units over every consumer thread, then head and tail
    const int64_t nthreads = (int64_t)gridDim.x * kConsumers;
    for (int64_t rb = gt; rb + 1 < rows; rb += nthreads) {
        const int64_t eb = (rb + 1) * F - head;
        if (eb % 8 != 0 && eb / 8 < units) {
            const int64_t eu = head + (eb / 8) * 8;
            for (int q = 0; q < 8; ++q)
                glu_elem<T, KIND, WEIGHTED, BWD>(g, x, bias, w, out, F, eu + q);
        }
    }
    if (blockIdx.x == 0 && t == 0) {
        for (int q = 0; q < head; ++q)
            glu_elem<T, KIND, WEIGHTED, BWD>(g, x, bias, w, out, F, q);
        for (int q = 0; q < tail; ++q)
            glu_elem<T, KIND, WEIGHTED, BWD>(g, x, bias, w, out, F, head + 8 * units + q);
    }
}

// ---------------------------------------------------------------------------
// Weighted SwiGLU backward.  The weight gradient is a sum over a whole row,
// so one block owns a row at a time: thread t takes column units t, t + 256,
// ... and accumulates its terms in column order; the block then adds the 256
// partial sums with a fixed xor-shuffle tree per warp and a fixed sequential
// pass over the 8 warp sums.  The order depends only on F, never on timing
// or grid size, so dweight is bitwise reproducible.
// ---------------------------------------------------------------------------
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads, VEC ? MFX_MINB_WBWD : MFX_MINB_WBWD_ANY)
swiglu_bwd_weighted(const T* g, const T* x, const T* __restrict__ bias, const float* __restrict__ w,
                    T* dx, float* __restrict__ dw, int64_t rows, int64_t F)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    // column units in flight per thread: packed vectors when aligned
    constexpr int U = VEC ? (kPrecise ? 2 : MFX_UNROLL_WBWD) : 1;
    __shared__ float warp_sums[2][kThreads / 32];
    const int64_t gpr = (F + 7) / 8;
    int parity = 0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, parity ^= 1) {
        if (VEC && MFX_PREFETCH_WBWD && r + gridDim.x < rows) {
            // the block's next row goes to L2: warp w takes column units
            // [256 (w + 8 i), +256) of each stream
            const int64_t rn = r + gridDim.x;
            const bool all = true;
            const int64_t lim = gpr * MFX_PREFETCH_WBWD_PART / 8;
            for (int64_t q = (int64_t)(threadIdx.x >> 5) * kThreads; q < lim; q += (int64_t)kThreads * 8) {
                prefetch_block_span<true>(g + rn * F, q, gpr, 8 * sizeof(T), all);
                prefetch_block_span<true>(x + rn * 2 * F, q, gpr, 8 * sizeof(T), all);
                prefetch_block_span<true>(x + rn * 2 * F + F, q, gpr, 8 * sizeof(T), all);
            }
        }
        const float wr = w[r];
        const T* gr = g + r * F;
        const T* xr = x + r * 2 * F;
        T* dxr = dx + r * 2 * F;
        float acc = 0.0f;
        if constexpr (!VEC) {
            // any width or alignment: the same units and order, the runs read
            // through aligned vectors (ld8_any) and written through the warp
            // (st8_any_warp); the loop runs while the warp's first lane has a
            // unit, so every lane reaches the warp-wide stores
            const uintptr_t g_lo = reinterpret_cast<uintptr_t>(g), x_lo = reinterpret_cast<uintptr_t>(x);
            const uintptr_t g_hi = g_lo + (uintptr_t)(rows * F * sizeof(T)), x_hi = x_lo + 2 * (g_hi - g_lo);
            const uintptr_t b_lo = reinterpret_cast<uintptr_t>(bias), b_hi = b_lo + (uintptr_t)(2 * F * sizeof(T));
            if (MFX_WBWD_ANY_PF && r + gridDim.x < rows) {
                // the block's next row to L2: the aligned vectors of its g
                // and x runs that lie inside the buffers, 4 KB per warp
                const int64_t rn = r + gridDim.x;
                const uintptr_t runs[2][2] = {
                    {reinterpret_cast<uintptr_t>(g + rn * F), reinterpret_cast<uintptr_t>(g + rn * F + F)},
                    {reinterpret_cast<uintptr_t>(x + rn * 2 * F), reinterpret_cast<uintptr_t>(x + rn * 2 * F + 2 * F)}};
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uintptr_t lo0 = (runs[q][0] + 15) & ~(uintptr_t)15, hi0 = runs[q][1] & ~(uintptr_t)15;
                    for (uintptr_t a = lo0 + (uintptr_t)(threadIdx.x >> 5) * 4096; a < hi0;
                         a += (uintptr_t)(kThreads / 32) * 4096)
                        prefetch_l2_if(reinterpret_cast<const void*>(a),
                                       (uint32_t)(hi0 - a < 4096 ? hi0 - a : 4096), (threadIdx.x & 31) == 0);
                }
            }
            // MFX_WBWD_ANY_U units of each lane in flight: loads first, then
            // the units in column order (the order of the sum stays t, t + 256, ...)
            constexpr int UA = MFX_WBWD_ANY_U;
            for (int64_t base = threadIdx.x & ~31; base < gpr; base += (int64_t)UA * kThreads) {
                Raw8<T> rg[UA], ra[UA], rb[UA];
                int cnt[UA];
                bool vec[UA];
#pragma unroll
                for (int u = 0; u < UA; ++u) {
                    const int64_t cg0 = base + (int64_t)u * kThreads + (threadIdx.x & 31);
                    const int64_t c0 = cg0 * 8;
                    cnt[u] = cg0 < gpr ? (F - c0 < 8 ? (int)(F - c0) : 8) : 0;
                    vec[u] = cnt[u] == 8 && in_vectors(gr + c0, g_lo, g_hi) && in_vectors(xr + c0, x_lo, x_hi) &&
                             in_vectors(xr + F + c0, x_lo, x_hi);
                    if (vec[u]) {
                        ld8_any(gr + c0, rg[u]);
                        ld8_any(xr + c0, ra[u]);
                        ld8_any(xr + F + c0, rb[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < UA; ++u) {
                    const int64_t c0 = (base + (int64_t)u * kThreads + (threadIdx.x & 31)) * 8;
                    const int n = cnt[u];
                    float fg[8], fa[8], fb[8], ba[8], bb[8];
                    if (vec[u]) {
                        widen8(rg[u], fg);
                        widen8(ra[u], fa);
                        widen8(rb[u], fb);
                    } else if (n > 0) {
                        load8f(gr + c0, false, n, fg);
                        load8f(xr + c0, false, n, fa);
                        load8f(xr + F + c0, false, n, fb);
                    }
                    if (MFX_WBWD_ANY_BIASVEC && bias && n == 8 && in_vectors(bias + c0, b_lo, b_hi) &&
                        in_vectors(bias + F + c0, b_lo, b_hi)) {
                        Raw8<T> r0, r1;
                        ld8_any(bias + c0, r0);
                        ld8_any(bias + F + c0, r1);
                        widen8(r0, ba);
                        widen8(r1, bb);
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            ba[j] = j < n ? bias1(bias, c0 + j) : 0.0f;
                            bb[j] = j < n ? bias1(bias, F + c0 + j) : 0.0f;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j < n) {
                            float da, db;
                            const float term = glu_bwd1<SWIGLU, kPrecise, true>(fa[j] + ba[j], fb[j] + bb[j],
                                                                                fg[j], wr, &da, &db);
                            acc += fg[j] * term;
                            fa[j] = da;
                            fb[j] = db;
                        }
                    }
                    Raw8<T> oa, ob;
                    narrow8(fa, oa);
                    narrow8(fb, ob);
                    if (MFX_WBWD_ANY_WORDST && DTypeInfo<T>::kBf16) {
                        if (n == 8) {
                            st8_words(dxr + c0, oa);
                            st8_words(dxr + F + c0, ob);
                        }
                    } else {
                        st8_any_warp(dxr + c0, oa, n == 8);
                        st8_any_warp(dxr + F + c0, ob, n == 8);
                    }
                    if (n > 0 && n < 8) {
                        store8f(dxr + c0, false, n, fa);
                        store8f(dxr + F + c0, false, n, fb);
                    }
                }
            }
        }
        for (int64_t cg0 = threadIdx.x; VEC && cg0 < gpr; cg0 += (int64_t)U * kThreads) {
            Raw8<T> rg[U], ra[U], rb[U];
            if (VEC) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c0 = (cg0 + (int64_t)u * kThreads) * 8;
                    if (c0 < F) {
                        ld8(gr + c0, rg[u]);
                        ld8(xr + c0, ra[u]);
                        ld8(xr + F + c0, rb[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c0 = (cg0 + (int64_t)u * kThreads) * 8;
                if (c0 >= F)
                    continue;
                const int cnt = F - c0 < 8 ? (int)(F - c0) : 8;
                float fg[8], fa[8], fb[8], ba[8], bb[8];
                if (VEC) {
                    widen8(rg[u], fg);
                    widen8(ra[u], fa);
                    widen8(rb[u], fb);
                    bias8(bias, c0, ba);
                    bias8(bias, F + c0, bb);
                } else {
                    load8f(gr + c0, false, cnt, fg);
                    load8f(xr + c0, false, cnt, fa);
                    load8f(xr + F + c0, false, cnt, fb);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        ba[j] = j < cnt ? bias1(bias, c0 + j) : 0.0f;
                        bb[j] = j < cnt ? bias1(bias, F + c0 + j) : 0.0f;
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j < cnt) {
                        float da, db;
                        const float term = glu_bwd1<SWIGLU, kPrecise, true>(fa[j] + ba[j], fb[j] + bb[j],
                                                                            fg[j], wr, &da, &db);
                        acc += fg[j] * term;
                        fa[j] = da;
                        fb[j] = db;
                    }
                }
                store8f(dxr + c0, VEC, cnt, fa);
                store8f(dxr + F + c0, VEC, cnt, fb);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if ((threadIdx.x & 31) == 0)
            warp_sums[parity][threadIdx.x >> 5] = acc;
        // One barrier per row: the buffer written here is next written two
        // rows later, after another barrier that thread 0 passes only once it
        // has read this one.
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

// ---------------------------------------------------------------------------
// Pipelined weighted SwiGLU backward.  Rows stay owned by blocks (block b
// takes rows b, b + grid, ...), so the weight gradient is still one
// fixed-order sum per block; the producer warp streams each row as chunks of
// 256 column units of g, a and b.  Consumer t takes column unit
// chunk * 256 + t, so it adds its terms in increasing column order exactly
// like swiglu_bwd_weighted (same bits), and the 256 consumers combine their
// sums at the row's last chunk behind a named barrier the producer does not
// join.
// ---------------------------------------------------------------------------
template <typename T>
struct WbwdPipe {
    static constexpr int kU = MFX_UNROLL_WBWD_PIPE;  // units per consumer per stage
    static constexpr uint32_t kUnitBytes = 8 * sizeof(T);
    static constexpr uint32_t kSpan = kU * kConsumers * kUnitBytes;
    static constexpr uint32_t kStage = 3 * kSpan;
    static constexpr int kStages = ring_stages(MFX_RING_KB_WBWD * 1024, kStage);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kStage;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

template <typename T>
__global__ void __launch_bounds__(kPipeThreads, MFX_PIPE_MINB_WBWD)
swiglu_bwd_weighted_pipe(const T* g, const T* x, const T* __restrict__ bias, const float* __restrict__ w,
                         T* dx, float* __restrict__ dw, int64_t rows, int64_t F)
{
    using P = WbwdPipe<T>;
    constexpr int NS = P::kStages, U = P::kU;
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float warp_sums[2][kConsumerWarps];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int64_t gpr = F / 8;
    const int64_t nchunk = (gpr + U * kConsumers - 1) / (U * kConsumers);
    const int64_t my_rows = rows > blockIdx.x ? (rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t iters = my_rows * nchunk;
    constexpr uint32_t kA = 0, kB = P::kSpan, kG = 2 * P::kSpan;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) != 0)
            return;
        // row r and chunk of iteration it advance incrementally (no division)
        int64_t r = blockIdx.x, chunk = 0;
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
            const uint32_t bytes = (uint32_t)cnt * P::kUnitBytes;
            mbar_arrive_expect_tx(ring.full(s), 3u * bytes);
            const uint32_t st = smem_addr(data + (size_t)s * P::kStage);
            const T* xa = x + r * 2 * F + c0 * 8;
            bulk_g2s(st + kA, xa, bytes, ring.full(s));
            bulk_g2s(st + kB, xa + F, bytes, ring.full(s));
            bulk_g2s(st + kG, g + r * F + c0 * 8, bytes, ring.full(s));
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
    // A consumer whose wait ran out stops waiting and computing but keeps
    // meeting the row-end barrier, so no other consumer is left behind it.
    bool dead = false;
    int64_t r = blockIdx.x, chunk = 0;
    int s = 0;        // stage of iteration it (it % NS)
    uint32_t ph = 0;  // its parity ((it / NS) & 1)
    for (int64_t it = 0; it < iters; ++it) {
        // the bias and the row weight do not come through the ring: load
        // them before waiting for the stage so their latency overlaps it
        float ba[U][8], bb[U][8];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t cg = chunk * U * kConsumers + k * kConsumers + t;
            const int64_t cgb = cg < gpr ? cg : 0;
            bias8(bias, cgb * 8, ba[k]);
            bias8(bias, F + cgb * 8, bb[k]);
        }
        const float wr = w[r];
        if (!dead && !mbar_wait(ring.full(s), ph)) {
            atomicOr(&g_device_error, 1u);
            dead = true;
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t cu = k * kConsumers + t;           // unit within the chunk
            const int64_t cg = chunk * U * kConsumers + cu;  // unit within the row
            if (!dead && cg < gpr) {
                const unsigned char* st = data + (size_t)s * P::kStage + cu * P::kUnitBytes;
                Raw8<T> ra, rb, rg;
                lds8(st + kA, ra);
                lds8(st + kB, rb);
                lds8(st + kG, rg);
                float fa[8], fb[8], fg[8];
                widen8(ra, fa);
                widen8(rb, fb);
                widen8(rg, fg);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float da, db;
                    const float term =
                        glu_bwd1<SWIGLU, kPrecise, true>(fa[j] + ba[k][j], fb[j] + bb[k][j], fg[j], wr, &da, &db);
                    acc += fg[j] * term;
                    fa[j] = da;
                    fb[j] = db;
                }
                narrow8(fa, ra);
                narrow8(fb, rb);
                T* dxr = dx + r * 2 * F + cg * 8;
                st8(dxr, ra);
                st8(dxr + F, rb);
            }
        }
        if (!dead) {
            __syncwarp();
            if ((t & 31) == 0)
                mbar_arrive(ring.empty(s));
        }
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
        if (chunk == nchunk - 1) {
            // the row is done: fixed xor-shuffle tree, then the 8 warp sums in order
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
            if ((t & 31) == 0)
                warp_sums[parity][t >> 5] = acc;
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
            if (t == 0) {
                float sum = 0.0f;
#pragma unroll
                for (int i = 0; i < kConsumerWarps; ++i)
                    sum += warp_sums[parity][i];
                dw[r] = sum;
            }
            acc = 0.0f;
            parity ^= 1;
            chunk = 0;
            r += gridDim.x;
        } else {
            ++chunk;
        }
    }
}

// The weighted SwiGLU backward pipeline for short rows (at most 256 units):
// a stage holds R = 512 / gpad whole rows, gpad = the row's units rounded up
// to a warp, row slot k on the stage's virtual threads [k gpad, (k+1) gpad)
// (virtual thread v = u * 256 + t: consumer t's unit u).  Every warp lies in
// one row, so a row's dweight is the same xor tree per warp and the same
// in-order sum over its warps as in swiglu_bwd_weighted_pipe (whose other
// warps add exact zeros): the same bits.
template <typename T>
__global__ void __launch_bounds__(kPipeThreads, MFX_PIPE_MINB_WBWD)
swiglu_bwd_weighted_pipe_rows(const T* g, const T* x, const T* __restrict__ bias, const float* __restrict__ w,
                              T* dx, float* __restrict__ dw, int64_t rows, int64_t F)
{
    using P = WbwdPipe<T>;
    constexpr int NS = P::kStages, U = P::kU;
    constexpr int kV = U * kConsumers;  // virtual threads of a stage
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float warp_sums[2][kV / 32];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int gpr = (int)(F / 8);
    const int gpad = (gpr + 31) & ~31;
    const int R = kV / gpad;
    const int64_t my_rows = rows > blockIdx.x ? (rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t iters = (my_rows + R - 1) / R;
    constexpr uint32_t kA = 0, kB = P::kSpan, kG = 2 * P::kSpan;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) != 0)
            return;
        const uint32_t bytes = (uint32_t)gpr * P::kUnitBytes;
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
            const int nr = my_rows - it * R < R ? (int)(my_rows - it * R) : R;
            mbar_arrive_expect_tx(ring.full(s), 3u * bytes * (uint32_t)nr);
            const uint32_t st = smem_addr(data + (size_t)s * P::kStage);
            for (int k = 0; k < nr; ++k) {
                const int64_t r = blockIdx.x + (it * R + k) * gridDim.x;
                const uint32_t off = (uint32_t)(k * gpad) * P::kUnitBytes;
                const T* xa = x + r * 2 * F;
                bulk_g2s(st + kA + off, xa, bytes, ring.full(s));
                bulk_g2s(st + kB + off, xa + F, bytes, ring.full(s));
                bulk_g2s(st + kG + off, g + r * F, bytes, ring.full(s));
            }
        }
        return;
    }

    const int t = threadIdx.x;
    // this consumer's row slot and unit for each u (fixed for the launch)
    int slot_of[U], cu_of[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int v = u * kConsumers + t;
        slot_of[u] = v / gpad;
        cu_of[u] = v - slot_of[u] * gpad;
    }
    int parity = 0;
    bool dead = false;
    for (int64_t it = 0; it < iters; ++it) {
        const int s = (int)(it % NS);
        const int nr = my_rows - it * R < R ? (int)(my_rows - it * R) : R;
        // the bias and row weights do not come through the ring: loaded
        // before the stage wait so their latency overlaps it
        float ba[U][8], bb[U][8], wr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cub = cu_of[u] < gpr ? cu_of[u] : 0;
            bias8(bias, (int64_t)cub * 8, ba[u]);
            bias8(bias, F + (int64_t)cub * 8, bb[u]);
            wr[u] = slot_of[u] < nr ? w[blockIdx.x + (it * R + slot_of[u]) * gridDim.x] : 0.0f;
        }
        if (!dead && !mbar_wait(ring.full(s), (uint32_t)((it / NS) & 1))) {
            atomicOr(&g_device_error, 1u);
            dead = true;
        }
        float acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc[u] = 0.0f;
            const int k = slot_of[u], cu = cu_of[u];
            if (!dead && k < nr && cu < gpr) {
                const int64_t r = blockIdx.x + (it * R + k) * gridDim.x;
                const unsigned char* st = data + (size_t)s * P::kStage + (uint32_t)(k * gpad + cu) * P::kUnitBytes;
                Raw8<T> ra, rb, rg;
                lds8(st + kA, ra);
                lds8(st + kB, rb);
                lds8(st + kG, rg);
                float fa[8], fb[8], fg[8];
                widen8(ra, fa);
                widen8(rb, fb);
                widen8(rg, fg);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float da, db;
                    const float term =
                        glu_bwd1<SWIGLU, kPrecise, true>(fa[j] + ba[u][j], fb[j] + bb[u][j], fg[j], wr[u], &da, &db);
                    acc[u] += fg[j] * term;
                    fa[j] = da;
                    fb[j] = db;
                }
                narrow8(fa, ra);
                narrow8(fb, rb);
                T* dxr = dx + r * 2 * F + (int64_t)cu * 8;
                st8(dxr, ra);
                st8(dxr + F, rb);
            }
        }
        if (!dead) {
            __syncwarp();
            if ((t & 31) == 0)
                mbar_arrive(ring.empty(s));
        }
        // every row of the stage is done: per warp the xor tree, then each
        // row's warps in order
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc[u] += __shfl_xor_sync(0xFFFFFFFFu, acc[u], o);
            if ((t & 31) == 0)
                warp_sums[parity][u * kConsumerWarps + (t >> 5)] = acc[u];
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
        if (t < nr) {
            float sum = 0.0f;
            for (int i = 0; i < gpad / 32; ++i)
                sum += warp_sums[parity][t * (gpad / 32) + i];
            dw[blockIdx.x + (it * R + t) * gridDim.x] = sum;
        }
        parity ^= 1;
    }
}

// The weighted SwiGLU backward at any width and alignment through the ring:
// the same rows, chunks, units, per-thread order and row-end tree as
// swiglu_bwd_weighted_pipe (so dweight has the same bits), but each stage
// holds, per stream (a, b, g), the 16-byte vectors that cover the chunk's
// run; a consumer reads its unit at the run's phase (img_ld8).  A chunk
// never leaves its row.  Copies are clipped to the aligned vectors inside x
// and g, so units of the first and last rows whose vectors were clipped read
// global memory instead.
template <typename T>
struct WbwdRPipe {
    static constexpr int kU = MFX_UNROLL_WBWD_RPIPE;
    static constexpr uint32_t kImg = kU * kConsumers * 8 * (uint32_t)sizeof(T) + 32;
    static constexpr uint32_t kStage = 3 * kImg;
    static constexpr int kStages = ring_stages(MFX_RING_KB_WBWD_RPIPE * 1024, kStage);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kStage;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

template <typename T>
__global__ void __launch_bounds__(kPipeThreads, MFX_PIPE_MINB_WBWD)
swiglu_bwd_weighted_rpipe(const T* g, const T* x, const T* __restrict__ bias, const float* __restrict__ w,
                          T* dx, float* __restrict__ dw, int64_t rows, int64_t F)
{
    using P = WbwdRPipe<T>;
    constexpr int NS = P::kStages, U = P::kU;
    constexpr int ES = (int)sizeof(T);
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    extern __shared__ __align__(128) unsigned char smem[];
    // row-end sums without a block barrier: each warp posts its sum in the
    // row's slot and counts itself in; the last warp adds the 8 sums in warp
    // order.  A warp runs at most NS stages ahead of the slowest, so a slot
    // is reused only after its previous row was finished (kRowSlots > NS).
    constexpr int kRowSlots = 16;
    static_assert(NS < kRowSlots, "row slots");
    __shared__ float warp_sums[kRowSlots][kConsumerWarps];
    __shared__ unsigned row_arrived[kRowSlots];
    if (threadIdx.x < kRowSlots)
        row_arrived[threadIdx.x] = 0;
    const Ring ring = ring_setup<NS>(smem);  // (its barrier publishes the zeros)
    unsigned char* data = smem + kRingHeader;
    const int64_t gpr = (F + 7) / 8;
    const int64_t nchunk = (gpr + U * kConsumers - 1) / (U * kConsumers);
    const int64_t my_rows = rows > blockIdx.x ? (rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t iters = my_rows * nchunk;
    const uintptr_t x_lo = reinterpret_cast<uintptr_t>(x), g_lo = reinterpret_cast<uintptr_t>(g);
    const uintptr_t g_hi = g_lo + (uintptr_t)(rows * F * ES), x_hi = x_lo + 2 * (g_hi - g_lo);

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) != 0)
            return;
        const uintptr_t lo16[2] = {(x_lo + 15) & ~(uintptr_t)15, (g_lo + 15) & ~(uintptr_t)15};
        const uintptr_t hi16[2] = {x_hi & ~(uintptr_t)15, g_hi & ~(uintptr_t)15};
        int64_t r = blockIdx.x, chunk = 0;
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
            const int64_t e0 = chunk * U * kConsumers * 8;
            const int64_t len = F - e0 < U * kConsumers * 8 ? F - e0 : U * kConsumers * 8;
            const uintptr_t s0[3] = {reinterpret_cast<uintptr_t>(x + r * 2 * F + e0),
                                     reinterpret_cast<uintptr_t>(x + r * 2 * F + F + e0),
                                     reinterpret_cast<uintptr_t>(g + r * F + e0)};
            uintptr_t lo[3], hi[3];
            uint32_t total = 0;
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                const int b = q == 2;  // which buffer
                const uintptr_t b16 = s0[q] & ~(uintptr_t)15;
                const uintptr_t e16 = (s0[q] + (uintptr_t)(len * ES) + 15) & ~(uintptr_t)15;
                lo[q] = b16 > lo16[b] ? b16 : lo16[b];
                hi[q] = e16 < hi16[b] ? e16 : hi16[b];
                if (hi[q] <= lo[q])
                    hi[q] = lo[q] = b16;
                total += (uint32_t)(hi[q] - lo[q]);
            }
            mbar_arrive_expect_tx(ring.full(s), total);
            unsigned char* st = data + (size_t)s * P::kStage;
#pragma unroll
            for (int q = 0; q < 3; ++q)
                if (hi[q] > lo[q])
                    bulk_g2s(smem_addr(st + q * P::kImg + (lo[q] - (s0[q] & ~(uintptr_t)15))),
                             reinterpret_cast<const void*>(lo[q]), (uint32_t)(hi[q] - lo[q]), ring.full(s));
            if (++chunk == nchunk) {
                chunk = 0;
                r += gridDim.x;
            }
        }
        return;
    }

    const int t = threadIdx.x;
    float acc = 0.0f;
    int slot = 0;
    bool dead = false;
    int64_t r = blockIdx.x, chunk = 0;
    int s = 0;
    uint32_t ph = 0;
    for (int64_t it = 0; it < iters; ++it) {
        const float wr = w[r];
        if (!dead && !mbar_wait(ring.full(s), ph)) {
            atomicOr(&g_device_error, 1u);
            dead = true;
        }
        const int64_t e0 = chunk * U * kConsumers * 8;
        const T* pa0 = x + r * 2 * F + e0;
        const T* pg0 = g + r * F + e0;
        const uint32_t pha = (uint32_t)(reinterpret_cast<uintptr_t>(pa0) & 15u);
        const uint32_t phb = (uint32_t)(reinterpret_cast<uintptr_t>(pa0 + F) & 15u);
        const uint32_t phg = (uint32_t)(reinterpret_cast<uintptr_t>(pg0) & 15u);
        const bool edge = r == 0 || r == rows - 1;
        const unsigned char* st = data + (size_t)s * P::kStage;
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int cu = k * kConsumers + t;
            const int64_t cg = chunk * U * kConsumers + cu;
            if (!dead && cg < gpr) {
                const int n = F - cg * 8 < 8 ? (int)(F - cg * 8) : 8;
                const T* pa = pa0 + cu * 8;
                const T* pg = pg0 + cu * 8;
                float fa[8], fb[8], fg[8];
                if (!edge || (in_vectors(pa, x_lo, x_hi) && in_vectors(pa + F, x_lo, x_hi) &&
                              in_vectors(pg, g_lo, g_hi))) {
                    const uint32_t d = (uint32_t)cu * 8u * ES;
                    Raw8<T> ra, rb, rg;
                    img_ld8(st, pha + d, ra);
                    img_ld8(st + P::kImg, phb + d, rb);
                    img_ld8(st + 2 * P::kImg, phg + d, rg);
                    widen8(ra, fa);
                    widen8(rb, fb);
                    widen8(rg, fg);
                } else {
                    load8f(pa, false, n, fa);
                    load8f(pa + F, false, n, fb);
                    load8f(pg, false, n, fg);
                }
                // the bias per unit (L1 hits: every row reads the same columns)
                const int64_t c0 = cg * 8;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j < n) {
                        float da, db;
                        const float term = glu_bwd1<SWIGLU, kPrecise, true>(
                            fa[j] + bias1(bias, c0 + j), fb[j] + bias1(bias, F + c0 + j), fg[j], wr, &da, &db);
                        acc += fg[j] * term;
                        fa[j] = da;
                        fb[j] = db;
                    }
                }
                T* pd = dx + r * 2 * F + e0 + cu * 8;
                if (n == 8) {
                    Raw8<T> oa, ob;
                    narrow8(fa, oa);
                    narrow8(fb, ob);
                    st8_words(pd, oa);
                    st8_words(pd + F, ob);
                } else {
                    store8f(pd, false, n, fa);
                    store8f(pd + F, false, n, fb);
                }
            }
        }
        if (!dead) {
            __syncwarp();
            if ((t & 31) == 0)
                mbar_arrive(ring.empty(s));
        }
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
        if (chunk == nchunk - 1) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
            if ((t & 31) == 0) {
                warp_sums[slot][t >> 5] = acc;
                __threadfence_block();
                if (atomicAdd(&row_arrived[slot], 1u) == kConsumerWarps - 1) {
                    __threadfence_block();
                    const volatile float* ws = warp_sums[slot];
                    float sum = 0.0f;
#pragma unroll
                    for (int i = 0; i < kConsumerWarps; ++i)
                        sum += ws[i];
                    dw[r] = sum;
                    row_arrived[slot] = 0;
                }
            }
            __syncwarp();
            acc = 0.0f;
            slot = slot + 1 == kRowSlots ? 0 : slot + 1;
            chunk = 0;
            r += gridDim.x;
        } else {
            ++chunk;
        }
    }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
// The realigning form for the widths and alignments the fixed forms cannot
// take, from kRealignMinF columns on (narrower rows keep the element-wise
// form).  Returns false (nothing launched) when it does not apply: a pointer
// not on an element boundary, or too few elements for one unit.
constexpr int64_t kRealignMinF = 64;

template <typename T, int KIND, bool WEIGHTED, bool BWD>
bool launch_realign(const T* g, const T* x, const T* bias, const float* w, T* out, int64_t rows, int64_t F,
                    cudaStream_t s)
{
    const T* ref = BWD ? g : out;  // the flat [rows, F] grid the units tile
    const uintptr_t mis = reinterpret_cast<uintptr_t>(ref) & 15u;
    if (mis % sizeof(T) || (reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out) |
                            reinterpret_cast<uintptr_t>(bias) | reinterpret_cast<uintptr_t>(g)) % sizeof(T))
        return false;
    const int head = (int)(((16u - mis) & 15u) / sizeof(T));
    const int64_t n = rows * F;
    if (n - head < 8)
        return false;
    const int64_t units = (n - head) / 8;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(x), hi = lo + (uintptr_t)(n * 2 * sizeof(T));
    if (MFX_GLU_RPIPE && F >= kConsumers * 8) {
        const void* k = (const void*)glu_rpipe<T, KIND, WEIGHTED, BWD>;
        constexpr size_t smem = GluRPipe<T, BWD>::kSmem;
        const Grid grid = plan_fixed_any(k, kPipeThreads, smem, units, F);
        if (grid.fixed) {
            glu_rpipe<T, KIND, WEIGHTED, BWD><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                g, x, bias, w, out, rows, F, units, grid.S, head, (int)((n - head) % 8), lo, hi);
            return true;
        }
    }
    const void* k = (const void*)glu_realign<T, KIND, WEIGHTED, BWD>;
    const Grid grid = plan_fixed_any(k, kThreads, 0, units, F);
    if (!grid.fixed)
        return false;
    glu_realign<T, KIND, WEIGHTED, BWD><<<(unsigned)grid.blocks, kThreads, 0, s>>>(
        g, x, bias, w, out, rows, F, units, grid.S, head, (int)((n - head) % 8), lo, hi);
    return true;
}

template <typename T, int KIND, bool WEIGHTED>
int launch_fwd(const void* x, const void* bias, const float* w, void* out, int64_t rows, int64_t F,
               cudaStream_t s)
{
    const T* xp = static_cast<const T*>(x);
    const T* bp = static_cast<const T*>(bias);
    T* op = static_cast<T*>(out);
    const bool vec = F % 8 == 0 && aligned16(x) && aligned16(out) && (!bias || aligned16(bias));
    if (vec && MFX_PIPE_GLU && F / 8 >= 32) {
        const void* k = (const void*)glu_pipe<T, KIND, WEIGHTED, false>;
        constexpr size_t smem = GluPipe<T, KIND, false>::kSmem;
        const Grid grid = plan_grid_ex(k, kPipeThreads, smem, rows * (F / 8), F / 8, true);
        if (grid.fixed) {
            glu_pipe<T, KIND, WEIGHTED, false><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                nullptr, xp, bp, w, op, rows, F);
            return launch_status();
        }
    }
    if (vec) {
        const Grid grid = plan_grid((const void*)glu_fwd_fixed<T, KIND, WEIGHTED>, rows * (F / 8), F / 8, true);
        if (grid.fixed) {
            glu_fwd_fixed<T, KIND, WEIGHTED><<<(unsigned)grid.blocks, kThreads, 0, s>>>(xp, bp, w, op, rows, F);
            return launch_status();
        }
    }
    if (F >= kRealignMinF && launch_realign<T, KIND, WEIGHTED, false>(nullptr, xp, bp, w, op, rows, F, s))
        return launch_status();
    const int64_t gpr = (F + 7) / 8;
    const Grid grid = plan_grid((const void*)glu_fwd_generic<T, KIND, WEIGHTED>, rows * gpr, 0, false);
    const int64_t S = grid.blocks * kThreads;
    glu_fwd_generic<T, KIND, WEIGHTED><<<(unsigned)grid.blocks, kThreads, 0, s>>>(
        xp, bp, w, op, rows, F, gpr, S % gpr, S / gpr, vec);
    return launch_status();
}

template <typename T, int KIND>
int launch_bwd(const void* g, const void* x, const void* bias, const float* w, void* dx, float* dw,
               int64_t rows, int64_t F, cudaStream_t s)
{
    const T* gp = static_cast<const T*>(g);
    const T* xp = static_cast<const T*>(x);
    const T* bp = static_cast<const T*>(bias);
    T* dxp = static_cast<T*>(dx);
    const bool vec = F % 8 == 0 && aligned16(g) && aligned16(x) && aligned16(dx) &&
                     (!bias || aligned16(bias));
    if (w && vec && MFX_PIPE_WBWD && MFX_WBWD_ROWS && F / 8 <= kConsumers) {
        // short rows: several whole rows per stage
        const void* k = (const void*)swiglu_bwd_weighted_pipe_rows<T>;
        constexpr size_t smem = WbwdPipe<T>::kSmem;
        const int64_t gpad = (F / 8 + 31) & ~31, R = WbwdPipe<T>::kU * kConsumers / gpad;
        const Grid grid = plan_grid_ex(k, kPipeThreads, smem, (rows + R - 1) / R * kThreads, 0, false);
        swiglu_bwd_weighted_pipe_rows<T><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(gp, xp, bp, w, dxp, dw,
                                                                                             rows, F);
        return launch_status();
    }
    if (w && vec && MFX_PIPE_WBWD) {
        const void* k = (const void*)swiglu_bwd_weighted_pipe<T>;
        constexpr size_t smem = WbwdPipe<T>::kSmem;
        // one block per row at a time: min(rows, resident blocks) blocks
        const Grid grid = plan_grid_ex(k, kPipeThreads, smem, rows * kThreads, 0, false);
        swiglu_bwd_weighted_pipe<T><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(gp, xp, bp, w, dxp, dw, rows, F);
        return launch_status();
    }
    // the realigning ring where it measured faster: bf16 rows of a width
    // that is a multiple of 8 behind misaligned pointers (0.49 of the copy
    // peak against 0.39); at odd widths the grid-stride form is faster (0.44
    // against 0.39 at 65536 x 4099).  Both give dweight the same bits.
    if (w && !vec && MFX_WBWD_RPIPE && DTypeInfo<T>::kBf16 && F % 8 == 0 && F >= kRealignMinF) {
        const void* k = (const void*)swiglu_bwd_weighted_rpipe<T>;
        constexpr size_t smem = WbwdRPipe<T>::kSmem;
        const Grid grid = plan_grid_ex(k, kPipeThreads, smem, rows * kThreads, 0, false);
        swiglu_bwd_weighted_rpipe<T><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(gp, xp, bp, w, dxp, dw, rows,
                                                                                         F);
        return launch_status();
    }
    if (w) {
        const void* k = vec ? (const void*)swiglu_bwd_weighted<T, true> : (const void*)swiglu_bwd_weighted<T, false>;
        const int64_t cap = (int64_t)sm_count() * blocks_per_sm(k);
        const unsigned blocks = (unsigned)(rows < cap ? rows : cap);
        if (vec)
            swiglu_bwd_weighted<T, true><<<blocks, kThreads, 0, s>>>(gp, xp, bp, w, dxp, dw, rows, F);
        else
            swiglu_bwd_weighted<T, false><<<blocks, kThreads, 0, s>>>(gp, xp, bp, w, dxp, dw, rows, F);
        return launch_status();
    }
    if (vec && MFX_PIPE_GLU && F / 8 >= 32) {
        const void* k = (const void*)glu_pipe<T, KIND, false, true>;
        constexpr size_t smem = GluPipe<T, KIND, true>::kSmem;
        const Grid grid = plan_grid_ex(k, kPipeThreads, smem, rows * (F / 8), F / 8, true);
        if (grid.fixed) {
            glu_pipe<T, KIND, false, true><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                gp, xp, bp, nullptr, dxp, rows, F);
            return launch_status();
        }
    }
    if (vec) {
        const Grid grid = plan_grid((const void*)glu_bwd_fixed<T, KIND>, rows * (F / 8), F / 8, true);
        if (grid.fixed) {
            glu_bwd_fixed<T, KIND><<<(unsigned)grid.blocks, kThreads, 0, s>>>(gp, xp, bp, dxp, rows, F);
            return launch_status();
        }
    }
    if (F >= kRealignMinF && launch_realign<T, KIND, false, true>(gp, xp, bp, nullptr, dxp, rows, F, s))
        return launch_status();
    const int64_t gpr = (F + 7) / 8;
    const Grid grid = plan_grid((const void*)glu_bwd_generic<T, KIND>, rows * gpr, 0, false);
    const int64_t S = grid.blocks * kThreads;
    glu_bwd_generic<T, KIND><<<(unsigned)grid.blocks, kThreads, 0, s>>>(gp, xp, bp, dxp, rows, F, gpr,
                                                                       S % gpr, S / gpr, vec);
    return launch_status();
}

// GLU backward plus the fused bias gradient (width 2F).  The weighted
// SwiGLU backward owns rows, not columns, so with a weight the partials come
// from a pass over the stored dx instead.
template <typename T, int KIND>
int launch_bwd_dbias(const void* g, const void* x, const void* bias, const float* w, void* dx, float* dw,
                     void* dbias, int64_t rows, int64_t F, void* workspace, size_t* ws_bytes, cudaStream_t s)
{
    const void* k = (const void*)glu_pipe<T, KIND, false, true, true>;
    constexpr size_t smem = GluPipe<T, KIND, true>::kSmem;
    const int64_t W = 2 * F, gpr = F / 8;
    int64_t J_pipe = 0;
    Grid grid;
    if (MFX_PIPE_GLU && !w && F % 8 == 0 && gpr >= 32) {
        grid = plan_grid_ex(k, kPipeThreads, smem, rows * gpr, gpr, true);
        if (grid.fixed)
            J_pipe = grid.blocks * kThreads / gpr;
    }
    const int64_t J_gen = dbias_generic_lanes(rows);
    bool query = false;
    int st = dbias_workspace(J_pipe > J_gen ? J_pipe : J_gen, W, workspace, ws_bytes, &query);
    if (st != MFX_OK || query)
        return st;
    float* ws = static_cast<float*>(workspace);
    const bool pipe_ok = J_pipe > 0 && aligned16(g) && aligned16(x) && aligned16(dx) && (!bias || aligned16(bias));
    if (pipe_ok) {
        glu_pipe<T, KIND, false, true, true><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
            static_cast<const T*>(g), static_cast<const T*>(x), static_cast<const T*>(bias), nullptr,
            static_cast<T*>(dx), rows, F, ws);
        st = launch_status();
        return st != MFX_OK ? st : launch_dbias_finish(dtype_code<T>(), ws, J_pipe, W, dbias, s);
    }
    st = launch_bwd<T, KIND>(g, x, bias, w, dx, dw, rows, F, s);
    if (st == MFX_OK)
        st = launch_column_partials(dtype_code<T>(), dx, rows, W, J_gen, ws, s);
    return st != MFX_OK ? st : launch_dbias_finish(dtype_code<T>(), ws, J_gen, W, dbias, s);
}

// Shapes: rows x 2F input; returns MFX_OK with *empty set when nothing to do.
int check_glu(int dt, int64_t rows, int64_t F, bool* empty)
{
    *empty = false;
    if (!valid_dtype(dt))
        return MFX_ERR_DTYPE;
    if (rows < 0 || F < 0)
        return MFX_ERR_SHAPE;
    int64_t n = 0, bytes = 0;
    if (!mul_ok(rows, F, &n) || !mul_ok(n, 32, &bytes))
        return MFX_ERR_SHAPE;
    *empty = n == 0;
    return MFX_OK;
}

template <int KIND>
int glu_fwd_entry(int dt, int64_t rows, int64_t F, const void* x, const void* bias, const float* w,
                  void* out, void* stream)
{
    bool empty = false;
    int st = check_glu(dt, rows, F, &empty);
    if (st != MFX_OK || empty)
        return st;
    if (!x || !out)
        return MFX_ERR_NULL;
    const int64_t es = dtype_bytes(dt);
    const int64_t xb = rows * 2 * F * es, ob = rows * F * es;
    if (overlaps(x, xb, out, ob) || overlaps(bias, 2 * F * es, out, ob) || overlaps(w, rows * 4, out, ob))
        return MFX_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (w)
        return dt == MFX_BF16 ? launch_fwd<bf16, KIND, true>(x, bias, w, out, rows, F, s)
                              : launch_fwd<float, KIND, true>(x, bias, w, out, rows, F, s);
    return dt == MFX_BF16 ? launch_fwd<bf16, KIND, false>(x, bias, nullptr, out, rows, F, s)
                          : launch_fwd<float, KIND, false>(x, bias, nullptr, out, rows, F, s);
}

// Null and overlap checks of the GLU backward (nonempty shapes).
int glu_bwd_entry_check(int dt, int64_t rows, int64_t F, const void* g, const void* x, const void* bias,
                        const float* w, void* dx, float* dw)
{
    if (!g || !x || !dx || (w && !dw))
        return MFX_ERR_NULL;
    const int64_t es = dtype_bytes(dt);
    const int64_t xb = rows * 2 * F * es, gb = rows * F * es;
    if (partial_overlap(x, xb, dx, xb) || overlaps(g, gb, dx, xb) || overlaps(bias, 2 * F * es, dx, xb) ||
        overlaps(w, rows * 4, dx, xb))
        return MFX_ERR_ALIAS;
    if (w && (overlaps(dw, rows * 4, dx, xb) || overlaps(dw, rows * 4, x, xb) ||
              overlaps(dw, rows * 4, g, gb) || overlaps(dw, rows * 4, w, rows * 4) ||
              overlaps(dw, rows * 4, bias, 2 * F * es)))
        return MFX_ERR_ALIAS;
    return MFX_OK;
}

template <int KIND>
int glu_bwd_entry(int dt, int64_t rows, int64_t F, const void* g, const void* x, const void* bias,
                  const float* w, void* dx, float* dw, void* stream)
{
    bool empty = false;
    int st = check_glu(dt, rows, F, &empty);
    if (st != MFX_OK || empty)
        return st;
    st = glu_bwd_entry_check(dt, rows, F, g, x, bias, w, dx, dw);
    if (st != MFX_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == MFX_BF16 ? launch_bwd<bf16, KIND>(g, x, bias, w, dx, dw, rows, F, s)
                          : launch_bwd<float, KIND>(g, x, bias, w, dx, dw, rows, F, s);
}

template <int KIND>
int glu_bwd_dbias_entry(int dt, int64_t rows, int64_t F, const void* g, const void* x, const void* bias,
                        const float* w, void* dx, float* dw, void* dbias, void* workspace, size_t* ws_bytes,
                        void* stream)
{
    bool empty = false;
    int st = check_glu(dt, rows, F, &empty);
    if (st != MFX_OK)
        return st;
    if (!ws_bytes)
        return MFX_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t es = dtype_bytes(dt), W = 2 * F;
    if (empty) {
        if (!workspace) {
            *ws_bytes = 0;
            return MFX_OK;
        }
        if (W == 0)
            return MFX_OK;
        if (!dbias)
            return MFX_ERR_NULL;
        return cudaMemsetAsync(dbias, 0, (size_t)(W * es), s) == cudaSuccess ? MFX_OK
                                                                             : cuda_failure(cudaGetLastError());
    }
    if (workspace) {
        if (!dbias)
            return MFX_ERR_NULL;
        const int64_t xb = rows * W * es, wsb = (int64_t)*ws_bytes;
        if (overlaps(dbias, W * es, dx, xb) || overlaps(dbias, W * es, x, xb) ||
            overlaps(dbias, W * es, g, rows * F * es) || overlaps(dbias, W * es, bias, W * es) ||
            overlaps(workspace, wsb, dx, xb) || overlaps(workspace, wsb, x, xb) ||
            overlaps(workspace, wsb, g, rows * F * es) || overlaps(workspace, wsb, dbias, W * es) ||
            (w && overlaps(dbias, W * es, dw, rows * 4)) || (w && overlaps(workspace, wsb, dw, rows * 4)))
            return MFX_ERR_ALIAS;
        // the plain backward's own checks (nulls, overlaps) without launching
        st = glu_bwd_entry_check(dt, rows, F, g, x, bias, w, dx, dw);
        if (st != MFX_OK)
            return st;
    }
    return dt == MFX_BF16 ? launch_bwd_dbias<bf16, KIND>(g, x, bias, w, dx, dw, dbias, rows, F, workspace, ws_bytes, s)
                          : launch_bwd_dbias<float, KIND>(g, x, bias, w, dx, dw, dbias, rows, F, workspace, ws_bytes, s);
}

}  // namespace

unsigned take_device_error_glu()
{
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess)
        return 0xFFu;
    if (v)
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    return v;
}

}  // namespace mfx

extern "C" int mfx_bias_geglu_fwd(int dt, int64_t rows, int64_t F, const void* x, const void* bias,
                                  void* out, void* stream)
{
    return mfx::glu_fwd_entry<mfx::GEGLU>(dt, rows, F, x, bias, nullptr, out, stream);
}

extern "C" int mfx_bias_geglu_bwd(int dt, int64_t rows, int64_t F, const void* g, const void* x,
                                  const void* bias, void* dx, void* stream)
{
    return mfx::glu_bwd_entry<mfx::GEGLU>(dt, rows, F, g, x, bias, nullptr, dx, nullptr, stream);
}

extern "C" int mfx_bias_swiglu_fwd(int dt, int64_t rows, int64_t F, const void* x, const void* bias,
                                   const float* weight, void* out, void* stream)
{
    return mfx::glu_fwd_entry<mfx::SWIGLU>(dt, rows, F, x, bias, weight, out, stream);
}

extern "C" int mfx_bias_swiglu_bwd(int dt, int64_t rows, int64_t F, const void* g, const void* x,
                                   const void* bias, const float* weight, void* dx, float* dweight,
                                   void* stream)
{
    return mfx::glu_bwd_entry<mfx::SWIGLU>(dt, rows, F, g, x, bias, weight, dx, dweight, stream);
}

extern "C" int mfx_bias_geglu_bwd_dbias(int dt, int64_t rows, int64_t F, const void* g, const void* x,
                                        const void* bias, void* dx, void* dbias, void* workspace,
                                        size_t* workspace_bytes, void* stream)
{
    return mfx::glu_bwd_dbias_entry<mfx::GEGLU>(dt, rows, F, g, x, bias, nullptr, dx, nullptr, dbias, workspace,
                                                workspace_bytes, stream);
}

extern "C" int mfx_bias_swiglu_bwd_dbias(int dt, int64_t rows, int64_t F, const void* g, const void* x,
                                         const void* bias, const float* weight, void* dx, float* dweight,
                                         void* dbias, void* workspace, size_t* workspace_bytes, void* stream)
{
    return mfx::glu_bwd_dbias_entry<mfx::SWIGLU>(dt, rows, F, g, x, bias, weight, dx, dweight, dbias, workspace,
                                                 workspace_bytes, stream);
}
