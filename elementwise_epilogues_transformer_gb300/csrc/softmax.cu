// softmax.cu -- fused scale-mask-softmax, forward and backward.
//
// Megatron-LM operator fusion walkthrough (www.wmrh.cn/news/51426), §6.2:
// ScaledSoftmax (scale, softmax), ScaledMaskedSoftmax (scale, the given
// additive mask broadcast over [b, np, sq, sk], softmax) and
// ScaledUpperTriangMaskedSoftmax (scale, the causal mask k > q, softmax, on
// [attn_batches, sq, sq]); the three share one backward that needs only the
// softmax results and the scale (§6.2), dx = scale * y * (dy - sum_k dy_k y_k).
// §6.3: with a scale the softmax runs in fp32; inputs and outputs keep the
// input dtype.
//
// Layout: rows of sk contiguous elements, one softmax per row.  A "team" of
// 2^lg threads (1 .. 256) owns one row at a time and holds it in registers,
// C chunks of 8 elements per thread, so the row is read from HBM once and
// written once; the row maximum and sum are team reductions (shuffles, and
// for teams wider than a warp a fixed-order pass over the warps' partials in
// shared memory behind a named barrier per team).  Rows longer than
// 8 x C x 256 take a block-per-row kernel that reads the row three times
// (max, sum, write); the second and third reads hit L2.
//
// Accuracy: the exponent of each element is formed as one fused multiply-add
// x * scale + (mask - max), so large scores lose nothing to the rounding of
// x * scale; the row maximum only shifts every exponent by the same amount.
// The fp32 kernels evaluate exp with expf and add the row sum with the
// compensated summation of Ogita, Rump and Oishi ("Accurate sum and dot
// product", SIAM J. Sci. Comput. 26(6), 2005: Knuth's TwoSum per addition,
// the rounding errors summed alongside).  The bf16 kernels use the hardware
// base-2 exponential.  The backward's row sum of dy * y is that paper's
// compensated dot product (FMA TwoProduct plus TwoSum) in both dtypes, so
// dy_k - sum keeps its accuracy where the two nearly cancel.
#include <initializer_list>

#include "mfx_device.cuh"
#include "mfx_host.h"

#ifndef MFX_SOFTMAX_C
#define MFX_SOFTMAX_C 4  // chunks of 8 elements per thread in the register kernels
#endif
#ifndef MFX_MINB_SOFTMAX
#define MFX_MINB_SOFTMAX 2
#endif

namespace mfx {
namespace {

constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------
// Error-free transformations (Knuth's TwoSum; the FMA form of TwoProduct).
// ---------------------------------------------------------------------------
struct Acc {
    float s, c;  // running sum and the sum of its rounding errors
};

// A sum that is no longer finite keeps its error term as it is (the error
// of an infinite or NaN sum would be NaN and spoil an infinite result).
__device__ __forceinline__ void two_sum_add(Acc& a, float v)
{
    const float s = __fadd_rn(a.s, v);
    const float z = __fsub_rn(s, a.s);
    const float e = __fadd_rn(__fsub_rn(a.s, __fsub_rn(s, z)), __fsub_rn(v, z));
    a.s = s;
    a.c = fabsf(s) < INFINITY ? __fadd_rn(a.c, e) : a.c;
}

__device__ __forceinline__ void two_prod_add(Acc& a, float x, float y)
{
    const float p = __fmul_rn(x, y);
    const float pe = fabsf(p) < INFINITY ? fmaf(x, y, -p) : 0.0f;
    two_sum_add(a, p);
    a.c = __fadd_rn(a.c, pe);
}

__device__ __forceinline__ Acc acc_merge(Acc a, Acc b)
{
    two_sum_add(a, b.s);
    a.c = __fadd_rn(a.c, b.c);
    return a;
}

__device__ __forceinline__ float acc_value(Acc a) { return __fadd_rn(a.s, a.c); }

// ---------------------------------------------------------------------------
// Team reductions.  Teams of up to 32 threads are aligned lane groups of one
// warp; wider teams are whole warps (team `tm` owns warps tm*W .. tm*W+W-1)
// and meet at named barrier 1 + tm.  `slot` selects one of two shared-memory
// buffers so that consecutive reductions need one barrier each.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void team_bar(int tm, int tpr)
{
    asm volatile("bar.sync %0, %1;" ::"r"(1 + tm), "r"(tpr) : "memory");
}

__device__ __forceinline__ float team_max(float v, int lg, int tm, float (*buf)[kWarps], int slot)
{
    const int tpr = 1 << lg;
    const int w = lg < 5 ? lg : 5;
    for (int o = (1 << w) >> 1; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if (lg > 5) {
        if ((threadIdx.x & 31) == 0)
            buf[slot][threadIdx.x >> 5] = v;
        team_bar(tm, tpr);
        const int w0 = tm << (lg - 5), nw = 1 << (lg - 5);
        v = buf[slot][w0];
        for (int i = 1; i < nw; ++i)
            v = fmaxf(v, buf[slot][w0 + i]);
    }
    return v;
}

__device__ __forceinline__ Acc team_acc(Acc a, int lg, int tm, float (*bs)[kWarps], float (*bc)[kWarps], int slot)
{
    const int tpr = 1 << lg;
    const int w = lg < 5 ? lg : 5;
    for (int o = (1 << w) >> 1; o > 0; o >>= 1) {
        Acc b{__shfl_xor_sync(0xFFFFFFFFu, a.s, o), __shfl_xor_sync(0xFFFFFFFFu, a.c, o)};
        // both partners merge in the same order (lower lane's value first)
        a = (threadIdx.x & o) ? acc_merge(b, a) : acc_merge(a, b);
    }
    if (lg > 5) {
        if ((threadIdx.x & 31) == 0) {
            bs[slot][threadIdx.x >> 5] = a.s;
            bc[slot][threadIdx.x >> 5] = a.c;
        }
        team_bar(tm, tpr);
        const int w0 = tm << (lg - 5), nw = 1 << (lg - 5);
        a = Acc{bs[slot][w0], bc[slot][w0]};
        for (int i = 1; i < nw; ++i)
            a = acc_merge(a, Acc{bs[slot][w0 + i], bc[slot][w0 + i]});
    }
    return a;
}

// Plain fp32 sum for the bf16 forward (the bf16 rounding of y hides the
// difference); same fixed order.
__device__ __forceinline__ float team_sum(float v, int lg, int tm, float (*buf)[kWarps], int slot)
{
    const int tpr = 1 << lg;
    const int w = lg < 5 ? lg : 5;
    for (int o = (1 << w) >> 1; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = (threadIdx.x & o) ? u + v : v + u;
    }
    if (lg > 5) {
        if ((threadIdx.x & 31) == 0)
            buf[slot][threadIdx.x >> 5] = v;
        team_bar(tm, tpr);
        const int w0 = tm << (lg - 5), nw = 1 << (lg - 5);
        v = buf[slot][w0];
        for (int i = 1; i < nw; ++i)
            v += buf[slot][w0 + i];
    }
    return v;
}

// ---------------------------------------------------------------------------
// Row geometry.
// ---------------------------------------------------------------------------
struct SoftmaxGeom {
    int64_t rows;          // b * np * sq
    int64_t sq, np, sk;    // query rows per (batch, head), heads, row length
    int64_t mb, mnp, msq;  // mask sizes (each 1 = broadcast, or the input's)
};

// Offset of the mask row that applies to input row r.
__device__ __forceinline__ int64_t mask_row(const SoftmaxGeom& g, int64_t r)
{
    const int64_t q = r % g.sq, bh = r / g.sq;
    const int64_t h = bh % g.np, i = bh / g.np;
    return (((g.mb == 1 ? 0 : i) * g.mnp + (g.mnp == 1 ? 0 : h)) * g.msq + (g.msq == 1 ? 0 : q)) * g.sk;
}

// exp(d) for d <= 0 (or NaN): expf in fp32; in bf16 the hardware 2^t at
// t = d log2(e), evaluated at t + 64 as ex2_neg does so that results down to
// 2^-190 survive.
template <bool PRECISE>
__device__ __forceinline__ float exp_le0(float d)
{
    if (PRECISE)
        return expf(d);
    return ex2_neg(fmaf(d, (float)kLog2e, 64.0f));
}

// ---------------------------------------------------------------------------
// Forward, register kernel.
// ---------------------------------------------------------------------------
template <typename T, int C, bool MASK, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, MFX_MINB_SOFTMAX)
softmax_fwd_team(const T* x, const T* __restrict__ mask, T* y, SoftmaxGeom g, float scale, int lg, int64_t iters,
                 bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    __shared__ float red_s[2][kWarps], red_c[2][kWarps];
    const int tpr = 1 << lg;
    const int tm = threadIdx.x >> lg, t = threadIdx.x & (tpr - 1);
    const int teams = kThreads >> lg;
    const int64_t G = (g.sk + 7) / 8;
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = ((int64_t)blockIdx.x + it * gridDim.x) * teams + tm;
        const bool active = r < g.rows;
        const int64_t valid = CAUSAL ? (active ? r % g.sq + 1 : 0) : (active ? g.sk : 0);
        const T* xr = x + (active ? r : 0) * g.sk;
        const T* mr = MASK ? mask + (active ? mask_row(g, r) : 0) : nullptr;
        float a[C][8], b[MASK ? C : 1][8];
        int n[C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int64_t e0 = (int64_t)(t + c * tpr) * 8;
            const int64_t left = valid - e0;
            n[c] = left <= 0 ? 0 : (left < 8 ? (int)left : 8);
            if (n[c] > 0) {
                load8f(xr + e0, vec, n[c], a[c]);
                if (MASK)
                    load8f(mr + e0, vec, n[c], b[MASK ? c : 0]);
            }
        }
        // row maximum of the scores x * scale + mask
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < C; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n[c])
                    m = fmaxf(m, MASK ? fmaf(a[c][j], scale, b[MASK ? c : 0][j]) : a[c][j] * scale);
        m = team_max(m, lg, tm, red_s, 0);
        // a row with no finite score left: all zeros
        const float mneg = m == -INFINITY ? 0.0f : -m;
        Acc acc{0.0f, 0.0f};
        float s = 0.0f;
#pragma unroll
        for (int c = 0; c < C; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float e = 0.0f;
                if (j < n[c]) {
                    const float d = fmaf(a[c][j], scale, MASK ? b[MASK ? c : 0][j] + mneg : mneg);
                    e = exp_le0<kPrecise>(d);
                }
                a[c][j] = e;
                if (kPrecise)
                    two_sum_add(acc, e);
                else
                    s += e;
            }
        float sum;
        if (kPrecise)
            sum = acc_value(team_acc(acc, lg, tm, red_s, red_c, 1));
        else
            sum = team_sum(s, lg, tm, red_s, 1);
        const bool none = m == -INFINITY;
        const float rs = __frcp_rn(sum);
        if (active) {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int64_t e0 = (int64_t)(t + c * tpr) * 8;
                if (e0 < g.sk) {
                    const int cnt = g.sk - e0 < 8 ? (int)(g.sk - e0) : 8;
                    float o[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        o[j] = j < n[c] && !none ? a[c][j] * rs : 0.0f;
                    store8f(y + r * g.sk + e0, vec, cnt, o);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Forward, long rows: one block per row, three passes over the row.
// ---------------------------------------------------------------------------
template <typename T, bool MASK, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
softmax_fwd_long(const T* x, const T* __restrict__ mask, T* y, SoftmaxGeom g, float scale, bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    __shared__ float red_s[2][kWarps], red_c[2][kWarps];
    const int t = threadIdx.x;
    for (int64_t r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const int64_t valid = CAUSAL ? r % g.sq + 1 : g.sk;
        const T* xr = x + r * g.sk;
        const T* mr = MASK ? mask + mask_row(g, r) : nullptr;
        float m = -INFINITY;
        for (int64_t e0 = (int64_t)t * 8; e0 < valid; e0 += kThreads * 8) {
            const int cnt = valid - e0 < 8 ? (int)(valid - e0) : 8;
            float a[8], b[8];
            load8f(xr + e0, vec, cnt, a);
            if (MASK)
                load8f(mr + e0, vec, cnt, b);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < cnt)
                    m = fmaxf(m, MASK ? fmaf(a[j], scale, b[j]) : a[j] * scale);
        }
        m = team_max(m, 8, 0, red_s, 0);
        const float mneg = m == -INFINITY ? 0.0f : -m;
        Acc acc{0.0f, 0.0f};
        float s = 0.0f;
        for (int64_t e0 = (int64_t)t * 8; e0 < valid; e0 += kThreads * 8) {
            const int cnt = valid - e0 < 8 ? (int)(valid - e0) : 8;
            float a[8], b[8];
            load8f(xr + e0, vec, cnt, a);
            if (MASK)
                load8f(mr + e0, vec, cnt, b);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < cnt) {
                    const float e = exp_le0<kPrecise>(fmaf(a[j], scale, MASK ? b[j] + mneg : mneg));
                    if (kPrecise)
                        two_sum_add(acc, e);
                    else
                        s += e;
                }
        }
        float sum;
        if (kPrecise)
            sum = acc_value(team_acc(acc, 8, 0, red_s, red_c, 1));
        else
            sum = team_sum(s, 8, 0, red_s, 1);
        const float rs = __frcp_rn(sum);
        for (int64_t e0 = (int64_t)t * 8; e0 < g.sk; e0 += kThreads * 8) {
            const int cnt = g.sk - e0 < 8 ? (int)(g.sk - e0) : 8;
            const int nv = m == -INFINITY ? 0 : valid - e0 <= 0 ? 0 : (valid - e0 < 8 ? (int)(valid - e0) : 8);
            float a[8], b[8], o[8];
            if (nv > 0) {
                load8f(xr + e0, vec, nv, a);
                if (MASK)
                    load8f(mr + e0, vec, nv, b);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o[j] = j < nv ? exp_le0<kPrecise>(fmaf(a[j], scale, MASK ? b[j] + mneg : mneg)) * rs : 0.0f;
            store8f(y + r * g.sk + e0, vec, cnt, o);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward, register kernel: dx = scale * y * (dy - sum_k dy_k y_k).
// ---------------------------------------------------------------------------
template <typename T, int C, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, MFX_MINB_SOFTMAX)
softmax_bwd_team(const T* dy, const T* y, T* dx, int64_t rows, int64_t sk, float scale, int lg, int64_t iters,
                 bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    __shared__ float red_s[2][kWarps], red_c[2][kWarps];
    const int tpr = 1 << lg;
    const int tm = threadIdx.x >> lg, t = threadIdx.x & (tpr - 1);
    const int teams = kThreads >> lg;
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = ((int64_t)blockIdx.x + it * gridDim.x) * teams + tm;
        const bool active = r < rows;
        const int64_t valid = active ? (CAUSAL ? r % sk + 1 : sk) : 0;
        const int64_t base = (active ? r : 0) * sk;
        float gv[C][8], yv[C][8];
        int n[C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int64_t e0 = (int64_t)(t + c * tpr) * 8;
            const int64_t left = valid - e0;
            n[c] = left <= 0 ? 0 : (left < 8 ? (int)left : 8);
            if (n[c] > 0) {
                load8f(dy + base + e0, vec, n[c], gv[c]);
                load8f(y + base + e0, vec, n[c], yv[c]);
            }
        }
        Acc acc{0.0f, 0.0f};
#pragma unroll
        for (int c = 0; c < C; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n[c])
                    two_prod_add(acc, gv[c][j], yv[c][j]);
        const float s = acc_value(team_acc(acc, lg, tm, red_s, red_c, (int)(it & 1)));
        if (active) {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int64_t e0 = (int64_t)(t + c * tpr) * 8;
                if (e0 < sk) {
                    const int cnt = sk - e0 < 8 ? (int)(sk - e0) : 8;
                    float o[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        o[j] = j < n[c] ? __fmul_rn(__fmul_rn(scale, yv[c][j]), __fsub_rn(gv[c][j], s)) : 0.0f;
                    store8f(dx + base + e0, vec, cnt, o);
                }
            }
        }
    }
}

template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
softmax_bwd_long(const T* dy, const T* y, T* dx, int64_t rows, int64_t sk, float scale, bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    __shared__ float red_s[2][kWarps], red_c[2][kWarps];
    const int t = threadIdx.x;
    int parity = 0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, parity ^= 1) {
        const int64_t valid = CAUSAL ? r % sk + 1 : sk;
        const int64_t base = r * sk;
        Acc acc{0.0f, 0.0f};
        for (int64_t e0 = (int64_t)t * 8; e0 < valid; e0 += kThreads * 8) {
            const int cnt = valid - e0 < 8 ? (int)(valid - e0) : 8;
            float gv[8], yv[8];
            load8f(dy + base + e0, vec, cnt, gv);
            load8f(y + base + e0, vec, cnt, yv);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < cnt)
                    two_prod_add(acc, gv[j], yv[j]);
        }
        const float s = acc_value(team_acc(acc, 8, 0, red_s, red_c, parity));
        for (int64_t e0 = (int64_t)t * 8; e0 < sk; e0 += kThreads * 8) {
            const int cnt = sk - e0 < 8 ? (int)(sk - e0) : 8;
            const int nv = valid - e0 <= 0 ? 0 : (valid - e0 < 8 ? (int)(valid - e0) : 8);
            float gv[8], yv[8], o[8];
            if (nv > 0) {
                load8f(dy + base + e0, vec, nv, gv);
                load8f(y + base + e0, vec, nv, yv);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o[j] = j < nv ? __fmul_rn(__fmul_rn(scale, yv[j]), __fsub_rn(gv[j], s)) : 0.0f;
            store8f(dx + base + e0, vec, cnt, o);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
constexpr int kC = MFX_SOFTMAX_C;
constexpr int64_t kMaxTeamChunks = (int64_t)kC * kThreads;

// Team width 2^lg for rows of G chunks: the smallest power of two with
// C * 2^lg >= G; -1 when the row needs the long kernel.
int team_lg(int64_t G)
{
    if (G > kMaxTeamChunks)
        return -1;
    int lg = 0;
    while ((int64_t)kC << lg < G)
        ++lg;
    return lg;
}

template <typename K>
void team_launch_dims(K kernel, int64_t rows, int lg, unsigned* blocks, int64_t* iters)
{
    const int teams = kThreads >> lg;
    const int64_t need = (rows + teams - 1) / teams;
    const int64_t cap = (int64_t)sm_count() * blocks_per_sm((const void*)kernel);
    const int64_t nb = need < cap ? need : cap;
    *blocks = (unsigned)(nb > 0 ? nb : 1);
    *iters = (need + *blocks - 1) / *blocks;
}

unsigned long_blocks(const void* kernel, int64_t rows)
{
    const int64_t cap = (int64_t)sm_count() * blocks_per_sm(kernel);
    return (unsigned)(rows < cap ? rows : cap);
}

template <typename T, bool MASK, bool CAUSAL>
int launch_fwd(const SoftmaxGeom& g, const void* x, const void* mask, void* y, float scale, cudaStream_t s)
{
    const T* xp = static_cast<const T*>(x);
    const T* mp = static_cast<const T*>(mask);
    T* yp = static_cast<T*>(y);
    const bool vec = g.sk % 8 == 0 && aligned16(x) && aligned16(y) && (!MASK || aligned16(mask));
    const int lg = team_lg((g.sk + 7) / 8);
    if (lg >= 0) {
        auto k = softmax_fwd_team<T, kC, MASK, CAUSAL>;
        unsigned blocks;
        int64_t iters;
        team_launch_dims(k, g.rows, lg, &blocks, &iters);
        k<<<blocks, kThreads, 0, s>>>(xp, mp, yp, g, scale, lg, iters, vec);
        return launch_status();
    }
    auto k = softmax_fwd_long<T, MASK, CAUSAL>;
    k<<<long_blocks((const void*)k, g.rows), kThreads, 0, s>>>(xp, mp, yp, g, scale, vec);
    return launch_status();
}

template <typename T, bool CAUSAL>
int launch_bwd(int64_t rows, int64_t sk, const void* dy, const void* y, void* dx, float scale, cudaStream_t s)
{
    const T* gp = static_cast<const T*>(dy);
    const T* yp = static_cast<const T*>(y);
    T* dp = static_cast<T*>(dx);
    const bool vec = sk % 8 == 0 && aligned16(dy) && aligned16(y) && aligned16(dx);
    const int lg = team_lg((sk + 7) / 8);
    if (lg >= 0) {
        auto k = softmax_bwd_team<T, kC, CAUSAL>;
        unsigned blocks;
        int64_t iters;
        team_launch_dims(k, rows, lg, &blocks, &iters);
        k<<<blocks, kThreads, 0, s>>>(gp, yp, dp, rows, sk, scale, lg, iters, vec);
        return launch_status();
    }
    auto k = softmax_bwd_long<T, CAUSAL>;
    k<<<long_blocks((const void*)k, rows), kThreads, 0, s>>>(gp, yp, dp, rows, sk, scale, vec);
    return launch_status();
}

template <typename T>
int dispatch_fwd(const SoftmaxGeom& g, const void* x, const void* mask, bool causal, void* y, float scale,
                 cudaStream_t s)
{
    if (causal)
        return launch_fwd<T, false, true>(g, x, nullptr, y, scale, s);
    if (mask)
        return launch_fwd<T, true, false>(g, x, mask, y, scale, s);
    return launch_fwd<T, false, false>(g, x, nullptr, y, scale, s);
}

int check_sizes(int dt, std::initializer_list<int64_t> dims, int64_t* n_out)
{
    *n_out = 0;
    if (!valid_dtype(dt))
        return MFX_ERR_DTYPE;
    int64_t n = 1;
    for (int64_t d : dims) {
        if (d < 0)
            return MFX_ERR_SHAPE;
        if (!mul_ok(n, d, &n))
            return MFX_ERR_SHAPE;
    }
    int64_t bytes = 0;
    if (!mul_ok(n, 16, &bytes))
        return MFX_ERR_SHAPE;
    *n_out = n;
    return MFX_OK;
}

int bwd_entry(int dt, int64_t rows, int64_t sk, const void* dy, const void* y, float scale, void* dx, bool causal,
              void* stream)
{
    int64_t n = 0;
    const int st = check_sizes(dt, {rows, sk}, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!dy || !y || !dx)
        return MFX_ERR_NULL;
    const int64_t b = n * dtype_bytes(dt);
    if (partial_overlap(dy, b, dx, b) || partial_overlap(y, b, dx, b))
        return MFX_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == MFX_BF16)
        return causal ? launch_bwd<bf16, true>(rows, sk, dy, y, dx, scale, s)
                      : launch_bwd<bf16, false>(rows, sk, dy, y, dx, scale, s);
    return causal ? launch_bwd<float, true>(rows, sk, dy, y, dx, scale, s)
                  : launch_bwd<float, false>(rows, sk, dy, y, dx, scale, s);
}

}  // namespace
}  // namespace mfx

extern "C" int mfx_scaled_masked_softmax_fwd(int dt, int64_t b, int64_t np, int64_t sq, int64_t sk, const void* x,
                                             const void* mask, int64_t mask_b, int64_t mask_np, int64_t mask_sq,
                                             float scale, void* y, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check_sizes(dt, {b, np, sq, sk}, &n);
    if (st != MFX_OK)
        return st;
    if (mask && ((mask_b != 1 && mask_b != b) || (mask_np != 1 && mask_np != np) ||
                 (mask_sq != 1 && mask_sq != sq)))
        return MFX_ERR_SHAPE;
    if (n == 0)
        return MFX_OK;
    if (!x || !y)
        return MFX_ERR_NULL;
    const int64_t bytes = n * dtype_bytes(dt);
    int64_t mbytes = 0;
    if (mask) {
        // each mask size is 1 or the input's, so the mask is no larger than x
        mbytes = mask_b * mask_np * mask_sq * sk * dtype_bytes(dt);
    }
    if (partial_overlap(x, bytes, y, bytes) || overlaps(mask, mbytes, y, bytes))
        return MFX_ERR_ALIAS;
    const SoftmaxGeom g{b * np * sq, sq, np, sk, mask ? mask_b : 1, mask ? mask_np : 1, mask ? mask_sq : 1};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == MFX_BF16 ? dispatch_fwd<bf16>(g, x, mask, false, y, scale, s)
                          : dispatch_fwd<float>(g, x, mask, false, y, scale, s);
}

extern "C" int mfx_scaled_upper_triang_masked_softmax_fwd(int dt, int64_t attn_batches, int64_t sq, const void* x,
                                                          float scale, void* y, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check_sizes(dt, {attn_batches, sq, sq}, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!x || !y)
        return MFX_ERR_NULL;
    const int64_t bytes = n * dtype_bytes(dt);
    if (partial_overlap(x, bytes, y, bytes))
        return MFX_ERR_ALIAS;
    const SoftmaxGeom g{attn_batches * sq, sq, 1, sq, 1, 1, 1};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == MFX_BF16 ? dispatch_fwd<bf16>(g, x, nullptr, true, y, scale, s)
                          : dispatch_fwd<float>(g, x, nullptr, true, y, scale, s);
}

extern "C" int mfx_scaled_masked_softmax_bwd(int dt, int64_t rows, int64_t sk, const void* dy, const void* y,
                                             float scale, void* dx, void* stream)
{
    return mfx::bwd_entry(dt, rows, sk, dy, y, scale, dx, false, stream);
}

extern "C" int mfx_scaled_upper_triang_masked_softmax_bwd(int dt, int64_t attn_batches, int64_t sq, const void* dy,
                                                          const void* y, float scale, void* dx, void* stream)
{
    int64_t rows = 0;
    if (attn_batches < 0 || sq < 0 || !mfx::mul_ok(attn_batches, sq, &rows))
        return MFX_ERR_SHAPE;
    return mfx::bwd_entry(dt, rows, sq, dy, y, scale, dx, true, stream);
}
