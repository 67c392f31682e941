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
// Layout: rows of sk contiguous elements, one softmax per row, in three
// regimes by row length G = ceil(sk / 8) chunks of 8 elements:
//  - G < 64: a "team" of 1 .. 16 lanes owns a row in registers (4 chunks per
//    lane) and reduces with shuffles (softmax_*_team);
//  - 64 <= G <= 2048: one warp per row (softmax_*_warp, softmax_*_rowpipe):
//    the forward makes three passes over the row (maximum, sum, output), the
//    backward two; aligned rows come through a shared-memory row ring filled
//    by bulk copies (the causal backward's rows in pairs q, sq - 1 - q, so
//    that every stage is full), unaligned ones straight from global memory;
//  - longer rows: one block per row, three passes (softmax_*_long), the
//    later reads hitting L2.
// Each regime runs the same code whatever the source of the row, so aligned
// and unaligned calls give the same bits.
//
// Accuracy: the exponent of each element is formed with x * scale + (mask -
// max) in one fused multiply-add, so large scores lose nothing to the
// rounding of x * scale; the row maximum only shifts every exponent by the
// same amount.  Row sums are per-chunk trees combined with the compensated
// summation of Ogita, Rump and Oishi ("Accurate sum and dot product", SIAM
// J. Sci. Comput. 26(6), 2005: Knuth's TwoSum per addition, the rounding
// errors summed alongside); the backward's row sum of dy * y adds the
// rounded products the same way, so dy_k - sum keeps its accuracy where the
// two nearly cancel.  The exponentials: see the bf16 and fp32 warp-row
// forwards (the team and long kernels use expf in fp32).
#include <initializer_list>

#include "mfx_device.cuh"
#include "mfx_host.h"
#include "mfx_pipe.cuh"

#ifndef MFX_SOFTMAX_C
#define MFX_SOFTMAX_C 4  // chunks of 8 elements per thread in the register kernels
#endif
#ifndef MFX_MINB_SOFTMAX
#define MFX_MINB_SOFTMAX 2
#endif
#ifndef MFX_PIPE_SOFTMAX
#define MFX_PIPE_SOFTMAX 1      // aligned warp-per-row rows through the bulk-copy pipeline
#endif
#ifndef MFX_RING_KB_SOFTMAX
#define MFX_RING_KB_SOFTMAX 96  // shared-memory ring of a forward row-pipeline block (KB; two blocks per SM)
#endif
#ifndef MFX_RING_KB_SOFTMAX_BWD
#define MFX_RING_KB_SOFTMAX_BWD 64  // the same for the backward (fewer bytes in flight measured faster)
#endif
#ifndef MFX_SOFTMAX_PAIR_RPS
#define MFX_SOFTMAX_PAIR_RPS 8  // most causal row pairs per ring stage
#endif
#ifndef MFX_SOFTMAX_PAIRS_FWD
#define MFX_SOFTMAX_PAIRS_FWD 0 // causal forward pipeline moves row pairs (0: single rows)
#endif
#ifndef MFX_SOFTMAX_PAIRS_BWD
#define MFX_SOFTMAX_PAIRS_BWD 1 // causal backward pipeline moves row pairs (0: single rows)
#endif

namespace mfx {
namespace {

__device__ unsigned g_device_error;

constexpr int kWarps = kThreads / 32;
constexpr int kC_ = MFX_SOFTMAX_C;  // chunks of 8 elements per thread
static_assert(MFX_SOFTMAX_PAIR_RPS == 1 || MFX_SOFTMAX_PAIR_RPS == 2 || MFX_SOFTMAX_PAIR_RPS == 4 ||
                  MFX_SOFTMAX_PAIR_RPS == 8,
              "units per stage must divide the 8 consumer warps");

// ---------------------------------------------------------------------------
// Compensated summation (Knuth's TwoSum per addition).
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
// Unsigned 32-bit division by an invariant divisor as a multiply-high, add
// and shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, the round-up method of their section 4):
// with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (mulhi(m, n) + n) >> l for every 32-bit n.
struct Div32 {
    uint32_t d, m, l;
    __device__ __forceinline__ uint32_t div(uint32_t n) const
    {
        return (uint32_t)(((uint64_t)__umulhi(m, n) + n) >> l);
    }
};

inline Div32 make_div32(uint32_t d)
{
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d)
        ++l;
    const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return Div32{d, (uint32_t)m, l};
}

struct SoftmaxGeom {
    int64_t rows;          // b * np * sq
    int64_t sq, np, sk;    // query rows per (batch, head), heads, row length
    int64_t mb, mnp, msq;  // mask sizes (each 1 = broadcast, or the input's)
    Div32 dsq, dnp;        // division by sq and np (row indices below 2^32)
};

// Offset of the mask row that applies to input row r (64-bit arithmetic).
__device__ __forceinline__ int64_t mask_row(const SoftmaxGeom& g, int64_t r)
{
    const int64_t q = r % g.sq, bh = r / g.sq;
    const int64_t h = bh % g.np, i = bh / g.np;
    return (((g.mb == 1 ? 0 : i) * g.mnp + (g.mnp == 1 ? 0 : h)) * g.msq + (g.msq == 1 ? 0 : q)) * g.sk;
}

// The same for row indices below 2^32 (the team and pipelined kernels).
__device__ __forceinline__ int64_t mask_row32(const SoftmaxGeom& g, uint32_t r)
{
    const uint32_t bh = g.dsq.div(r), q = r - bh * (uint32_t)g.sq;
    const uint32_t i = g.dnp.div(bh), h = bh - i * (uint32_t)g.np;
    return (((g.mb == 1 ? 0 : (int64_t)i) * g.mnp + (g.mnp == 1 ? 0 : h)) * g.msq + (g.msq == 1 ? 0 : q)) * g.sk;
}

// Query index of row r (causal rows: r mod sq), for r below 2^32.
__device__ __forceinline__ int64_t query32(const SoftmaxGeom& g, uint32_t r)
{
    return r - g.dsq.div(r) * (uint32_t)g.sq;
}

// e^d for d <= 0 (or NaN) in the precise (fp32) tier.  The bf16 tier returns
// 2^64 e^d from the hardware base-2 exponential at d log2(e) + 64: the factor
// 2^64 is common to every term of the row sum and cancels in e / sum, and it
// keeps results down to 2^-190 clear of the hardware's flush to zero.
template <bool PRECISE>
__device__ __forceinline__ float exp_row(float d)
{
    if (PRECISE)
        return expf(d);
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(fmaf(d, (float)kLog2e, 64.0f)));
    return r;
}

// Sum of one chunk of 8 as a fixed tree.
__device__ __forceinline__ float sum8(const float (&v)[8])
{
    return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

// ---------------------------------------------------------------------------
// Per-row arithmetic shared by the register and the pipelined kernels, so
// that both give the same bits.  A thread holds C chunks of 8 elements of
// its row: chunk c covers elements (t + c * tpr) * 8 .. + 7 of which the
// first n[c] are valid (0 <= n[c] <= 8; the loaders set the others to 0).
// Sums: a fixed tree over each chunk, the chunks and then the team's threads
// combined with TwoSum, so a row sum's error stays a few units of roundoff of
// the sum of its terms' magnitudes whatever the row length.
// ---------------------------------------------------------------------------
template <int C, bool MASK, int MB>
__device__ __forceinline__ float row_max(const float (&a)[C][8], const float (&b)[MB][8], const int (&n)[C],
                                         float scale)
{
    if (MASK) {
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            if (n[c] == 8) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    m = fmaxf(m, fmaf(a[c][j], scale, b[MASK ? c : 0][j]));
            } else if (n[c] > 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < n[c])
                        m = fmaxf(m, fmaf(a[c][j], scale, b[MASK ? c : 0][j]));
            }
        }
        return m;
    }
    // max_k fl(x_k scale) = fl(max_k x_k scale) for scale >= 0 (rounding is
    // monotone), and the same with the minimum for scale < 0
    const float sg = scale < 0.0f ? -1.0f : 1.0f;
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < C; ++c) {
        if (n[c] == 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                mx = fmaxf(mx, sg * a[c][j]);
        } else if (n[c] > 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n[c])
                    mx = fmaxf(mx, sg * a[c][j]);
        }
    }
    return mx == -INFINITY ? -INFINITY : (sg * mx) * scale;
}

// a <- exponentials of the scores shifted by -max (0 past n[c]); returns the
// row partial sum in `s` (bf16 tier) or `acc` (fp32 tier).
template <bool PRECISE, int C, bool MASK, int MB>
__device__ __forceinline__ void row_exp(float (&a)[C][8], const float (&b)[MB][8], const int (&n)[C], float scale,
                                        float mneg, float& s, Acc& acc)
{
#pragma unroll
    for (int c = 0; c < C; ++c) {
        if (n[c] == 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                a[c][j] = exp_row<PRECISE>(fmaf(a[c][j], scale, MASK ? b[MASK ? c : 0][j] + mneg : mneg));
        } else if (n[c] > 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                a[c][j] = j < n[c] ? exp_row<PRECISE>(fmaf(a[c][j], scale, MASK ? b[MASK ? c : 0][j] + mneg : mneg))
                                   : 0.0f;
        }
        if (n[c] > 0) {
            if (PRECISE)
                two_sum_add(acc, sum8(a[c]));
            else
                s += sum8(a[c]);
        }
    }
}

// Output chunk c: the normalised exponentials, exact zeros past n[c] and for
// a row with nothing left.
template <int C>
__device__ __forceinline__ void row_out(const float (&a)[C][8], const int (&n)[C], int c, float rs, bool none,
                                        float (&o)[8])
{
    if (n[c] == 8 && !none) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = a[c][j] * rs;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = j < n[c] && !none ? a[c][j] * rs : 0.0f;
    }
}

// Row partial of sum_k dy_k y_k (chunks zero past n[c]).
template <int C>
__device__ __forceinline__ Acc row_dot(const float (&gv)[C][8], const float (&yv)[C][8], const int (&n)[C])
{
    Acc acc{0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < C; ++c) {
        if (n[c] > 0) {
            float p[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                p[j] = gv[c][j] * yv[c][j];
            two_sum_add(acc, sum8(p));
        }
    }
    return acc;
}

template <int C>
__device__ __forceinline__ void row_dx(const float (&gv)[C][8], const float (&yv)[C][8], const int (&n)[C], int c,
                                       float scale, float s, float (&o)[8])
{
    if (n[c] == 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = (scale * yv[c][j]) * (gv[c][j] - s);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = j < n[c] ? (scale * yv[c][j]) * (gv[c][j] - s) : 0.0f;
    }
}

// Valid elements of chunk c (first element e0) in a row whose first `valid`
// elements take part.
__device__ __forceinline__ int chunk_count(int64_t valid, int e0)
{
    const int64_t left = valid - e0;
    return left <= 0 ? 0 : (left < 8 ? (int)left : 8);
}

// The forward's reductions and output for one row held by a team.
template <typename T, int C, bool MASK, int MB>
__device__ __forceinline__ void fwd_row_finish(float (&a)[C][8], const float (&b)[MB][8], const int (&n)[C],
                                               float scale, int lg, int tm, int t, float (*red_s)[kWarps],
                                               float (*red_c)[kWarps], bool active, T* yr, int64_t sk, bool vec)
{
    constexpr bool kPrecise = !DTypeInfo<T>::kBf16;
    const int tpr = 1 << lg;
    float m = row_max<C, MASK, MB>(a, b, n, scale);
    m = team_max(m, lg, tm, red_s, 0);
    const bool none = m == -INFINITY;  // a row with no finite score left: all zeros
    const float mneg = none ? 0.0f : -m;
    Acc acc{0.0f, 0.0f};
    float s = 0.0f;
    row_exp<kPrecise, C, MASK, MB>(a, b, n, scale, mneg, s, acc);
    const float sum = kPrecise ? acc_value(team_acc(acc, lg, tm, red_s, red_c, 1)) : team_sum(s, lg, tm, red_s, 1);
    const float rs = __frcp_rn(sum);
    if (active) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int e0 = (t + c * tpr) * 8;
            if (e0 < sk) {
                float o[8];
                row_out<C>(a, n, c, rs, none, o);
                store8f(yr + e0, vec, sk - e0 < 8 ? (int)(sk - e0) : 8, o);
            }
        }
    }
}

template <typename T, int C>
__device__ __forceinline__ void bwd_row_finish(const float (&gv)[C][8], const float (&yv)[C][8], const int (&n)[C],
                                               float scale, int lg, int tm, int t, float (*red_s)[kWarps],
                                               float (*red_c)[kWarps], int slot, bool active, T* dxr, int64_t sk,
                                               bool vec)
{
    const int tpr = 1 << lg;
    const float s = acc_value(team_acc(row_dot<C>(gv, yv, n), lg, tm, red_s, red_c, slot));
    if (active) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int e0 = (t + c * tpr) * 8;
            if (e0 < sk) {
                float o[8];
                row_dx<C>(gv, yv, n, c, scale, s, o);
                store8f(dxr + e0, vec, sk - e0 < 8 ? (int)(sk - e0) : 8, o);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// bf16 rows.  Raw bf16 pairs stay packed until they are needed in fp32: the
// row maximum of the scores without a mask is taken on the packed pairs
// (max.bf16x2: a NaN operand yields the other, as fmaxf does), and the fp32
// arithmetic runs on pairs (the .f32x2 forms of add, mul and fma), each pair
// rounded exactly as two scalar operations would be.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float ex2_ftz(float t)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}


// One chunk of 8 bf16 as four packed pairs, from global memory (16-byte
// vector when `vec` and the chunk is full, else element by element with
// zeros past n) or from shared memory.
__device__ __forceinline__ void load_words(const bf16* p, bool vec, int n, uint32_t (&w)[4])
{
    if (vec && n == 8) {
        const uint4 v = ld16(p);
        w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = 2 * k < n ? p[2 * k].bits : 0u;
            const uint32_t hi = 2 * k + 1 < n ? p[2 * k + 1].bits : 0u;
            w[k] = lo | hi << 16;
        }
    }
}

// Zero the elements of a chunk of words past its count.
__device__ __forceinline__ void zero_tail_words(uint32_t (&w)[4], int cnt)
{
    if (cnt < 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (2 * k >= cnt)
                w[k] &= 0xFFFF0000u;
            if (2 * k + 1 >= cnt)
                w[k] &= 0x0000FFFFu;
        }
    }
}

// Element j of a chunk of packed words, in fp32.
__device__ __forceinline__ float word_elem(const uint32_t (&w)[4], int j)
{
    return __uint_as_float(j & 1 ? w[j >> 1] & 0xFFFF0000u : w[j >> 1] << 16);
}

// Forward of one bf16 row held by a team: C chunks of packed x (and mask).
// The exponent of element j is t_j = (z_j - M) log2(e) + 64 with z_j = x_j
// scale (+ mask_j) and M the row maximum; for |M| <= 64 it is formed as one
// fused multiply-add x_j (scale log2 e) + (64 - M log2 e) (+ mask_j log2 e),
// whose roundings stay below 2^-17 of the result's relative accuracy, and for
// larger |M| as ((x_j scale + mask_j) - M) log2 e + 64, exact in the shift
// by M.  e_j = 2^t_j carries the factor 2^64 common to the row sum.
template <int C, bool MASK, int MB>
__device__ __forceinline__ void fwd_row_fast(const uint32_t (&xw)[C][4], const uint32_t (&mw)[MB][4], const int (&n)[C],
                                             float scale, int lg, int tm, int t, float (*red_s)[kWarps], bool active,
                                             bf16* yr, int64_t sk, bool vec)
{
    const int tpr = 1 << lg;
    const float kL2e = (float)kLog2e;
    // 1) the thread's maximum score
    float m = -INFINITY;
    if (!MASK) {
        const bool neg = scale < 0.0f;
        uint32_t acc = neg ? 0x7F807F80u : 0xFF80FF80u;  // (+inf, +inf) / (-inf, -inf)
        float part = neg ? INFINITY : -INFINITY;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            if (n[c] == 8) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    acc = neg ? bmin2(acc, xw[c][k]) : bmax2(acc, xw[c][k]);
            } else if (n[c] > 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < n[c])
                        part = neg ? fminf(part, word_elem(xw[c], j)) : fmaxf(part, word_elem(xw[c], j));
            }
        }
        const float2 h = widen2(acc);
        const float xm = neg ? fminf(fminf(h.x, h.y), part) : fmaxf(fmaxf(h.x, h.y), part);
        if (n[0] > 0)
            m = xm * scale;
    } else {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            if (n[c] == 8) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 z = fma2(widen2(xw[c][k]), f2(scale), widen2(mw[MASK ? c : 0][k]));
                    m = fmaxf(m, fmaxf(z.x, z.y));
                }
            } else if (n[c] > 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < n[c])
                        m = fmaxf(m, fmaf(word_elem(xw[c], j), scale, word_elem(mw[MASK ? c : 0], j)));
            }
        }
    }
    m = team_max(m, lg, tm, red_s, 0);
    const bool none = m == -INFINITY;
    // 2) exponentials and the row sum
    const bool near = fabsf(m) <= 64.0f;
    const float2 sL = f2(scale * kL2e);
    const float2 cL = f2(fmaf(-m, kL2e, 64.0f));
    float2 e[C][4];
    float2 s2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int c = 0; c < C; ++c) {
        if (n[c] > 0 && !none) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = widen2(xw[c][k]);
                float2 tt;
                if (near) {
                    const float2 base = MASK ? fma2(widen2(mw[MASK ? c : 0][k]), f2(kL2e), cL) : cL;
                    tt = fma2(x, sL, base);
                } else {
                    const float2 d = MASK ? fma2(x, f2(scale), add2(widen2(mw[MASK ? c : 0][k]), f2(-m)))
                                          : fma2(x, f2(scale), f2(-m));
                    tt = fma2(d, f2(kL2e), f2(64.0f));
                }
                e[c][k] = make_float2(ex2_ftz(tt.x), ex2_ftz(tt.y));
            }
            if (n[c] < 8) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j >= n[c])
                        (j & 1 ? e[c][j >> 1].y : e[c][j >> 1].x) = 0.0f;
            }
            s2 = add2(s2, add2(add2(e[c][0], e[c][1]), add2(e[c][2], e[c][3])));
        }
    }
    const float sum = team_sum(s2.x + s2.y, lg, tm, red_s, 1);
    // 3) normalise and store
    const float2 rs = f2(__frcp_rn(sum));
    if (active) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int e0 = (t + c * tpr) * 8;
            if (e0 < sk) {
                uint4 o = make_uint4(0u, 0u, 0u, 0u);
                if (n[c] > 0 && !none) {
                    const float2 y0 = mul2(e[c][0], rs), y1 = mul2(e[c][1], rs);
                    const float2 y2 = mul2(e[c][2], rs), y3 = mul2(e[c][3], rs);
                    o = make_uint4(pack_bf16x2(y0.x, y0.y), pack_bf16x2(y1.x, y1.y), pack_bf16x2(y2.x, y2.y),
                                   pack_bf16x2(y3.x, y3.y));
                }
                if (vec && sk - e0 >= 8) {
                    st16(yr + e0, o);
                } else {
                    const int cnt = sk - e0 < 8 ? (int)(sk - e0) : 8;
                    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
                    for (int j = 0; j < cnt; ++j)
                        yr[e0 + j].bits = (uint16_t)(j & 1 ? ow[j >> 1] >> 16 : ow[j >> 1] & 0xFFFFu);
                }
            }
        }
    }
}

// Backward of one bf16 row: s = sum_k dy_k y_k (products exact in fp32;
// chunk trees of pairs, chunks and threads combined with TwoSum), then
// dx = (scale y)(dy - s).
template <int C>
__device__ __forceinline__ void bwd_row_fast(const uint32_t (&gw)[C][4], const uint32_t (&yw)[C][4], const int (&n)[C],
                                             float scale, int lg, int tm, int t, float (*red_s)[kWarps],
                                             float (*red_c)[kWarps], int slot, bool active, bf16* dxr, int64_t sk,
                                             bool vec)
{
    const int tpr = 1 << lg;
    Acc acc{0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < C; ++c) {
        if (n[c] > 0) {
            const float2 p0 = mul2(widen2(gw[c][0]), widen2(yw[c][0]));
            const float2 p1 = mul2(widen2(gw[c][1]), widen2(yw[c][1]));
            const float2 p2 = mul2(widen2(gw[c][2]), widen2(yw[c][2]));
            const float2 p3 = mul2(widen2(gw[c][3]), widen2(yw[c][3]));
            const float2 q = add2(add2(p0, p1), add2(p2, p3));
            two_sum_add(acc, q.x + q.y);
        }
    }
    const float s = acc_value(team_acc(acc, lg, tm, red_s, red_c, slot));
    if (active) {
        const float2 ms = f2(-s), sc = f2(scale);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int e0 = (t + c * tpr) * 8;
            if (e0 < sk) {
                uint32_t ow[4] = {0u, 0u, 0u, 0u};
                if (n[c] > 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 d = mul2(mul2(sc, widen2(yw[c][k])), add2(widen2(gw[c][k]), ms));
                        ow[k] = pack_bf16x2(d.x, d.y);
                    }
                    if (n[c] < 8) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (2 * k >= n[c])
                                ow[k] &= 0xFFFF0000u;
                            if (2 * k + 1 >= n[c])
                                ow[k] &= 0x0000FFFFu;
                        }
                    }
                }
                if (vec && sk - e0 >= 8) {
                    st16(dxr + e0, make_uint4(ow[0], ow[1], ow[2], ow[3]));
                } else {
                    const int cnt = sk - e0 < 8 ? (int)(sk - e0) : 8;
                    for (int j = 0; j < cnt; ++j)
                        dxr[e0 + j].bits = (uint16_t)(j & 1 ? ow[j >> 1] >> 16 : ow[j >> 1] & 0xFFFFu);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Register kernels: each team loads its row from global memory.
// ---------------------------------------------------------------------------
template <typename T, int C, bool MASK, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, MFX_MINB_SOFTMAX)
softmax_fwd_team(const T* x, const T* __restrict__ mask, T* y, SoftmaxGeom g, float scale, int lg, int64_t iters,
                 bool vec)
{
    constexpr int MB = MASK ? C : 1;
    __shared__ float red_s[2][kWarps], red_c[2][kWarps];
    const int tpr = 1 << lg;
    const int tm = threadIdx.x >> lg, t = threadIdx.x & (tpr - 1);
    const int teams = kThreads >> lg;
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = ((int64_t)blockIdx.x + it * gridDim.x) * teams + tm;
        const bool active = r < g.rows;
        const int64_t valid = active ? (CAUSAL ? query32(g, (uint32_t)r) + 1 : g.sk) : 0;
        const T* xr = x + (active ? r : 0) * g.sk;
        const T* mr = MASK ? mask + (active ? mask_row32(g, (uint32_t)r) : 0) : nullptr;
        int n[C];
#pragma unroll
        for (int c = 0; c < C; ++c)
            n[c] = chunk_count(valid, (t + c * tpr) * 8);
        if constexpr (DTypeInfo<T>::kBf16) {
            uint32_t xw[C][4], mw[MB][4];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int e0 = (t + c * tpr) * 8;
                if (n[c] > 0) {
                    load_words(xr + e0, vec, n[c], xw[c]);
                    if (MASK)
                        load_words(mr + e0, vec, n[c], mw[MASK ? c : 0]);
                }
            }
            fwd_row_fast<C, MASK, MB>(xw, mw, n, scale, lg, tm, t, red_s, active, y + (active ? r : 0) * g.sk, g.sk,
                                      vec);
        } else {
            float a[C][8], b[MB][8];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int e0 = (t + c * tpr) * 8;
                if (n[c] > 0) {
                    load8f(xr + e0, vec, n[c], a[c]);
                    if (MASK)
                        load8f(mr + e0, vec, n[c], b[MASK ? c : 0]);
                }
            }
            fwd_row_finish<T, C, MASK, MB>(a, b, n, scale, lg, tm, t, red_s, red_c, active,
                                           y + (active ? r : 0) * g.sk, g.sk, vec);
        }
    }
}

template <typename T, int C, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, MFX_MINB_SOFTMAX)
softmax_bwd_team(const T* dy, const T* y, T* dx, int64_t rows, int64_t sk, Div32 dsk, float scale, int lg,
                 int64_t iters, bool vec)
{
    __shared__ float red_s[2][kWarps], red_c[2][kWarps];
    const int tpr = 1 << lg;
    const int tm = threadIdx.x >> lg, t = threadIdx.x & (tpr - 1);
    const int teams = kThreads >> lg;
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = ((int64_t)blockIdx.x + it * gridDim.x) * teams + tm;
        const bool active = r < rows;
        const int64_t valid = active ? (CAUSAL ? (uint32_t)r - dsk.div((uint32_t)r) * (uint32_t)sk + 1 : sk) : 0;
        const int64_t base = (active ? r : 0) * sk;
        int n[C];
#pragma unroll
        for (int c = 0; c < C; ++c)
            n[c] = chunk_count(valid, (t + c * tpr) * 8);
        if constexpr (DTypeInfo<T>::kBf16) {
            uint32_t gw[C][4], yw[C][4];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int e0 = (t + c * tpr) * 8;
                if (n[c] > 0) {
                    load_words(dy + base + e0, vec, n[c], gw[c]);
                    load_words(y + base + e0, vec, n[c], yw[c]);
                }
            }
            bwd_row_fast<C>(gw, yw, n, scale, lg, tm, t, red_s, red_c, (int)(it & 1), active, dx + base, sk, vec);
        } else {
            float gv[C][8], yv[C][8];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int e0 = (t + c * tpr) * 8;
                if (n[c] > 0) {
                    load8f(dy + base + e0, vec, n[c], gv[c]);
                    load8f(y + base + e0, vec, n[c], yv[c]);
                }
            }
            bwd_row_finish<T, C>(gv, yv, n, scale, lg, tm, t, red_s, red_c, (int)(it & 1), active, dx + base, sk,
                                 vec);
        }
    }
}

// ---------------------------------------------------------------------------
// Long rows: one block per row; the forward reads the row three times (max,
// sum, output), the backward twice; the later reads hit L2.  Same chunk
// arithmetic, with the chunks of a thread at stride 256 x 8.
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
            float a[1][8], b[1][8];
            int n[1] = {chunk_count(valid - e0, 0)};
            load8f(xr + e0, vec, n[0], a[0]);
            if (MASK)
                load8f(mr + e0, vec, n[0], b[0]);
            m = fmaxf(m, row_max<1, MASK, 1>(a, b, n, scale));
        }
        m = team_max(m, 8, 0, red_s, 0);
        const bool none = m == -INFINITY;
        const float mneg = none ? 0.0f : -m;
        Acc acc{0.0f, 0.0f};
        float s = 0.0f;
        for (int64_t e0 = (int64_t)t * 8; e0 < valid; e0 += kThreads * 8) {
            float a[1][8], b[1][8];
            int n[1] = {chunk_count(valid - e0, 0)};
            load8f(xr + e0, vec, n[0], a[0]);
            if (MASK)
                load8f(mr + e0, vec, n[0], b[0]);
            row_exp<kPrecise, 1, MASK, 1>(a, b, n, scale, mneg, s, acc);
        }
        const float sum = kPrecise ? acc_value(team_acc(acc, 8, 0, red_s, red_c, 1)) : team_sum(s, 8, 0, red_s, 1);
        const float rs = __frcp_rn(sum);
        for (int64_t e0 = (int64_t)t * 8; e0 < g.sk; e0 += kThreads * 8) {
            float a[1][8], b[1][8], o[8];
            int n[1] = {chunk_count(valid - e0, 0)};
            if (n[0] > 0) {
                load8f(xr + e0, vec, n[0], a[0]);
                if (MASK)
                    load8f(mr + e0, vec, n[0], b[0]);
                float s2 = 0.0f;
                Acc a2{0.0f, 0.0f};
                row_exp<kPrecise, 1, MASK, 1>(a, b, n, scale, mneg, s2, a2);
            }
            row_out<1>(a, n, 0, rs, none, o);
            store8f(y + r * g.sk + e0, vec, g.sk - e0 < 8 ? (int)(g.sk - e0) : 8, o);
        }
    }
}

template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
softmax_bwd_long(const T* dy, const T* y, T* dx, int64_t rows, int64_t sk, float scale, bool vec)
{
    __shared__ float red_s[2][kWarps], red_c[2][kWarps];
    const int t = threadIdx.x;
    int parity = 0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, parity ^= 1) {
        const int64_t valid = CAUSAL ? r % sk + 1 : sk;
        const int64_t base = r * sk;
        Acc acc{0.0f, 0.0f};
        for (int64_t e0 = (int64_t)t * 8; e0 < valid; e0 += kThreads * 8) {
            float gv[1][8], yv[1][8];
            int n[1] = {chunk_count(valid - e0, 0)};
            load8f(dy + base + e0, vec, n[0], gv[0]);
            load8f(y + base + e0, vec, n[0], yv[0]);
            acc = acc_merge(acc, row_dot<1>(gv, yv, n));
        }
        const float s = acc_value(team_acc(acc, 8, 0, red_s, red_c, parity));
        for (int64_t e0 = (int64_t)t * 8; e0 < sk; e0 += kThreads * 8) {
            float gv[1][8], yv[1][8], o[8];
            int n[1] = {chunk_count(valid - e0, 0)};
            if (n[0] > 0) {
                load8f(dy + base + e0, vec, n[0], gv[0]);
                load8f(y + base + e0, vec, n[0], yv[0]);
            }
            row_dx<1>(gv, yv, n, 0, scale, s, o);
            store8f(dx + base + e0, vec, sk - e0 < 8 ? (int)(sk - e0) : 8, o);
        }
    }
}

constexpr int kMaxStages = 8;  // the ring header holds 8 full and 8 empty barriers

// ---------------------------------------------------------------------------
// Warp-per-row kernels (rows of 64 .. 2048 chunks of 8).  One warp owns a
// row: lane l takes chunks l, l + 32, ...; the row is read three times in
// the forward (maximum, sum of exponentials, output) and twice in the
// backward (row sum of dy * y, output), and every reduction is a warp
// shuffle tree, so a row costs no block barrier and little per-row work.
// The pipelined form reads the row from a shared-memory stage that a
// producer warp filled with bulk copies (one copy per stage of consecutive
// rows; the causal form copies each row's first q + 1 elements rounded up to
// 8); the direct form, for unaligned buffers, reads global memory (the
// second and third reads hit L2).  Both run the same per-row code, so they
// give the same bits.
// ---------------------------------------------------------------------------
template <typename T>
struct ChunkT;
template <>
struct ChunkT<bf16> {
    uint32_t w[4];
};
template <>
struct ChunkT<float> {
    float f[8];
};

// Sources of a row's chunks: a shared-memory stage (16-byte aligned rows,
// sk a multiple of 8) or global memory (any alignment).
template <typename T>
struct SmemRow {
    static constexpr bool kKeeps = true;  // the fp32 forward may park e^d in the stage
    const unsigned char* x;
    const unsigned char* m;
    __device__ __forceinline__ void chunk(const unsigned char* base, int i, int, ChunkT<T>& c) const;
    __device__ __forceinline__ void put(const unsigned char* base, int i, const ChunkT<float>& c) const
    {
        float4* q = reinterpret_cast<float4*>(const_cast<unsigned char*>(base) + (size_t)i * 32);
        q[0] = make_float4(c.f[0], c.f[1], c.f[2], c.f[3]);
        q[1] = make_float4(c.f[4], c.f[5], c.f[6], c.f[7]);
    }
};
template <>
__device__ __forceinline__ void SmemRow<bf16>::chunk(const unsigned char* base, int i, int, ChunkT<bf16>& c) const
{
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(c.w[0]), "=r"(c.w[1]), "=r"(c.w[2]), "=r"(c.w[3])
                 : "r"(smem_addr(base) + (uint32_t)i * 16u));
}
template <>
__device__ __forceinline__ void SmemRow<float>::chunk(const unsigned char* base, int i, int, ChunkT<float>& c) const
{
    const float4 a = *reinterpret_cast<const float4*>(base + (size_t)i * 32);
    const float4 b = *reinterpret_cast<const float4*>(base + (size_t)i * 32 + 16);
    c.f[0] = a.x, c.f[1] = a.y, c.f[2] = a.z, c.f[3] = a.w;
    c.f[4] = b.x, c.f[5] = b.y, c.f[6] = b.z, c.f[7] = b.w;
}

template <typename T>
struct GlobalRow {
    static constexpr bool kKeeps = false;
    const T* x;
    const T* m;
    bool vec;
    __device__ __forceinline__ void put(const T*, int, const ChunkT<float>&) const {}
    __device__ __forceinline__ void chunk(const T* base, int i, int n, ChunkT<T>& c) const;
};
template <>
__device__ __forceinline__ void GlobalRow<bf16>::chunk(const bf16* base, int i, int n, ChunkT<bf16>& c) const
{
    load_words(base + (size_t)i * 8, vec, n, c.w);
}
template <>
__device__ __forceinline__ void GlobalRow<float>::chunk(const float* base, int i, int n, ChunkT<float>& c) const
{
    load8f(base + (size_t)i * 8, vec, n, c.f);
}

// Mask rows in global memory, read through the read-only (L1) path.
template <typename T>
struct MaskRow {
    bool vec;
    __device__ __forceinline__ void chunk(const T* base, int i, int n, ChunkT<T>& c) const;
};
template <>
__device__ __forceinline__ void MaskRow<bf16>::chunk(const bf16* base, int i, int n, ChunkT<bf16>& c) const
{
    if (vec && n == 8) {
        const uint4 v = ld16_ro(base + (size_t)i * 8);
        c.w[0] = v.x, c.w[1] = v.y, c.w[2] = v.z, c.w[3] = v.w;
    } else {
        load_words(base + (size_t)i * 8, false, n, c.w);
    }
}
template <>
__device__ __forceinline__ void MaskRow<float>::chunk(const float* base, int i, int n, ChunkT<float>& c) const
{
    if (vec && n == 8) {
        const uint4 a = ld16_ro(base + (size_t)i * 8), b = ld16_ro(base + (size_t)i * 8 + 4);
        c.f[0] = __uint_as_float(a.x), c.f[1] = __uint_as_float(a.y), c.f[2] = __uint_as_float(a.z);
        c.f[3] = __uint_as_float(a.w), c.f[4] = __uint_as_float(b.x), c.f[5] = __uint_as_float(b.y);
        c.f[6] = __uint_as_float(b.z), c.f[7] = __uint_as_float(b.w);
    } else {
        load8f(base + (size_t)i * 8, false, n, c.f);
    }
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = (threadIdx.x & o) ? u + v : v + u;
    }
    return v;
}

__device__ __forceinline__ Acc warp_acc(Acc a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const Acc b{__shfl_xor_sync(0xFFFFFFFFu, a.s, o), __shfl_xor_sync(0xFFFFFFFFu, a.c, o)};
        a = (threadIdx.x & o) ? acc_merge(b, a) : acc_merge(a, b);
    }
    return a;
}

// Elements of chunk i valid in a row of `valid` (0 .. 8).
__device__ __forceinline__ int chunk_n(int valid, int i)
{
    const int left = valid - i * 8;
    return left <= 0 ? 0 : (left < 8 ? left : 8);
}

// Store chunk i (8 outputs, of which the first cnt exist) of row yr.
__device__ __forceinline__ void store_chunk(bf16* yr, int i, int cnt, bool vec, const uint32_t (&w)[4])
{
    if (vec && cnt == 8) {
        st16(yr + (size_t)i * 8, make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        for (int j = 0; j < cnt; ++j)
            yr[(size_t)i * 8 + j].bits = (uint16_t)(j & 1 ? w[j >> 1] >> 16 : w[j >> 1] & 0xFFFFu);
    }
}

// -------- bf16 forward of one row by one warp -------------------------------
// Chunks [0, Gf) of the valid prefix are full; chunk Gf holds the last
// valid % 8 elements (if any) and is handled by one lane; chunks past the
// valid prefix are zeros.  The hot loops have no per-element tests.  `src`
// reads x (a shared-memory stage or global memory), `msrc` the mask rows
// (global memory through the read-only cache: a mask broadcast over heads
// or queries is read by many rows and stays in L1 and L2).

// The eight exponentials 2^t of one full chunk (t as in fwd_row_fast).
template <bool NEAR, bool MASK>
__device__ __forceinline__ void exps8(const ChunkT<bf16>& c, const ChunkT<bf16>& k, float2 sL, float2 cL, float scale,
                                      float m, float2 (&e)[4])
{
    const float kL2e = (float)kLog2e;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float2 tt;
        if (NEAR) {
            const float2 base = MASK ? fma2(widen2(k.w[q]), f2(kL2e), cL) : cL;
            tt = fma2(widen2(c.w[q]), sL, base);
        } else {
            const float2 d = MASK ? fma2(widen2(c.w[q]), f2(scale), add2(widen2(k.w[q]), f2(-m)))
                                  : fma2(widen2(c.w[q]), f2(scale), f2(-m));
            tt = fma2(d, f2(kL2e), f2(64.0f));
        }
        e[q] = make_float2(ex2_ftz(tt.x), ex2_ftz(tt.y));
    }
}

__device__ __forceinline__ void zero_past(float2 (&e)[4], int n)
{
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j >= n)
            (j & 1 ? e[j >> 1].y : e[j >> 1].x) = 0.0f;
}

// Pass 2 (row sum) and pass 3 (output) of a row whose maximum is m.
template <bool NEAR, bool MASK, class Src, typename P, class MSrc, typename PM>
__device__ __forceinline__ void fwd_bf16_finish(const Src& src, P xb, const MSrc& msrc, PM mb, int valid, int sk,
                                                float scale, float m, bf16* yr, bool vec)
{
    const int lane = threadIdx.x & 31;
    const int G = (sk + 7) / 8, Gf = valid >> 3, tail = valid & 7, Gv = Gf + (tail ? 1 : 0);
    const float kL2e = (float)kLog2e;
    const float2 sL = f2(scale * kL2e), cL = f2(fmaf(-m, kL2e, 64.0f));
    ChunkT<bf16> k{};
    float2 s2 = make_float2(0.0f, 0.0f);
    for (int i = lane; i < Gf; i += 32) {
        ChunkT<bf16> c;
        if (MASK)
            msrc.chunk(mb, i, 8, k);
        src.chunk(xb, i, 8, c);
        float2 e[4];
        exps8<NEAR, MASK>(c, k, sL, cL, scale, m, e);
        s2 = add2(s2, add2(add2(e[0], e[1]), add2(e[2], e[3])));
    }
    if (tail && lane == (Gf & 31)) {
        ChunkT<bf16> c;
        if (MASK)
            msrc.chunk(mb, Gf, tail, k);
        src.chunk(xb, Gf, tail, c);
        float2 e[4];
        exps8<NEAR, MASK>(c, k, sL, cL, scale, m, e);
        zero_past(e, tail);
        s2 = add2(s2, add2(add2(e[0], e[1]), add2(e[2], e[3])));
    }
    const float2 rs = f2(__frcp_rn(warp_sum(s2.x + s2.y)));
    for (int i = lane; i < Gf; i += 32) {
        ChunkT<bf16> c;
        if (MASK)
            msrc.chunk(mb, i, 8, k);
        src.chunk(xb, i, 8, c);
        float2 e[4];
        exps8<NEAR, MASK>(c, k, sL, cL, scale, m, e);
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 yv = mul2(e[q], rs);
            o[q] = pack_bf16x2(yv.x, yv.y);
        }
        store_chunk(yr, i, 8, vec, o);
    }
    if (tail && lane == (Gf & 31)) {
        ChunkT<bf16> c;
        if (MASK)
            msrc.chunk(mb, Gf, tail, k);
        src.chunk(xb, Gf, tail, c);
        float2 e[4];
        exps8<NEAR, MASK>(c, k, sL, cL, scale, m, e);
        zero_past(e, tail);
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 yv = mul2(e[q], rs);
            o[q] = pack_bf16x2(yv.x, yv.y);
        }
        store_chunk(yr, Gf, chunk_n(sk, Gf), vec, o);
    }
    const uint32_t z[4] = {0u, 0u, 0u, 0u};
    for (int i = Gv + ((lane - Gv) & 31); i < G; i += 32)
        store_chunk(yr, i, chunk_n(sk, i), vec, z);
}

template <bool MASK, class Src, typename P, class MSrc, typename PM>
__device__ __forceinline__ void warp_row_fwd_bf16(const Src& src, P xb, const MSrc& msrc, PM mb, int valid, int sk,
                                                  float scale, bf16* yr, bool vec)
{
    const int lane = threadIdx.x & 31;
    const int G = (sk + 7) / 8, Gf = valid >> 3, tail = valid & 7;
    // pass 1: the row maximum of the scores
    float m = -INFINITY;
    if (!MASK) {
        // on the packed words; a negative scale takes the maximum of -x
        const uint32_t flip = scale < 0.0f ? 0x80008000u : 0u;
        uint32_t a0 = 0xFF80FF80u, a1 = 0xFF80FF80u;  // (-inf, -inf)
        for (int i = lane; i < Gf; i += 32) {
            ChunkT<bf16> c;
            src.chunk(xb, i, 8, c);
            a0 = bmax2(a0, c.w[0] ^ flip), a1 = bmax2(a1, c.w[1] ^ flip);
            a0 = bmax2(a0, c.w[2] ^ flip), a1 = bmax2(a1, c.w[3] ^ flip);
        }
        const float2 h = widen2(bmax2(a0, a1));
        float xm = fmaxf(h.x, h.y);
        if (tail && lane == (Gf & 31)) {
            ChunkT<bf16> c;
            src.chunk(xb, Gf, tail, c);
            for (int j = 0; j < tail; ++j)
                xm = fmaxf(xm, flip ? -word_elem(c.w, j) : word_elem(c.w, j));
        }
        xm = warp_max(xm);
        if (valid > 0)
            m = (flip ? -xm : xm) * scale;
    } else {
        for (int i = lane; i < Gf; i += 32) {
            ChunkT<bf16> c, k;
            msrc.chunk(mb, i, 8, k);
            src.chunk(xb, i, 8, c);
            const float2 z0 = fma2(widen2(c.w[0]), f2(scale), widen2(k.w[0]));
            const float2 z1 = fma2(widen2(c.w[1]), f2(scale), widen2(k.w[1]));
            const float2 z2 = fma2(widen2(c.w[2]), f2(scale), widen2(k.w[2]));
            const float2 z3 = fma2(widen2(c.w[3]), f2(scale), widen2(k.w[3]));
            m = fmaxf(m, fmaxf(fmaxf(fmaxf(z0.x, z0.y), fmaxf(z1.x, z1.y)),
                               fmaxf(fmaxf(z2.x, z2.y), fmaxf(z3.x, z3.y))));
        }
        if (tail && lane == (Gf & 31)) {
            ChunkT<bf16> c, k;
            msrc.chunk(mb, Gf, tail, k);
            src.chunk(xb, Gf, tail, c);
            for (int j = 0; j < tail; ++j)
                m = fmaxf(m, fmaf(word_elem(c.w, j), scale, word_elem(k.w, j)));
        }
        m = warp_max(m);
    }
    if (m == -INFINITY) {  // no finite score left: zeros
        const uint32_t z[4] = {0u, 0u, 0u, 0u};
        for (int i = lane; i < G; i += 32)
            store_chunk(yr, i, chunk_n(sk, i), vec, z);
        return;
    }
    if (fabsf(m) <= 64.0f)
        fwd_bf16_finish<true, MASK>(src, xb, msrc, mb, valid, sk, scale, m, yr, vec);
    else
        fwd_bf16_finish<false, MASK>(src, xb, msrc, mb, valid, sk, scale, m, yr, vec);
}

// -------- fp32 forward of one row by one warp -------------------------------
// e^d = 2^(d log2 e) by the hardware base-2 exponential, with d = x scale +
// (mask - M) formed by one fused multiply-add: the relative error of e^d is
// about 2^-22 plus the rounding of d log2 e (|d| 2^-24), so y = e^d / sum is
// within 3e-7 of the exact value everywhere (|d| e^d <= 1/e).
template <bool MASK>
__device__ __forceinline__ void exps8_f32(ChunkT<float>& c, const ChunkT<float>& k, float scale, float mneg)
{
    const float kL2e = (float)kLog2e;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        c.f[j] = ex2_ftz(fmaf(c.f[j], scale, MASK ? k.f[j] + mneg : mneg) * kL2e);
}

template <bool MASK, class Src, typename P, class MSrc, typename PM>
__device__ __forceinline__ void warp_row_fwd_f32(const Src& src, P xb, const MSrc& msrc, PM mb, int valid, int sk,
                                                 float scale, float* yr, bool vec)
{
    const int lane = threadIdx.x & 31;
    const int G = (sk + 7) / 8, Gf = valid >> 3, tail = valid & 7, Gv = Gf + (tail ? 1 : 0);
    // pass 1: the row maximum (without a mask: the maximum of sg x times
    // scale; rounding is monotone, so it equals the maximum of x scale)
    float m = -INFINITY;
    if (!MASK) {
        float xm = -INFINITY;
        if (scale >= 0.0f) {
            for (int i = lane; i < Gf; i += 32) {
                ChunkT<float> c;
                src.chunk(xb, i, 8, c);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    xm = fmaxf(xm, c.f[j]);
            }
        } else {
            for (int i = lane; i < Gf; i += 32) {
                ChunkT<float> c;
                src.chunk(xb, i, 8, c);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    xm = fmaxf(xm, -c.f[j]);
            }
        }
        if (xm != -INFINITY)
            m = (scale < 0.0f ? -xm : xm) * scale;
    } else {
        for (int i = lane; i < Gf; i += 32) {
            ChunkT<float> c, k;
            msrc.chunk(mb, i, 8, k);
            src.chunk(xb, i, 8, c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                m = fmaxf(m, fmaf(c.f[j], scale, k.f[j]));
        }
    }
    if (tail && lane == (Gf & 31)) {
        ChunkT<float> c, k;
        if (MASK)
            msrc.chunk(mb, Gf, tail, k);
        src.chunk(xb, Gf, tail, c);
        for (int j = 0; j < tail; ++j)
            m = fmaxf(m, MASK ? fmaf(c.f[j], scale, k.f[j]) : c.f[j] * scale);
    }
    m = warp_max(m);
    if (m == -INFINITY) {  // no finite score left: zeros
        float z[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        for (int i = lane; i < G; i += 32)
            store8f(yr + (size_t)i * 8, vec, chunk_n(sk, i), z);
        return;
    }
    const float mneg = -m;
    // pass 2: exponentials (parked in the stage when it allows) and the sum
    Acc acc{0.0f, 0.0f};
    for (int i = lane; i < Gv; i += 32) {
        ChunkT<float> c, k;
        const int n = i < Gf ? 8 : tail;
        if (MASK)
            msrc.chunk(mb, i, n, k);
        src.chunk(xb, i, n, c);
        exps8_f32<MASK>(c, k, scale, mneg);
        if (n < 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j >= n)
                    c.f[j] = 0.0f;
        }
        two_sum_add(acc, sum8(c.f));
        if constexpr (Src::kKeeps)
            src.put(xb, i, c);  // the output pass reads e^d back instead of recomputing it
    }
    const float rs = __frcp_rn(acc_value(warp_acc(acc)));
    // pass 3: normalise and store, zeros past the valid prefix
    for (int i = lane; i < G; i += 32) {
        float o[8];
        if (i < Gv) {
            ChunkT<float> c, k;
            const int n = i < Gf ? 8 : tail;
            src.chunk(xb, i, n, c);
            if constexpr (!Src::kKeeps) {
                if (MASK)
                    msrc.chunk(mb, i, n, k);
                exps8_f32<MASK>(c, k, scale, mneg);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o[j] = j < n ? c.f[j] * rs : 0.0f;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o[j] = 0.0f;
        }
        store8f(yr + (size_t)i * 8, vec, chunk_n(sk, i), o);
    }
}

// -------- backward of one row by one warp -----------------------------------
template <class Src, typename P>
__device__ __forceinline__ void warp_row_bwd_bf16(const Src& src, P gb, P yb, int valid, int sk, float scale, bf16* dxr,
                                                  bool vec)
{
    const int lane = threadIdx.x & 31;
    const int G = (sk + 7) / 8, Gv = (valid + 7) / 8;
    Acc acc{0.0f, 0.0f};
    for (int i = lane; i < Gv; i += 32) {
        ChunkT<bf16> g, y;
        const int n = chunk_n(valid, i);
        src.chunk(gb, i, n, g);
        src.chunk(yb, i, n, y);
        zero_tail_words(g.w, n);
        zero_tail_words(y.w, n);
        const float2 p0 = mul2(widen2(g.w[0]), widen2(y.w[0]));
        const float2 p1 = mul2(widen2(g.w[1]), widen2(y.w[1]));
        const float2 p2 = mul2(widen2(g.w[2]), widen2(y.w[2]));
        const float2 p3 = mul2(widen2(g.w[3]), widen2(y.w[3]));
        const float2 q = add2(add2(p0, p1), add2(p2, p3));
        two_sum_add(acc, q.x + q.y);
    }
    const float s = acc_value(warp_acc(acc));
    const float2 ms = f2(-s), sc = f2(scale);
    for (int i = lane; i < G; i += 32) {
        const int n = chunk_n(valid, i);
        uint32_t o[4] = {0u, 0u, 0u, 0u};
        if (n > 0) {
            ChunkT<bf16> g, y;
            src.chunk(gb, i, n, g);
            src.chunk(yb, i, n, y);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 d = mul2(mul2(sc, widen2(y.w[q])), add2(widen2(g.w[q]), ms));
                o[q] = pack_bf16x2(d.x, d.y);
            }
            zero_tail_words(o, n);
        }
        store_chunk(dxr, i, chunk_n(sk, i), vec, o);
    }
}

template <class Src, typename P>
__device__ __forceinline__ void warp_row_bwd_f32(const Src& src, P gb, P yb, int valid, int sk, float scale, float* dxr,
                                                 bool vec)
{
    const int lane = threadIdx.x & 31;
    const int G = (sk + 7) / 8, Gv = (valid + 7) / 8;
    Acc acc{0.0f, 0.0f};
    for (int i = lane; i < Gv; i += 32) {
        ChunkT<float> g, y;
        const int n = chunk_n(valid, i);
        src.chunk(gb, i, n, g);
        src.chunk(yb, i, n, y);
        float p[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            p[j] = j < n ? g.f[j] * y.f[j] : 0.0f;
        two_sum_add(acc, sum8(p));
    }
    const float s = acc_value(warp_acc(acc));
    for (int i = lane; i < G; i += 32) {
        const int n = chunk_n(valid, i);
        float o[8];
        ChunkT<float> g, y;
        if (n > 0) {
            src.chunk(gb, i, n, g);
            src.chunk(yb, i, n, y);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = j < n ? (scale * y.f[j]) * (g.f[j] - s) : 0.0f;
        store8f(dxr + (size_t)i * 8, vec, chunk_n(sk, i), o);
    }
}

template <typename T, bool MASK, class Src, typename P>
__device__ __forceinline__ void warp_row_fwd(const Src& src, P xb, const T* mb, int valid, int sk, float scale, T* yr,
                                             bool vec, bool mvec)
{
    const MaskRow<T> msrc{mvec};
    if constexpr (DTypeInfo<T>::kBf16)
        warp_row_fwd_bf16<MASK>(src, xb, msrc, mb, valid, sk, scale, yr, vec);
    else
        warp_row_fwd_f32<MASK>(src, xb, msrc, mb, valid, sk, scale, yr, vec);
}

template <typename T, class Src, typename P>
__device__ __forceinline__ void warp_row_bwd(const Src& src, P gb, P yb, int valid, int sk, float scale, T* dxr, bool vec)
{
    if constexpr (DTypeInfo<T>::kBf16)
        warp_row_bwd_bf16(src, gb, yb, valid, sk, scale, dxr, vec);
    else
        warp_row_bwd_f32(src, gb, yb, valid, sk, scale, dxr, vec);
}

// Direct forms: warp w of the grid takes rows w, w + warps, ...
template <typename T, bool MASK, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
softmax_fwd_warp(const T* x, const T* __restrict__ mask, T* y, SoftmaxGeom g, float scale, bool vec)
{
    const int64_t warps = (int64_t)gridDim.x * kWarps;
    const GlobalRow<T> src{x, mask, vec};
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < g.rows; r += warps) {
        const int valid = (int)(CAUSAL ? query32(g, (uint32_t)r) + 1 : g.sk);
        const T* mr = MASK ? mask + mask_row32(g, (uint32_t)r) : nullptr;
        warp_row_fwd<T, MASK>(src, x + r * g.sk, mr, valid, (int)g.sk, scale, y + r * g.sk, vec, vec);
    }
}

template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
softmax_bwd_warp(const T* dy, const T* y, T* dx, SoftmaxGeom g, float scale, bool vec)
{
    const int64_t warps = (int64_t)gridDim.x * kWarps;
    const GlobalRow<T> src{dy, y, vec};
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < g.rows; r += warps) {
        const int valid = (int)(CAUSAL ? query32(g, (uint32_t)r) + 1 : g.sk);
        warp_row_bwd<T>(src, dy + r * g.sk, y + r * g.sk, valid, (int)g.sk, scale, dx + r * g.sk, vec);
    }
}

// Pipelined forms.  The pipeline moves units: a row, or under the causal
// mask a pair of rows (below).  Stage `it` of block b holds RPS consecutive
// units [(b + it * grid) * RPS, + RPS) of each of the NT tensors (x alone in
// the forward, whose mask rows come from global memory; dy and y in the
// backward), at a pitch of row_bytes; consumer warp w serves unit w % RPS of
// the iterations it = w / RPS (mod 8 / RPS).
struct RowPipe {
    int rps, ns;          // units per stage, stages
    uint32_t row_bytes;   // pitch of a unit: sk * sizeof(T), plus 8 elements for a pair
    uint32_t slot_bytes;  // rps * row_bytes: one tensor's units in a stage
    uint32_t stage_bytes; // NT * slot_bytes
    int64_t units;        // rows, or pairs
    uint32_t hp;          // pairs per head: ceil(sq / 2)
    Div32 dhp;            // division by hp
    bool pairs;           // causal units are row pairs (else single causal rows)
};

// Causal pairs.  Row q of a head keeps q + 1 scores, so a stage of whole
// rows carries half its capacity on average.  Pair p of head h instead
// holds rows q = p and sq - 1 - p (P = h * hp + p), sq + 1 kept scores
// together: every stage is full.  The two rows sit back to back in the
// unit, each rounded up to whole chunks of 8 (at most sq + 8 elements in
// all, as sq is a multiple of 8 here).  When sq is odd the middle row is
// alone (vb = 0).
struct PairRows {
    int64_t ra, rb;  // global row indices
    int va, vb;      // kept scores (vb = 0: no second row)
};

__device__ __forceinline__ PairRows pair_rows(const SoftmaxGeom& g, const RowPipe& p, uint32_t P)
{
    if (!p.pairs)  // a single causal row
        return PairRows{P, P, (int)query32(g, P) + 1, 0};
    const uint32_t h = p.dhp.div(P), q = P - h * p.hp;
    const uint32_t sq = (uint32_t)g.sq, q2 = sq - 1u - q;
    const int64_t base = (int64_t)h * sq;
    return PairRows{base + q, base + q2, (int)q + 1, q2 != q ? (int)q2 + 1 : 0};
}

// Bytes of the first v scores of a row rounded up to whole chunks.
template <typename T>
__device__ __forceinline__ uint32_t kept_bytes(int v)
{
    return (uint32_t)(((v + 7) / 8) * 8 * (int)sizeof(T));
}

// A consumer group waits for use n of a stage whose uses n - 1, n - 2, ...
// belong to other groups and may not have completed yet.  A parity wait
// cannot tell use n from use n - 2 (both have parity n & 1, and a wait on the
// parity of the phase before the current one returns at once), so the
// producer also publishes, per stage, how many uses it has started: once
// `issued[s]` exceeds n, every earlier use of s has been released, the full
// barrier is in phase n, and the parity wait is exact.
struct RowRing {
    Ring ring;
    volatile int* issued;  // [kMaxStages], in shared memory
};

__device__ __forceinline__ RowRing ring_setup_rt(unsigned char* smem, int ns, uint32_t empty_count, volatile int* issued)
{
    Ring r{smem_addr(smem), smem_addr(smem) + 8u * kMaxStages};
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(r.full(s), 1);
            mbar_init(r.empty(s), empty_count);
            issued[s] = 0;
        }
        mbar_init_fence();
    }
    __syncthreads();
    return RowRing{r, issued};
}

// Consumer wait for use n = it / ns of stage s = it % ns (bounded; the same
// outcome for every lane of the warp).
__device__ __forceinline__ bool row_acquire(const RowRing& rr, int ns, int64_t it)
{
    const int s = (int)(it % ns);
    const int64_t n = it / ns;
    bool ok = false;
    for (uint32_t k = 0; k < kWaitLimit; ++k) {
        if (rr.issued[s] > n) {
            ok = true;
            break;
        }
        __nanosleep(32);
    }
    ok = ok && mbar_wait(rr.ring.full(s), (uint32_t)(n & 1));
    return __all_sync(0xFFFFFFFFu, ok);
}

template <typename T, int NT, bool CAUSAL>
__device__ __forceinline__ void row_producer(const RowRing& rr, unsigned char* data, const RowPipe& p, const T* x,
                                             const T* second, const SoftmaxGeom& g, int64_t iters)
{
    const Ring& ring = rr.ring;
    const int lane = threadIdx.x & 31;
    for (int64_t it = 0; it < iters; ++it) {
        const int s = (int)(it % p.ns);
        const int64_t n = it / p.ns;
        if (n > 0) {
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(ring.empty(s), (uint32_t)((n - 1) & 1));
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    atomicOr(&g_device_error, 2u);
                    for (int64_t j = it - 1; j >= 0 && j > it - p.ns; --j)
                        if (!mbar_wait(ring.full((int)(j % p.ns)), (uint32_t)((j / p.ns) & 1)))
                            atomicOr(&g_device_error, 4u);
                }
                return;
            }
        }
        const int64_t r0 = ((int64_t)blockIdx.x + it * gridDim.x) * p.rps;
        const int nrows = (int)(p.units - r0 < p.rps ? p.units - r0 : p.rps);
        uint32_t part = 0;
        if (!CAUSAL) {
            part = lane == 0 ? NT * (uint32_t)nrows * p.row_bytes : 0u;
        } else {
            for (int l = lane; l < nrows; l += 32) {
                const PairRows q = pair_rows(g, p, (uint32_t)(r0 + l));
                part += NT * (kept_bytes<T>(q.va) + kept_bytes<T>(q.vb));
            }
        }
        const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, part);
        const uint32_t st = smem_addr(data + (size_t)s * p.stage_bytes);
        if (lane == 0) {
            rr.issued[s] = (int)(n + 1);
            mbar_arrive_expect_tx(ring.full(s), total);
        }
        __syncwarp();
        if (!CAUSAL) {
            if (lane == 0)
                bulk_g2s(st, x + r0 * g.sk, (uint32_t)nrows * p.row_bytes, ring.full(s));
            if (NT == 2 && lane == 0)
                bulk_g2s(st + p.slot_bytes, second + r0 * g.sk, (uint32_t)nrows * p.row_bytes, ring.full(s));
        } else {
            for (int l = lane; l < nrows; l += 32) {
                const PairRows q = pair_rows(g, p, (uint32_t)(r0 + l));
                const uint32_t ba = kept_bytes<T>(q.va), bb = kept_bytes<T>(q.vb);
                for (int t = 0; t < NT; ++t) {
                    const T* src = t == 0 ? x : second;
                    const uint32_t d = st + (uint32_t)t * p.slot_bytes + (uint32_t)l * p.row_bytes;
                    bulk_g2s(d, src + q.ra * g.sk, ba, ring.full(s));
                    if (bb)
                        bulk_g2s(d + ba, src + q.rb * g.sk, bb, ring.full(s));
                }
            }
        }
    }
}

template <typename T, bool MASK, bool CAUSAL>
__global__ void __launch_bounds__(kPipeThreads, 1)
softmax_fwd_rowpipe(const T* x, const T* __restrict__ mask, T* y, SoftmaxGeom g, float scale, RowPipe p)
{
    constexpr int NT = 1;  // x only: the mask is read from global memory
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int issued[kMaxStages];
    const RowRing rr = ring_setup_rt(smem, p.ns, (uint32_t)p.rps, issued);
    unsigned char* data = smem + kRingHeader;
    const int64_t nst = (p.units + p.rps - 1) / p.rps;
    const int64_t iters = nst > blockIdx.x ? (nst - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int w = threadIdx.x >> 5;
    if (w == kConsumerWarps) {
        row_producer<T, NT, CAUSAL>(rr, data, p, x, nullptr, g, iters);
        return;
    }
    const int groups = kConsumerWarps / p.rps, slot = w % p.rps;
    const SmemRow<T> src{nullptr, nullptr};
    for (int64_t it = w / p.rps; it < iters; it += groups) {
        const int s = (int)(it % p.ns);
        if (!row_acquire(rr, p.ns, it)) {
            if ((threadIdx.x & 31) == 0)
                atomicOr(&g_device_error, 1u);
            return;
        }
        const int64_t u = ((int64_t)blockIdx.x + it * gridDim.x) * p.rps + slot;
        if (u < p.units) {
            const unsigned char* xb = data + (size_t)s * p.stage_bytes + (size_t)slot * p.row_bytes;
            if (!CAUSAL) {
                const T* mb = MASK ? mask + mask_row32(g, (uint32_t)u) : nullptr;
                warp_row_fwd<T, MASK>(src, xb, mb, (int)g.sk, (int)g.sk, scale, y + u * g.sk, true, true);
            } else {
                // one copy of the row code for both rows of the pair
                const PairRows q = pair_rows(g, p, (uint32_t)u);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const int64_t r = h ? q.rb : q.ra;
                    const int v = h ? q.vb : q.va;
                    if (v == 0)
                        break;
                    const T* mr = MASK ? mask + mask_row32(g, (uint32_t)r) : nullptr;
                    warp_row_fwd<T, MASK>(src, xb + (h ? kept_bytes<T>(q.va) : 0u), mr, v, (int)g.sk, scale,
                                          y + r * g.sk, true, true);
                }
            }
        }
        if constexpr (!DTypeInfo<T>::kBf16) {
            // the fp32 rows parked values in the stage with ordinary stores;
            // order them before the bulk copies that will refill it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            mbar_arrive(rr.ring.empty(s));
    }
}

template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kPipeThreads, 1)
softmax_bwd_rowpipe(const T* dy, const T* y, T* dx, SoftmaxGeom g, float scale, RowPipe p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int issued[kMaxStages];
    const RowRing rr = ring_setup_rt(smem, p.ns, (uint32_t)p.rps, issued);
    unsigned char* data = smem + kRingHeader;
    const int64_t nst = (p.units + p.rps - 1) / p.rps;
    const int64_t iters = nst > blockIdx.x ? (nst - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int w = threadIdx.x >> 5;
    if (w == kConsumerWarps) {
        row_producer<T, 2, CAUSAL>(rr, data, p, dy, y, g, iters);
        return;
    }
    const int groups = kConsumerWarps / p.rps, slot = w % p.rps;
    const SmemRow<T> src{nullptr, nullptr};
    for (int64_t it = w / p.rps; it < iters; it += groups) {
        const int s = (int)(it % p.ns);
        if (!row_acquire(rr, p.ns, it)) {
            if ((threadIdx.x & 31) == 0)
                atomicOr(&g_device_error, 1u);
            return;
        }
        const int64_t u = ((int64_t)blockIdx.x + it * gridDim.x) * p.rps + slot;
        if (u < p.units) {
            const unsigned char* gb = data + (size_t)s * p.stage_bytes + (size_t)slot * p.row_bytes;
            const unsigned char* yb = gb + p.slot_bytes;
            if (!CAUSAL) {
                warp_row_bwd<T>(src, gb, yb, (int)g.sk, (int)g.sk, scale, dx + u * g.sk, true);
            } else {
                const PairRows q = pair_rows(g, p, (uint32_t)u);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const int64_t r = h ? q.rb : q.ra;
                    const int v = h ? q.vb : q.va;
                    if (v == 0)
                        break;
                    const uint32_t off = h ? kept_bytes<T>(q.va) : 0u;
                    warp_row_bwd<T>(src, gb + off, yb + off, v, (int)g.sk, scale, dx + r * g.sk, true);
                }
            }
        }
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            mbar_arrive(rr.ring.empty(s));
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
constexpr int kC = kC_;
constexpr int64_t kMaxTeamChunks = (int64_t)kC * kThreads;

SoftmaxGeom make_geom(int64_t rows, int64_t sq, int64_t np, int64_t sk, int64_t mb, int64_t mnp, int64_t msq)
{
    SoftmaxGeom g{rows, sq, np, sk, mb, mnp, msq, Div32{1, 1, 0}, Div32{1, 1, 0}};
    if (rows < (int64_t(1) << 32)) {  // sq, np <= rows (or the op is empty)
        g.dsq = make_div32((uint32_t)(sq > 0 ? sq : 1));
        g.dnp = make_div32((uint32_t)(np > 0 ? np : 1));
    }
    return g;
}

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

// Ring of the row pipeline: the most units per stage (8, 4, 2, 1) that keep
// three stages in the ring (two for single units); false when even that does
// not fit.  The count is planned on whole rows; a causal pair's pitch is 8
// elements longer (its chunk rounding), which the ring absorbs.  Causal
// pipelines need sq = sk (a multiple of 8) and rows a multiple of sq.
template <typename T, int NT, bool CAUSAL>
bool row_pipe_plan(int64_t rows, int64_t sk, RowPipe* p)
{
    const uint64_t row = (uint64_t)sk * sizeof(T);
    const bool pairs = CAUSAL && (NT == 1 ? MFX_SOFTMAX_PAIRS_FWD : MFX_SOFTMAX_PAIRS_BWD);
    const uint64_t pitch = pairs ? row + 8 * sizeof(T) : row;
    const uint64_t ring = (uint64_t)(NT == 2 ? MFX_RING_KB_SOFTMAX_BWD : MFX_RING_KB_SOFTMAX) * 1024;
    if (CAUSAL && (sk <= 0 || sk % 8 != 0 || rows % sk != 0))
        return false;
    const uint32_t hp = pairs ? (uint32_t)((sk + 1) / 2) : 1u;
    const int64_t units = pairs ? rows / sk * hp : rows;
    for (int rps = pairs ? MFX_SOFTMAX_PAIR_RPS : kConsumerWarps; rps >= 1; rps /= 2) {
        const uint64_t stage = (uint64_t)NT * rps * row;
        const uint64_t ns = ring / stage < (uint64_t)kMaxStages ? ring / stage : (uint64_t)kMaxStages;
        if (ns >= 3 || (rps == 1 && ns >= 2)) {
            *p = RowPipe{rps, (int)ns, (uint32_t)pitch, (uint32_t)(rps * pitch), (uint32_t)(NT * rps * pitch),
                         units, hp, make_div32(hp), pairs};
            return true;
        }
    }
    return false;
}

// Launch a row-pipeline kernel with its dynamic shared memory, one block per
// resident slot, no more blocks than stages.
template <typename K, typename... Args>
int launch_rowpipe(K kernel, const RowPipe& p, int64_t rows, cudaStream_t s, Args... args)
{
    const size_t smem = kRingHeader + (size_t)p.ns * p.stage_bytes;
    const int occ = occupancy((const void*)kernel, kPipeThreads, smem);
    const int64_t nst = (p.units + p.rps - 1) / p.rps;
    const int64_t cap = (int64_t)sm_count() * occ;
    const unsigned blocks = (unsigned)(nst < cap ? nst : cap);
    kernel<<<blocks, kPipeThreads, smem, s>>>(args..., p);
    return launch_status();
}

// Regimes by row length G = ceil(sk / 8) chunks: team kernels below 64
// chunks, warp-per-row kernels up to 2048 (pipelined when aligned and the
// ring fits, direct otherwise), block-per-row kernels beyond (and for more
// than 2^32 rows).
constexpr int64_t kWarpRowMin = 64, kWarpRowMax = 2048;

template <typename T, bool MASK, bool CAUSAL>
int launch_fwd(const SoftmaxGeom& g, const void* x, const void* mask, void* y, float scale, cudaStream_t s)
{
    const T* xp = static_cast<const T*>(x);
    const T* mp = static_cast<const T*>(mask);
    T* yp = static_cast<T*>(y);
    const bool vec = g.sk % 8 == 0 && aligned16(x) && aligned16(y) && (!MASK || aligned16(mask));
    const int64_t G = (g.sk + 7) / 8;
    const bool idx32 = g.rows < (int64_t(1) << 32);
    if (idx32 && G < kWarpRowMin) {
        auto k = softmax_fwd_team<T, kC, MASK, CAUSAL>;
        const int lg = team_lg(G);
        unsigned blocks;
        int64_t iters;
        team_launch_dims(k, g.rows, lg, &blocks, &iters);
        k<<<blocks, kThreads, 0, s>>>(xp, mp, yp, g, scale, lg, iters, vec);
        return launch_status();
    }
    if (idx32 && G <= kWarpRowMax) {
        RowPipe p;
        if (MFX_PIPE_SOFTMAX && vec && row_pipe_plan<T, 1, CAUSAL>(g.rows, g.sk, &p))
            return launch_rowpipe(softmax_fwd_rowpipe<T, MASK, CAUSAL>, p, g.rows, s, xp, mp, yp, g, scale);
        auto k = softmax_fwd_warp<T, MASK, CAUSAL>;
        const int64_t need = (g.rows + kWarps - 1) / kWarps;
        const int64_t cap = (int64_t)sm_count() * blocks_per_sm((const void*)k);
        k<<<(unsigned)(need < cap ? need : cap), kThreads, 0, s>>>(xp, mp, yp, g, scale, vec);
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
    const int64_t G = (sk + 7) / 8;
    const bool idx32 = rows < (int64_t(1) << 32);
    if (idx32 && G < kWarpRowMin) {
        auto k = softmax_bwd_team<T, kC, CAUSAL>;
        const int lg = team_lg(G);
        unsigned blocks;
        int64_t iters;
        team_launch_dims(k, rows, lg, &blocks, &iters);
        k<<<blocks, kThreads, 0, s>>>(gp, yp, dp, rows, sk, make_div32((uint32_t)sk), scale, lg, iters, vec);
        return launch_status();
    }
    if (idx32 && G <= kWarpRowMax) {
        const SoftmaxGeom g = make_geom(rows, CAUSAL ? sk : 1, 1, sk, 1, 1, 1);
        RowPipe p;
        if (MFX_PIPE_SOFTMAX && vec && row_pipe_plan<T, 2, CAUSAL>(rows, sk, &p))
            return launch_rowpipe(softmax_bwd_rowpipe<T, CAUSAL>, p, rows, s, gp, yp, dp, g, scale);
        auto k = softmax_bwd_warp<T, CAUSAL>;
        const int64_t need = (rows + kWarps - 1) / kWarps;
        const int64_t cap = (int64_t)sm_count() * blocks_per_sm((const void*)k);
        k<<<(unsigned)(need < cap ? need : cap), kThreads, 0, s>>>(gp, yp, dp, g, scale, vec);
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

unsigned take_device_error_softmax()
{
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess)
        return 0xFFu;
    if (v)
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    return v;
}

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
    const SoftmaxGeom g = make_geom(b * np * sq, sq, np, sk, mask ? mask_b : 1, mask ? mask_np : 1, mask ? mask_sq : 1);
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
    const SoftmaxGeom g = make_geom(attn_batches * sq, sq, 1, sq, 1, 1, 1);
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
