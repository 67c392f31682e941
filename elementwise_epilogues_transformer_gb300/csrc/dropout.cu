// dropout.cu -- fused bias + dropout + residual add, training and in-place
// inference.
//
// Megatron-LM operator fusion walkthrough (www.wmrh.cn/news/51426),
// §3.2-§3.3: _bias_dropout_add_func((x, bias), residual, prob, training)
// computes residual + dropout(x + bias); the residual is first cast to x's
// dtype; training and inference are separate entry points, and inference
// runs in place.
//
// Arithmetic is the fp32 sequence v = x + b; v = keep ? v * scale : 0;
// out = v + r~ with each step a separate IEEE rounding (explicit _rn
// intrinsics, so the compiler cannot contract them into an FMA) and one
// rounding to x's dtype at the store.  The keep mask comes from
// Philox4x32-10: element e = elem_base + i uses 16-bit word e % 8 of block
// e / 8 and is kept iff that word >= thresh.
//
// Memory per element (bf16 x, fp32 residual): training reads 2 + 4 bytes and
// writes 2 + 1 (mask); inference reads 2 + 4 and writes 2.
#include <cmath>

#include "mfx_device.cuh"
#include "mfx_host.h"
#include "mfx_pipe.cuh"

namespace mfx {
namespace {

// Timed-out waits of this file's pipelined kernels (see mfx_device_error).
__device__ unsigned g_device_error;

constexpr int kUnroll = MFX_UNROLL_BDA;

// The residual as x's dtype would hold it, widened back to fp32.
template <typename TX, typename TR>
__device__ __forceinline__ void cast_residual8(float r[8])
{
    if constexpr (DTypeInfo<TX>::kBf16 && !DTypeInfo<TR>::kBf16) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const uint32_t p = pack_bf16x2(r[j], r[j + 1]);
            r[j] = bf16lo(p);
            r[j + 1] = bf16hi(p);
        }
    }
}

// Dropout + residual on 8 elements whose keep words are w16(j).
template <bool TRAIN, typename WordFn>
__device__ __forceinline__ uint2 combine8(float v[8], const float b[8], const float r[8], float scale,
                                          uint32_t thresh, WordFn w16)
{
    uint32_t kb0 = 0, kb1 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float t = __fadd_rn(v[j], b[j]);
        if (TRAIN) {
            const bool keep = w16(j) >= thresh;
            t = keep ? __fmul_rn(t, scale) : 0.0f;
            if (j < 4)
                kb0 |= (uint32_t)keep << (8 * j);
            else
                kb1 |= (uint32_t)keep << (8 * (j - 4));
        }
        v[j] = __fadd_rn(t, r[j]);
    }
    return make_uint2(kb0, kb1);
}

// The keep bytes of a unit (0 or 1 each; bytes 0-3 in kb.x, 4-7 in kb.y) as
// the bits 0-7 of one byte.  x * 0x01020408 moves byte k's low bit to bit
// 24 + k and every other product term outside bits 24-27.
__device__ __forceinline__ uint32_t keep_bits8(uint2 kb)
{
    return ((kb.x * 0x01020408u) >> 24) | (((kb.y * 0x01020408u) >> 24) << 4);
}

// combine8 for bf16 x on packed pairs: the same three roundings per element
// (x + b, the scale, + r~), two elements per instruction.  xw: the unit's x
// as four bf16 pairs; rp: the cast residual as four pairs; blk: the unit's
// Philox block (16-bit word j keeps element j, compared here without
// extracting it: word j of a 32-bit word w is w << 16 for the low half and w
// for the high half, against thresh << 16).  Returns the output pairs in xw
// and the mask bytes.
template <bool TRAIN>
__device__ __forceinline__ uint2 combine8_pairs(uint32_t xw[4], const float b[8], const float2 rp[4], float scale,
                                                uint32_t thresh_hi, const uint4& blk)
{
    const uint32_t bw[4] = {blk.x, blk.y, blk.z, blk.w};
    uint32_t kb[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = add2(widen2(xw[i]), make_float2(b[2 * i], b[2 * i + 1]));
        if (TRAIN) {
            const float2 ts = mul2(t, f2(scale));
            const bool k0 = (bw[i] << 16) >= thresh_hi, k1 = bw[i] >= thresh_hi;
            t = make_float2(k0 ? ts.x : 0.0f, k1 ? ts.y : 0.0f);
            kb[i >> 1] |= (k0 ? 1u : 0u) << (16 * (i & 1)) | (k1 ? 1u : 0u) << (16 * (i & 1) + 8);
        }
        const float2 o = add2(t, rp[i]);
        xw[i] = pack_bf16x2(o.x, o.y);
    }
    return make_uint2(kb[0], kb[1]);
}

// ---------------------------------------------------------------------------
// Fixed-column kernel: cols % 8 == 0, elem_base % 8 == 0, 16-byte aligned
// x/out/residual/bias, 8-byte aligned mask, thread count a multiple of
// cols/8.  Unit u = elements [8u, 8u + 8) = exactly Philox block
// elem_base/8 + u, so one generator call serves the thread's 8 elements.
// ---------------------------------------------------------------------------
template <typename TX, typename TR, bool TRAIN>
__global__ void __launch_bounds__(kThreads, MFX_MINB_BDA)
bda_fixed(const TX* x, const TX* __restrict__ bias, const TR* __restrict__ res, TX* out,
          uint8_t* __restrict__ keep, int64_t units, int64_t cols, float scale, uint32_t thresh,
          uint64_t seed, uint64_t offset, uint64_t block_base)
{
    const int64_t S = (int64_t)gridDim.x * kThreads;
    int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    float b[8];
    bias8(bias, (u * 8) % cols, b);
    // warp k (< kUnroll) prefetches the block's k-th slice of the next iteration
    const int wk = threadIdx.x >> 5;
    const bool pf_warp = wk < kUnroll;
    const int64_t pf_off = (int64_t)(kUnroll + wk) * S - threadIdx.x;

    for (; u < units;) {
        const int nk = u + (kUnroll - 1) * S < units ? kUnroll : 1;
        prefetch_block_span<MFX_PREFETCH_BDA != 0>(x, u + pf_off, units, 8 * sizeof(TX), pf_warp);
        prefetch_block_span<MFX_PREFETCH_BDA != 0>(res, u + pf_off, units, 8 * sizeof(TR), pf_warp);
        Raw8<TX> rx[kUnroll];
        Raw8<TR> rr[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            if (k < nk) {
                ld8(x + (u + k * S) * 8, rx[k]);
                ld8(res + (u + k * S) * 8, rr[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            if (k < nk) {
                const int64_t uk = u + k * S;
                float v[8], r[8];
                widen8(rx[k], v);
                widen8(rr[k], r);
                cast_residual8<TX, TR>(r);
                uint4 blk = make_uint4(0, 0, 0, 0);
                if (TRAIN)
                    blk = mask_block(block_base + (uint64_t)uk, seed, offset);
                const uint2 kb = combine8<TRAIN>(v, b, r, scale, thresh,
                                                 [&](int j) { return word16(blk, j); });
                narrow8(v, rx[k]);
                st8(out + uk * 8, rx[k]);
                if (TRAIN)
                    st8(keep + uk * 8, kb);
            }
        }
        u += nk * S;
    }
}

// ---------------------------------------------------------------------------
// Pipelined fixed-column kernel.  Same unit ownership as bda_fixed (thread t
// of block b takes units b*256 + t + j*S, S = 256 * gridDim.x), but the
// block's 256-unit spans of x and the residual arrive in shared memory
// through a ring of NS stages of U spans each, filled by the producer warp
// with bulk copies; the consumers hold no data in flight.
// ---------------------------------------------------------------------------
// Spans per stage and ring size, per direction (measured: two 24.6 KB
// stages of bf16 x and fp32 residual for training, two blocks per SM; two
// spans per stage and four blocks per SM for inference, whose launch bounds
// ask for at least three).
// Training sizes its stages by bytes (as many 256-unit spans as fit
// MFX_BDA_STAGE_KB, at least one): measured, bf16 x with a bf16 residual
// runs 0.93 -> 0.98 of the copy peak with four spans (32 KB) instead of two,
// while bf16 x with an fp32 residual loses with more than two (24 KB).
template <typename TX, typename TR, bool TRAIN>
constexpr int pipe_u()
{
    constexpr int span = kConsumers * 8 * (int)(sizeof(TX) + sizeof(TR));
    return TRAIN ? (MFX_BDA_STAGE_KB * 1024 / span > 0 ? MFX_BDA_STAGE_KB * 1024 / span : 1)
                 : MFX_UNROLL_BDA_INF_PIPE;
}
template <typename TX, typename TR, bool TRAIN>
constexpr int pipe_stage_bytes()
{
    return pipe_u<TX, TR, TRAIN>() * kConsumers * 8 * (int)(sizeof(TX) + sizeof(TR));
}
template <typename TX, typename TR, bool TRAIN>
constexpr int pipe_stages()
{
    return ring_stages((TRAIN ? MFX_RING_KB_BDA : MFX_RING_KB_BDA_INF) * 1024, pipe_stage_bytes<TX, TR, TRAIN>());
}
template <typename TX, typename TR, bool TRAIN>
constexpr int pipe_smem_bytes()
{
    return kRingHeader + pipe_stages<TX, TR, TRAIN>() * pipe_stage_bytes<TX, TR, TRAIN>();
}
static_assert(pipe_smem_bytes<float, float, true>() <= (int)kMaxBlockSmem &&
                  pipe_smem_bytes<float, float, false>() <= (int)kMaxBlockSmem,
              "ring knobs: the stages do not fit in a block's shared memory");

// Elements [i0, i0 + cnt) one at a time (the first in column c and of
// global index e0), with the arithmetic of combine8: the head and tail of a
// pipelined call, whose elements are not whole 16-byte units.
// With PACKED the keep flags are bits of a bit mask and [i0, i0 + cnt) is
// one of its bytes (i0 % 8 == 0, cnt <= 8).
template <typename TX, typename TR, bool TRAIN, bool PACKED = false>
__device__ __forceinline__ void bda_elems(const TX* x, const TX* __restrict__ bias, const TR* __restrict__ res,
                                          TX* out, uint8_t* __restrict__ keep, int64_t i0, int cnt, int64_t c,
                                          int64_t cols, float scale, uint32_t thresh, uint64_t seed,
                                          uint64_t offset, uint64_t e0)
{
    uint32_t bits = 0;
    for (int j = 0; j < cnt; ++j) {
        float r = load1(res + i0 + j);
        if constexpr (DTypeInfo<TX>::kBf16 && !DTypeInfo<TR>::kBf16)
            r = round_to_bf16(r);
        float t = __fadd_rn(load1(x + i0 + j), bias1(bias, c));
        if (TRAIN) {
            const uint64_t e = e0 + (uint64_t)j;
            const bool kept = word16(mask_block(e >> 3, seed, offset), (int)(e & 7u)) >= thresh;
            t = kept ? __fmul_rn(t, scale) : 0.0f;
            if (PACKED)
                bits |= (uint32_t)kept << j;
            else
                keep[i0 + j] = (uint8_t)kept;
        }
        store1(out + i0 + j, __fadd_rn(t, r));
        if (++c == cols)
            c = 0;
    }
    if (TRAIN && PACKED && cnt > 0)
        keep[i0 / 8] = (uint8_t)bits;
}

// Any width and any common misalignment (see gelu_pipe): x, res, out and
// keep point at the 16-byte aligned body; unit u starts in column
// (c_off + 8u) mod cols and at global element 8 (block_base + u) + phase
// (its keep words: mask_block_at); S is the unit stride; the `head` elements
// before the body (global index e_head on) and the `tail` after its units
// are done one by one by thread 0 of block 0.
// With PACKED (training, no head) keep is a bit mask: unit u's flags are
// byte u.  PHASED (training, phase != 0) draws two generator blocks per unit;
// the other instances never carry that code.
template <typename TX, typename TR, bool TRAIN, bool PACKED = false, bool PHASED = false>
__global__ void __launch_bounds__(kPipeThreads, TRAIN ? MFX_PIPE_MINB_BDA_TRAIN : MFX_PIPE_MINB_BDA)
bda_pipe(const TX* x, const TX* __restrict__ bias, const TR* __restrict__ res, TX* out,
         uint8_t* __restrict__ keep, int64_t units, int64_t cols, float scale, uint32_t thresh,
         uint64_t seed, uint64_t offset, uint64_t block_base, int64_t S, int head, int tail, int64_t c_off,
         uint64_t e_head, int phase)
{
    constexpr int U = pipe_u<TX, TR, TRAIN>();
    constexpr int NS = pipe_stages<TX, TR, TRAIN>();
    constexpr uint32_t XB = kConsumers * 8 * sizeof(TX);  // one span of x
    constexpr uint32_t RB = kConsumers * 8 * sizeof(TR);  // one span of the residual
    constexpr uint32_t STAGE = U * (XB + RB);
    extern __shared__ __align__(128) unsigned char smem[];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    const int64_t ub0 = (int64_t)blockIdx.x * kConsumers;
    const int64_t iters = units > ub0 ? (units - ub0 + U * S - 1) / (U * S) : 0;
    const uint32_t active = S - ub0 < kConsumers ? (uint32_t)(S - ub0) : (uint32_t)kConsumers;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        // producer: one lane issues every copy
        if ((threadIdx.x & 31) == 0) {
            const void* const base[2] = {x, res};
            const uint32_t ub[2] = {8u * (uint32_t)sizeof(TX), 8u * (uint32_t)sizeof(TR)};
            const uint32_t off[2] = {0u, U * XB};
            flat_producer<NS, U, 2>(ring, data, STAGE, base, ub, off, ub0, S, units, iters, &g_device_error,
                                    active);
        }
        return;
    }

    // consumers
    const int t = threadIdx.x;
    const int64_t u0 = ub0 + t;
    const bool on = u0 < S;
    float b[8];
    bias8_at(bias, (c_off + (u0 % cols) * 8) % cols, cols, b);
    // PHASED: unit u needs generator blocks u and u + 1 (offset by block_base),
    // and block u + 1 is the first block of the unit one lane up.  Each lane
    // draws its first block; lane 31 takes the next warp's lane 0's from
    // shared memory, and the block's last lane also draws the block past
    // the block's units (slot kConsumerWarps).  One consumer-only barrier a
    // stage orders the writes and reads; the slots alternate between stages.
    // A consumer whose stage wait ran out keeps meeting the barrier (dead).
    __shared__ uint4 xch[PHASED ? 2 : 1][PHASED ? U : 1][kConsumerWarps + 1];
    bool dead = false;
    for (int64_t it = 0; it < iters; ++it) {
        // the mask does not depend on the data: generate it before waiting
        uint4 blks[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            blks[k] = !TRAIN                          ? make_uint4(0, 0, 0, 0)
                      : PHASED && !MFX_BDA_PHASED_SHARE ? mask_block_at(block_base + (uint64_t)(u0 + (it * U + k) * S),
                                                                         phase, seed, offset)
                                                         : mask_block(block_base + (uint64_t)(u0 + (it * U + k) * S),
                                                                      seed, offset);
        if constexpr (TRAIN && PHASED && MFX_BDA_PHASED_SHARE) {
            const int lane = t & 31, wp = t >> 5;
            uint4(*slot)[kConsumerWarps + 1] = xch[it & 1];
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < U; ++k)
                    slot[k][wp] = blks[k];
            }
            if (t == kConsumers - 1) {
#pragma unroll
                for (int k = 0; k < U; ++k)
                    slot[k][kConsumerWarps] =
                        mask_block(block_base + (uint64_t)(u0 + (it * U + k) * S) + 1, seed, offset);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
#pragma unroll
            for (int k = 0; k < U; ++k) {
                uint4 nx;
                nx.x = __shfl_down_sync(0xFFFFFFFFu, blks[k].x, 1);
                nx.y = __shfl_down_sync(0xFFFFFFFFu, blks[k].y, 1);
                nx.z = __shfl_down_sync(0xFFFFFFFFu, blks[k].z, 1);
                nx.w = __shfl_down_sync(0xFFFFFFFFu, blks[k].w, 1);
                if (lane == 31)
                    nx = slot[k][wp + 1];
                blks[k] = mask_words_at(blks[k], nx, phase);
            }
            if (dead)
                continue;
            if (!consumer_acquire<NS>(ring, it, &g_device_error)) {
                dead = true;
                continue;
            }
        } else if (!consumer_acquire<NS>(ring, it, &g_device_error)) {
            return;
        }
        const unsigned char* st = data + (size_t)(it % NS) * STAGE;
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t u = u0 + (it * U + k) * S;
            if (on && u < units) {
                Raw8<TX> rx;
                Raw8<TR> rr;
                lds8(st + k * XB + t * 8 * sizeof(TX), rx);
                lds8(st + U * XB + k * RB + t * 8 * sizeof(TR), rr);
                uint2 kb;
                if constexpr (DTypeInfo<TX>::kBf16 && MFX_BDA_PAIRED) {
                    float2 rp[4];
                    if constexpr (DTypeInfo<TR>::kBf16) {
                        rp[0] = widen2(rr.v.x), rp[1] = widen2(rr.v.y), rp[2] = widen2(rr.v.z), rp[3] = widen2(rr.v.w);
                    } else {
                        float r[8];
                        widen8(rr, r);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            rp[i] = widen2(pack_bf16x2(r[2 * i], r[2 * i + 1]));
                    }
                    uint32_t xw[4] = {rx.v.x, rx.v.y, rx.v.z, rx.v.w};
                    kb = combine8_pairs<TRAIN>(xw, b, rp, scale, thresh << 16, blks[k]);
                    rx.v = make_uint4(xw[0], xw[1], xw[2], xw[3]);
                } else {
                    float v[8], r[8];
                    widen8(rx, v);
                    widen8(rr, r);
                    cast_residual8<TX, TR>(r);
                    const uint4 blk = blks[k];
                    kb = combine8<TRAIN>(v, b, r, scale, thresh, [&](int j) { return word16(blk, j); });
                    narrow8(v, rx);
                }
                st8(out + u * 8, rx);
                if (TRAIN && PACKED)
                    keep[u] = (uint8_t)keep_bits8(kb);
                else if (TRAIN)
                    st8(keep + u * 8, kb);
            }
        }
        consumer_release<NS>(ring, it);
    }
    if (blockIdx.x == 0 && t == 0) {
        if (!PACKED)
            bda_elems<TX, TR, TRAIN>(x, bias, res, out, keep, -head, head, 0, cols, scale, thresh, seed, offset,
                                     e_head);
        bda_elems<TX, TR, TRAIN, PACKED>(x, bias, res, out, keep, units * 8, tail,
                                         (c_off + (units % cols) * 8) % cols, cols, scale, thresh, seed, offset,
                                         (block_base + (uint64_t)units) * 8 + phase);
    }
}

// ---------------------------------------------------------------------------
// Generic kernel: any width, alignment and elem_base.  Unit u = elements
// [8u, 8u + 8) of the call (the last may be short).  When elem_base % 8 = o
// is not 0 a unit straddles two generator blocks; element j then reads word
// (o + j) % 8 of block (elem_base + 8u) / 8 + (o + j) / 8.
// ---------------------------------------------------------------------------
template <typename TX, typename TR, bool TRAIN, bool PACKED = false>
__global__ void __launch_bounds__(kThreads)
bda_generic(const TX* x, const TX* __restrict__ bias, const TR* __restrict__ res, TX* out,
            uint8_t* __restrict__ keep, int64_t n, int64_t cols, int64_t dcol, float scale,
            uint32_t thresh, uint64_t seed, uint64_t offset, uint64_t elem_base, bool vec_x,
            bool vec_r, bool vec_m)
{
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t units = (n + 7) / 8;
    const int o = (int)(elem_base & 7u);
    int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    int64_t c = (u * 8) % cols;
    for (; u < units; u += S) {
        const int64_t i0 = u * 8;
        const int cnt = n - i0 < 8 ? (int)(n - i0) : 8;
        float v[8], r[8], b[8];
        load8f(x + i0, vec_x, cnt, v);
        load8f(res + i0, vec_r, cnt, r);
        cast_residual8<TX, TR>(r);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int64_t col = c + j;
            while (col >= cols)
                col -= cols;
            b[j] = bias1(bias, col);
        }
        uint4 blk0 = make_uint4(0, 0, 0, 0), blk1 = blk0;
        if (TRAIN) {
            const uint64_t j0 = (elem_base + (uint64_t)i0) >> 3;
            blk0 = mask_block(j0, seed, offset);
            blk1 = o ? mask_block(j0 + 1, seed, offset) : blk0;
        }
        const uint2 kb = combine8<TRAIN>(v, b, r, scale, thresh, [&](int j) {
            const int lane = o + j;
            return lane < 8 ? word16(blk0, lane) : word16(blk1, lane - 8);
        });
        store8f(out + i0, vec_x, cnt, v);
        if (TRAIN && PACKED) {
            keep[u] = (uint8_t)(keep_bits8(kb) & ((1u << cnt) - 1u));
        } else if (TRAIN) {
            if (vec_m && cnt == 8) {
                st8(keep + i0, kb);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < cnt)
                        keep[i0 + j] = (uint8_t)(((j < 4 ? kb.x : kb.y) >> (8 * (j & 3))) & 1u);
            }
        }
        c += dcol;
        if (c >= cols)
            c -= cols;
    }
}

// ---------------------------------------------------------------------------
// Backward (NEXT row f1): dx = keep ? g * scale : 0 in x's dtype, and
// optionally dres = g in the residual's dtype.  No column dependence, so the
// grid is a plain persistent one.  The mask is read from the forward's
// output (8 bytes per unit, streamed through the ring with g) or
// regenerated from Philox exactly as the forward drew it (no mask traffic).
// ---------------------------------------------------------------------------
template <typename TX, bool MASK, bool PACKED = false>
struct BwdPipe {
    static constexpr int kU = MFX_UNROLL_BDA_BWD * 2 / (int)sizeof(TX) > 0  // bf16 spans; halved for fp32
                                  ? MFX_UNROLL_BDA_BWD * 2 / (int)sizeof(TX) : 1;
    static constexpr uint32_t kSpan = kConsumers * 8 * sizeof(TX);
    static constexpr uint32_t kMaskUnit = PACKED ? 1 : 8;  // bytes of a read keep mask per unit
    static constexpr uint32_t kMaskSpan = MASK ? kConsumers * kMaskUnit : 0;
    static constexpr uint32_t kStage = kU * (kSpan + kMaskSpan);
    static constexpr int kStages = ring_stages(MFX_RING_KB_BDA_BWD * 1024, kStage);
    static constexpr size_t kSmem = kRingHeader + (size_t)kStages * kStage;
    static_assert(kSmem <= kMaxBlockSmem, "ring knobs: the stages do not fit in a block's shared memory");
};

template <typename TR>
__device__ __forceinline__ void store_dres8(TR* p, const float f[8])
{
    Raw8<TR> r;
    narrow8(f, r);
    st8(p, r);
}

// dres = g widened to fp32, stored by a warp over its 32 units (256
// elements) as two 512-byte runs: lane l of pass j takes elements
// [4 (32 j + l), +4), read from the staged g.  Stores of thread-owned units
// (8 fp32, 32 bytes) would write every 32-byte sector in two halves from
// two instructions; these write whole sectors.  `wspan` is the warp's g in
// the stage, `ubw` its first unit.
template <typename TX>
__device__ __forceinline__ void store_dres_warp(float* dres, int64_t ubw, int64_t units, const unsigned char* wspan)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int q = j * 32 + lane;  // 4-element quarter of the warp's units
        if (ubw + (q >> 1) < units) {
            uint4 v;
            if constexpr (DTypeInfo<TX>::kBf16) {
                const uint2 w = *reinterpret_cast<const uint2*>(wspan + q * 8);
                v = make_uint4(w.x << 16, w.x & 0xFFFF0000u, w.y << 16, w.y & 0xFFFF0000u);
            } else {
                v = *reinterpret_cast<const uint4*>(wspan + q * 16);
            }
            st16(dres + ubw * 8 + q * 4, v);
        }
    }
}

// Output slots of the bulk-store form: per consumer warp MFX_BDA_BWD_SLOTS
// slots, each the warp's 32 units of dx then of dres; a warp fills one while
// the copy engine still reads the others.  The form serves the byte-mask
// backward alone: at the D2 layer shape it lifts that kernel from 0.86 to
// 0.90 of the copy peak, where the regenerated-mask form (more ALU work per
// unit, two blocks per SM needed) fell from 0.84 to 0.81 and the bit-mask
// form gained nothing.
constexpr bool bwd_bulk_stores(bool regen, bool db, bool packed)
{
    return MFX_BDA_BWD_BULK_ST && !regen && !db && !packed;
}
template <typename TX, typename TR>
struct BwdOut {
    static constexpr uint32_t kDx = 32 * 8 * sizeof(TX), kDr = 32 * 8 * sizeof(TR);
    static constexpr uint32_t kSlot = kDx + kDr;
    static constexpr size_t kBytes = (size_t)kConsumerWarps * MFX_BDA_BWD_SLOTS * kSlot;
};

// dres of a warp's 32 units into its slot: fp32 from bf16 g by 4-element
// quarters read from the staged g (lane l of pass j takes quarter 32 j + l,
// so a warp's 16-byte shared stores are contiguous), otherwise by units from
// the thread's widened g.
template <typename TX, typename TR>
__device__ __forceinline__ void dres_to_slot(unsigned char* sd, const unsigned char* wspan, const float gv[8],
                                             int lane)
{
    if constexpr (DTypeInfo<TX>::kBf16 && !DTypeInfo<TR>::kBf16) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int q = j * 32 + lane;
            const uint2 w = *reinterpret_cast<const uint2*>(wspan + q * 8);
            *reinterpret_cast<uint4*>(sd + q * 16) = make_uint4(w.x << 16, w.x & 0xFFFF0000u, w.y << 16,
                                                                w.y & 0xFFFF0000u);
        }
    } else {
        Raw8<TR> r;
        narrow8(gv, r);
        stl8(sd + lane * 8 * sizeof(TR), r);
    }
}

// With DB the grid is a fixed-column one (thread count a multiple of
// cols / 8) and each consumer adds the dx values it stores into partial
// column sums written to ws[lane][columns], lane = first unit / (cols / 8).
// With PACKED the read mask is a bit mask: unit u's flags are byte u.
template <typename TX, typename TR, bool REGEN, bool DB = false, bool PACKED = false>
__global__ void __launch_bounds__(kPipeThreads, MFX_PIPE_MINB_BDA_BWD)
bda_bwd_pipe(const TX* g, const uint8_t* __restrict__ keep, TX* dx, TR* dres, int64_t units, float scale,
             uint32_t thresh, uint64_t seed, uint64_t offset, uint64_t block_base, int64_t cols = 0,
             float* __restrict__ ws = nullptr)
{
    using P = BwdPipe<TX, !REGEN, PACKED>;
    using BO = BwdOut<TX, TR>;
    constexpr int U = P::kU, NS = P::kStages;
    // byte mask read: outputs by bulk stores out of per-warp slots (after
    // the ring); the other forms measured faster with register stores
    constexpr bool kBulk = bwd_bulk_stores(REGEN, DB, PACKED);
    extern __shared__ __align__(128) unsigned char smem[];
    const Ring ring = ring_setup<NS>(smem);
    unsigned char* data = smem + kRingHeader;
    unsigned char* obuf = data + (size_t)NS * P::kStage;
    const int64_t S = (int64_t)gridDim.x * kConsumers;
    const int64_t ub0 = (int64_t)blockIdx.x * kConsumers;
    const int64_t iters = units > ub0 ? (units - ub0 + U * S - 1) / (U * S) : 0;

    if ((threadIdx.x >> 5) == kConsumerWarps) {
        if ((threadIdx.x & 31) == 0) {
            if (REGEN) {
                const void* const base[1] = {g};
                const uint32_t ub[1] = {8u * (uint32_t)sizeof(TX)};
                const uint32_t off[1] = {0u};
                flat_producer<NS, U, 1>(ring, data, P::kStage, base, ub, off, ub0, S, units, iters, &g_device_error);
            } else {
                // the mask comes through the ring too, after the g spans
                const void* const base[2] = {g, keep};
                const uint32_t ub[2] = {8u * (uint32_t)sizeof(TX), P::kMaskUnit};
                const uint32_t off[2] = {0u, U * P::kSpan};
                flat_producer<NS, U, 2>(ring, data, P::kStage, base, ub, off, ub0, S, units, iters, &g_device_error);
            }
        }
        return;
    }
    const int t = threadIdx.x;
    const int lane = t & 31, wb = t & ~31;
    const int64_t u0 = ub0 + t;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc[j] = 0.0f;
    uint32_t sl = 0;  // bulk form: the warp's next slot
    for (int64_t it = 0; it < iters; ++it) {
        // a regenerated mask is computed before the stage wait; a read one
        // comes through the ring (except an odd last unit, read directly)
        uint32_t kw[U][2];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t u = u0 + (it * U + k) * S;
            kw[k][0] = kw[k][1] = 0;
            if (REGEN) {
                const uint4 blk = mask_block(block_base + (uint64_t)u, seed, offset);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    kw[k][j >> 2] |= (uint32_t)(word16(blk, j) >= thresh) << (8 * (j & 3));
            } else if (u < units && (uint32_t)t >= copied_units((uint32_t)(units - (u - t) < kConsumers
                                                                                ? units - (u - t) : kConsumers),
                                                                  P::kMaskUnit)) {
                // the last units of the call's last span are not in the ring
                if (PACKED) {
                    kw[k][0] = keep[u];
                } else {
                    const uint2 m = *reinterpret_cast<const uint2*>(keep + u * 8);
                    kw[k][0] = m.x;
                    kw[k][1] = m.y;
                }
            }
        }
        if (!consumer_acquire<NS>(ring, it, &g_device_error)) {
            if (kBulk && lane == 0)
                bulk_wait_all();
            return;
        }
        const unsigned char* st = data + (size_t)(it % NS) * P::kStage + t * 8 * sizeof(TX);
        if (!REGEN) {
            const unsigned char* sm = data + (size_t)(it % NS) * P::kStage + U * P::kSpan + t * P::kMaskUnit;
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int64_t u = u0 + (it * U + k) * S;
                if (u < units && (uint32_t)t < copied_units((uint32_t)(units - (u - t) < kConsumers
                                                                          ? units - (u - t) : kConsumers),
                                                            P::kMaskUnit)) {
                    if (PACKED) {
                        kw[k][0] = sm[k * P::kMaskSpan];
                    } else {
                        const uint2 m = *reinterpret_cast<const uint2*>(sm + k * P::kMaskSpan);
                        kw[k][0] = m.x;
                        kw[k][1] = m.y;
                    }
                }
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t u = u0 + (it * U + k) * S;
            if constexpr (kBulk) {
                const int64_t first = u - lane;  // the warp's first unit
                if (first >= units)
                    continue;
                const uint32_t nv = units - first < 32 ? (uint32_t)(units - first) : 32u;
                unsigned char* slot = obuf + (size_t)((wb >> 5) * MFX_BDA_BWD_SLOTS + sl) * BO::kSlot;
                sl = sl + 1 == MFX_BDA_BWD_SLOTS ? 0u : sl + 1;
                if (lane == 0)
                    bulk_wait_read<MFX_BDA_BWD_SLOTS - 1>();  // the slot's previous copies have read it
                __syncwarp();
                float gv[8];
                if (u < units) {
                    Raw8<TX> rg;
                    lds8(st + k * P::kSpan, rg);
                    float d[8];
                    widen8(rg, gv);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        d[j] = (PACKED ? (kw[k][0] >> j) & 1u : (kw[k][j >> 2] >> (8 * (j & 3))) & 0xFFu)
                                   ? __fmul_rn(gv[j], scale)
                                   : 0.0f;
                    narrow8(d, rg);
                    stl8(slot + lane * 8 * sizeof(TX), rg);
                }
                if (dres)
                    dres_to_slot<TX, TR>(slot + BO::kDx,
                                         data + (size_t)(it % NS) * P::kStage + k * P::kSpan + wb * 8 * sizeof(TX),
                                         gv, lane);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    bulk_s2g(dx + first * 8, smem_addr(slot), nv * 8 * (uint32_t)sizeof(TX));
                    if (dres)
                        bulk_s2g(dres + first * 8, smem_addr(slot + BO::kDx), nv * 8 * (uint32_t)sizeof(TR));
                    bulk_commit();
                }
                continue;
            }
            if (u < units) {
                Raw8<TX> rg;
                lds8(st + k * P::kSpan, rg);
                float gv[8], d[8];
                widen8(rg, gv);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    d[j] = (PACKED ? (kw[k][0] >> j) & 1u : (kw[k][j >> 2] >> (8 * (j & 3))) & 0xFFu)
                               ? __fmul_rn(gv[j], scale)
                               : 0.0f;
                narrow8(d, rg);
                st8(dx + u * 8, rg);
                if (DTypeInfo<TR>::kBf16 && dres)  // fp32 dres: whole-sector runs below
                    store_dres8(dres + u * 8, gv);
                if (DB) {
                    widen8(rg, d);  // the stored values
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[j] += d[j];
                }
            }
        }
        if constexpr (!DTypeInfo<TR>::kBf16 && !kBulk) {
            if (dres) {
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const int wb = t & ~31;
                    store_dres_warp<TX>(reinterpret_cast<float*>(dres), ub0 + wb + (it * U + k) * S, units,
                                        data + (size_t)(it % NS) * P::kStage + k * P::kSpan + wb * 8 * sizeof(TX));
                }
            }
        }
        consumer_release<NS>(ring, it);
    }
    if (kBulk && lane == 0)
        bulk_wait_all();
    if (DB) {
        pdl_launch_dependents();
        const int64_t gpr = cols / 8;
        float4* w4 = reinterpret_cast<float4*>(ws + (u0 / gpr) * cols + (u0 % gpr) * 8);
        w4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        w4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// Generic backward: any alignment, length and elem_base (units of up to 8
// elements; a unit may straddle two generator blocks, as in bda_generic).
template <typename TX, typename TR, bool PACKED = false>
__global__ void __launch_bounds__(kThreads)
bda_bwd_generic(const TX* g, const uint8_t* keep, TX* dx, TR* dres, int64_t n, float scale, uint32_t thresh,
                uint64_t seed, uint64_t offset, uint64_t elem_base)
{
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t units = (n + 7) / 8;
    const int o = (int)(elem_base & 7u);
    for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < units; u += S) {
        const int64_t i0 = u * 8;
        const int cnt = n - i0 < 8 ? (int)(n - i0) : 8;
        float gv[8], d[8];
        load8f(g + i0, false, cnt, gv);
        uint4 blk0 = make_uint4(0, 0, 0, 0), blk1 = blk0;
        if (!keep) {
            const uint64_t j0 = (elem_base + (uint64_t)i0) >> 3;
            blk0 = mask_block(j0, seed, offset);
            blk1 = o ? mask_block(j0 + 1, seed, offset) : blk0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            bool k = false;
            if (j < cnt) {
                if (keep) {
                    k = PACKED ? (keep[u] >> j) & 1u : keep[i0 + j] != 0;
                } else {
                    const int lane = o + j;
                    k = (lane < 8 ? word16(blk0, lane) : word16(blk1, lane - 8)) >= thresh;
                }
            }
            d[j] = k ? __fmul_rn(gv[j], scale) : 0.0f;
        }
        store8f(dx + i0, false, cnt, d);
        if (dres)
            store8f(dres + i0, false, cnt, gv);
    }
}

template <typename TX, typename TR, bool PACKED = false>
int launch_bwd(const void* g, const uint8_t* keep, void* dx, void* dres, int64_t n, float p, uint64_t seed,
               uint64_t offset, uint64_t elem_base, cudaStream_t s)
{
    const TX* gp = static_cast<const TX*>(g);
    TX* dxp = static_cast<TX*>(dx);
    TR* drp = static_cast<TR*>(dres);
    double t = std::ceil((double)p * 65536.0);
    const uint32_t thresh = (uint32_t)(t > 65535.0 ? 65535.0 : t);
    const float scale = 1.0f / (1.0f - p);
    const bool pipe_ok = MFX_PIPE_BDA && n % 8 == 0 && aligned16(g) && aligned16(dx) &&
                         (!dres || aligned16(dres)) && (keep ? aligned16(keep) : elem_base % 8 == 0);
    if (pipe_ok) {
        const int64_t units = n / 8;
        if (keep) {
            constexpr size_t kOut = bwd_bulk_stores(false, false, PACKED) ? BwdOut<TX, TR>::kBytes : 0;
            constexpr size_t smem = BwdPipe<TX, true, PACKED>::kSmem + kOut;
            static_assert(smem <= kMaxBlockSmem, "ring and output slots do not fit in a block's shared memory");
            const Grid grid = plan_grid_ex((const void*)bda_bwd_pipe<TX, TR, false, false, PACKED>, kPipeThreads,
                                           smem, units, 0, false);
            bda_bwd_pipe<TX, TR, false, false, PACKED><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                gp, keep, dxp, drp, units, scale, thresh, seed, offset, 0);
        } else {
            constexpr size_t smem = BwdPipe<TX, false>::kSmem;
            const Grid grid = plan_grid_ex((const void*)bda_bwd_pipe<TX, TR, true>, kPipeThreads, smem, units, 0, false);
            bda_bwd_pipe<TX, TR, true><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                gp, nullptr, dxp, drp, units, scale, thresh, seed, offset, elem_base / 8);
        }
        return launch_status();
    }
    const Grid grid = plan_grid((const void*)bda_bwd_generic<TX, TR, PACKED>, (n + 7) / 8, 0, false);
    bda_bwd_generic<TX, TR, PACKED><<<(unsigned)grid.blocks, kThreads, 0, s>>>(gp, keep, dxp, drp, n, scale, thresh,
                                                                               seed, offset, elem_base);
    return launch_status();
}

// Backward plus the fused bias gradient.
template <typename TX, typename TR>
int launch_bwd_dbias(const void* g, const uint8_t* keep, void* dx, void* dres, void* dbias, int64_t rows,
                     int64_t cols, float p, uint64_t seed, uint64_t offset, uint64_t elem_base, void* workspace,
                     size_t* ws_bytes, cudaStream_t s)
{
    const int64_t n = rows * cols;
    const size_t smem = keep ? BwdPipe<TX, true>::kSmem : BwdPipe<TX, false>::kSmem;
    const void* k = keep ? (const void*)bda_bwd_pipe<TX, TR, false, true> : (const void*)bda_bwd_pipe<TX, TR, true, true>;
    int64_t J_pipe = 0;
    Grid grid;
    if (MFX_PIPE_BDA && cols % 8 == 0) {
        grid = plan_grid_ex(k, kPipeThreads, smem, n / 8, cols / 8, true);
        if (grid.fixed)
            J_pipe = grid.blocks * kThreads / (cols / 8);
    }
    const int64_t J_gen = dbias_generic_lanes(rows);
    bool query = false;
    int st = dbias_workspace(J_pipe > J_gen ? J_pipe : J_gen, cols, workspace, ws_bytes, &query);
    if (st != MFX_OK || query)
        return st;
    float* ws = static_cast<float*>(workspace);
    const bool pipe_ok = J_pipe > 0 && aligned16(g) && aligned16(dx) && (!dres || aligned16(dres)) &&
                         (keep ? aligned16(keep) : elem_base % 8 == 0);
    if (pipe_ok) {
        double t = std::ceil((double)p * 65536.0);
        const uint32_t thresh = (uint32_t)(t > 65535.0 ? 65535.0 : t);
        const float scale = 1.0f / (1.0f - p);
        const TX* gp = static_cast<const TX*>(g);
        if (keep)
            bda_bwd_pipe<TX, TR, false, true><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                gp, keep, static_cast<TX*>(dx), static_cast<TR*>(dres), n / 8, scale, thresh, seed, offset, 0,
                cols, ws);
        else
            bda_bwd_pipe<TX, TR, true, true><<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                gp, nullptr, static_cast<TX*>(dx), static_cast<TR*>(dres), n / 8, scale, thresh, seed, offset,
                elem_base / 8, cols, ws);
        st = launch_status();
        return st != MFX_OK ? st : launch_dbias_finish(dtype_code<TX>(), ws, J_pipe, cols, dbias, s);
    }
    st = launch_bwd<TX, TR>(g, keep, dx, dres, n, p, seed, offset, elem_base, s);
    if (st == MFX_OK)
        st = launch_column_partials(dtype_code<TX>(), dx, rows, cols, J_gen, ws, s);
    return st != MFX_OK ? st : launch_dbias_finish(dtype_code<TX>(), ws, J_gen, cols, dbias, s);
}

template <typename TX, typename TR, bool TRAIN, bool PACKED = false>
int launch(const void* x, const void* bias, const void* res, void* out, uint8_t* keep, int64_t n,
           int64_t cols, float p, uint64_t seed, uint64_t offset, uint64_t elem_base, cudaStream_t s)
{
    const TX* xp = static_cast<const TX*>(x);
    const TX* bp = static_cast<const TX*>(bias);
    const TR* rp = static_cast<const TR*>(res);
    TX* op = static_cast<TX*>(out);
    // keep iff u16 >= min(65535, ceil(p * 65536)); inverted-dropout scale in fp32
    double t = std::ceil((double)p * 65536.0);
    const uint32_t thresh = TRAIN ? (uint32_t)(t > 65535.0 ? 65535.0 : t) : 0u;
    const float scale = TRAIN ? 1.0f / (1.0f - p) : 1.0f;
    const bool vec_x = aligned16(x) && aligned16(out);
    const bool vec_r = aligned16(res);
    const bool vec_m = !TRAIN || aligned8(keep);
    const bool fixed_ok = vec_x && vec_r && vec_m && cols % 8 == 0 && elem_base % 8 == 0 &&
                          (!bias || aligned16(bias));
    // the pipeline takes any width when x, out and the residual sit the same
    // whole number of elements below a 16-byte boundary (those elements are
    // its head) and the mask too below an 8-byte one; a body that does not
    // start on a generator block draws two blocks per unit
    const uintptr_t mis = reinterpret_cast<uintptr_t>(x) & 15u;
    const int head = (int)(((16u - mis) & 15u) / sizeof(TX));
    // (a bit mask takes the pipeline without a head: its units are its bytes)
    const bool same = mis % sizeof(TX) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == mis &&
                      ((reinterpret_cast<uintptr_t>(res) + head * sizeof(TR)) & 15u) == 0 &&
                      (!TRAIN || PACKED || ((reinterpret_cast<uintptr_t>(keep) + head) & 7u) == 0) &&
                      (!PACKED || head == 0);
    if (same && MFX_PIPE_BDA && n - head >= 8) {
        const int phase = TRAIN ? (int)((elem_base + head) % 8) : 0;
        const auto kern = phase ? bda_pipe<TX, TR, TRAIN, PACKED, true> : bda_pipe<TX, TR, TRAIN, PACKED, false>;
        constexpr size_t smem = pipe_smem_bytes<TX, TR, TRAIN>();
        const int64_t units = (n - head) / 8;
        const Grid grid = plan_fixed_any((const void*)kern, kPipeThreads, smem, units, cols);
        if (grid.fixed) {
            kern<<<(unsigned)grid.blocks, kPipeThreads, smem, s>>>(
                xp + head, bp, rp + head, op + head, TRAIN ? keep + head : keep, units, cols, scale, thresh, seed,
                offset, (elem_base + head) / 8, grid.S, head, (int)((n - head) % 8), head % cols, elem_base, phase);
            return launch_status();
        }
    }
    if (fixed_ok && !PACKED) {
        const Grid grid = plan_grid((const void*)bda_fixed<TX, TR, TRAIN>, n / 8, cols / 8, true);
        if (grid.fixed) {
            bda_fixed<TX, TR, TRAIN><<<(unsigned)grid.blocks, kThreads, 0, s>>>(
                xp, bp, rp, op, keep, n / 8, cols, scale, thresh, seed, offset, elem_base / 8);
            return launch_status();
        }
    }
    const Grid grid = plan_grid((const void*)bda_generic<TX, TR, TRAIN, PACKED>, (n + 7) / 8, 0, false);
    const int64_t dcol = (grid.blocks * kThreads * 8) % cols;
    bda_generic<TX, TR, TRAIN, PACKED><<<(unsigned)grid.blocks, kThreads, 0, s>>>(
        xp, bp, rp, op, keep, n, cols, dcol, scale, thresh, seed, offset, elem_base, vec_x, vec_r, vec_m);
    return launch_status();
}

template <bool TRAIN, bool PACKED = false>
int dispatch(int x_dt, int r_dt, const void* x, const void* bias, const void* res, void* out,
             uint8_t* keep, int64_t n, int64_t cols, float p, uint64_t seed, uint64_t offset,
             uint64_t elem_base, cudaStream_t s)
{
    if (x_dt == MFX_BF16)
        return r_dt == MFX_BF16
                   ? launch<bf16, bf16, TRAIN, PACKED>(x, bias, res, out, keep, n, cols, p, seed, offset, elem_base, s)
                   : launch<bf16, float, TRAIN, PACKED>(x, bias, res, out, keep, n, cols, p, seed, offset, elem_base,
                                                        s);
    return r_dt == MFX_BF16
               ? launch<float, bf16, TRAIN, PACKED>(x, bias, res, out, keep, n, cols, p, seed, offset, elem_base, s)
               : launch<float, float, TRAIN, PACKED>(x, bias, res, out, keep, n, cols, p, seed, offset, elem_base, s);
}

int check(int x_dt, int r_dt, int64_t rows, int64_t cols, float p, int64_t* n_out)
{
    *n_out = 0;
    if (!valid_dtype(x_dt) || !valid_dtype(r_dt))
        return MFX_ERR_DTYPE;
    if (!(p >= 0.0f && p < 1.0f))  // also rejects NaN
        return MFX_ERR_PROB;
    if (rows < 0 || cols < 0)
        return MFX_ERR_SHAPE;
    int64_t n = 0, bytes = 0;
    if (!mul_ok(rows, cols, &n) || !mul_ok(n, 16, &bytes))
        return MFX_ERR_SHAPE;
    *n_out = n;
    return MFX_OK;
}

}  // namespace

unsigned take_device_error_dropout()
{
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess)
        return 0xFFu;
    if (v)
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    return v;
}

}  // namespace mfx

extern "C" int mfx_bias_dropout_add_train(int x_dt, int res_dt, int64_t rows, int64_t cols,
                                          const void* x, const void* bias, const void* residual,
                                          float p, uint64_t seed, uint64_t offset,
                                          uint64_t elem_base, void* out, uint8_t* keep_mask,
                                          void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(x_dt, res_dt, rows, cols, p, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!x || !residual || !out || !keep_mask)
        return MFX_ERR_NULL;
    if (elem_base > UINT64_MAX - (uint64_t)n)
        return MFX_ERR_SHAPE;
    const int64_t xe = dtype_bytes(x_dt), re = dtype_bytes(res_dt);
    const int64_t xb = n * xe, rb = n * re, bb = cols * xe;
    if (partial_overlap(x, xb, out, xb) || overlaps(residual, rb, out, xb) ||
        overlaps(bias, bb, out, xb) || overlaps(keep_mask, n, out, xb) ||
        overlaps(keep_mask, n, x, xb) || overlaps(keep_mask, n, residual, rb) ||
        overlaps(keep_mask, n, bias, bb))
        return MFX_ERR_ALIAS;
    return dispatch<true>(x_dt, res_dt, x, bias, residual, out, keep_mask, n, cols, p, seed, offset,
                          elem_base, static_cast<cudaStream_t>(stream));
}

namespace mfx {
namespace {
// Null and overlap checks of the backward (nonempty shapes).
// mask_bytes: the mask's size (n for the byte mask, ceil(n / 8) for bits).
int bwd_check(int x_dt, int res_dt, int64_t n, const void* g, const uint8_t* keep_mask, uint64_t elem_base,
              void* dx, void* dresidual, int64_t mask_bytes)
{
    if (!g || !dx)
        return MFX_ERR_NULL;
    if (!keep_mask && elem_base > UINT64_MAX - (uint64_t)n)
        return MFX_ERR_SHAPE;
    const int64_t xe = dtype_bytes(x_dt), re = dtype_bytes(res_dt);
    const int64_t xb = n * xe, rb = n * re;
    if (partial_overlap(g, xb, dx, xb) || overlaps(keep_mask, mask_bytes, dx, xb) ||
        overlaps(dresidual, rb, dx, xb) || overlaps(dresidual, rb, keep_mask, mask_bytes) ||
        (dresidual != g && overlaps(dresidual, rb, g, xb)))
        return MFX_ERR_ALIAS;
    if (dresidual == g && (res_dt != x_dt || dx == g))
        return MFX_ERR_ALIAS;
    return MFX_OK;
}
}  // namespace
}  // namespace mfx

extern "C" int mfx_bias_dropout_add_bwd(int x_dt, int res_dt, int64_t rows, int64_t cols, const void* g,
                                        const uint8_t* keep_mask, float p, uint64_t seed, uint64_t offset,
                                        uint64_t elem_base, void* dx, void* dresidual, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(x_dt, res_dt, rows, cols, p, &n);
    if (st != MFX_OK || n == 0)
        return st;
    st = bwd_check(x_dt, res_dt, n, g, keep_mask, elem_base, dx, dresidual, n);
    if (st != MFX_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* dr = dresidual == g ? nullptr : dresidual;  // same buffer, same dtype: already holds g
    if (x_dt == MFX_BF16)
        return res_dt == MFX_BF16 ? launch_bwd<bf16, bf16>(g, keep_mask, dx, dr, n, p, seed, offset, elem_base, s)
                                  : launch_bwd<bf16, float>(g, keep_mask, dx, dr, n, p, seed, offset, elem_base, s);
    return res_dt == MFX_BF16 ? launch_bwd<float, bf16>(g, keep_mask, dx, dr, n, p, seed, offset, elem_base, s)
                              : launch_bwd<float, float>(g, keep_mask, dx, dr, n, p, seed, offset, elem_base, s);
}

extern "C" int mfx_bias_dropout_add_train_packed(int x_dt, int res_dt, int64_t rows, int64_t cols,
                                                 const void* x, const void* bias, const void* residual, float p,
                                                 uint64_t seed, uint64_t offset, uint64_t elem_base, void* out,
                                                 uint8_t* keep_bits, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(x_dt, res_dt, rows, cols, p, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!x || !residual || !out || !keep_bits)
        return MFX_ERR_NULL;
    if (elem_base > UINT64_MAX - (uint64_t)n)
        return MFX_ERR_SHAPE;
    const int64_t xe = dtype_bytes(x_dt), re = dtype_bytes(res_dt);
    const int64_t xb = n * xe, rb = n * re, bb = cols * xe, mb = (n + 7) / 8;
    if (partial_overlap(x, xb, out, xb) || overlaps(residual, rb, out, xb) || overlaps(bias, bb, out, xb) ||
        overlaps(keep_bits, mb, out, xb) || overlaps(keep_bits, mb, x, xb) || overlaps(keep_bits, mb, residual, rb) ||
        overlaps(keep_bits, mb, bias, bb))
        return MFX_ERR_ALIAS;
    return dispatch<true, true>(x_dt, res_dt, x, bias, residual, out, keep_bits, n, cols, p, seed, offset,
                                elem_base, static_cast<cudaStream_t>(stream));
}

extern "C" int mfx_bias_dropout_add_bwd_packed(int x_dt, int res_dt, int64_t rows, int64_t cols, const void* g,
                                               const uint8_t* keep_bits, float p, void* dx, void* dresidual,
                                               void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(x_dt, res_dt, rows, cols, p, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!keep_bits)
        return MFX_ERR_NULL;
    st = bwd_check(x_dt, res_dt, n, g, keep_bits, 0, dx, dresidual, (n + 7) / 8);
    if (st != MFX_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* dr = dresidual == g ? nullptr : dresidual;
    if (x_dt == MFX_BF16)
        return res_dt == MFX_BF16 ? launch_bwd<bf16, bf16, true>(g, keep_bits, dx, dr, n, p, 0, 0, 0, s)
                                  : launch_bwd<bf16, float, true>(g, keep_bits, dx, dr, n, p, 0, 0, 0, s);
    return res_dt == MFX_BF16 ? launch_bwd<float, bf16, true>(g, keep_bits, dx, dr, n, p, 0, 0, 0, s)
                              : launch_bwd<float, float, true>(g, keep_bits, dx, dr, n, p, 0, 0, 0, s);
}

extern "C" int mfx_bias_dropout_add_inference(int x_dt, int res_dt, int64_t rows, int64_t cols,
                                              void* x, const void* bias, const void* residual,
                                              float p, uint64_t seed, uint64_t offset, void* stream)
{
    using namespace mfx;
    (void)seed;
    (void)offset;
    int64_t n = 0;
    int st = check(x_dt, res_dt, rows, cols, p, &n);
    if (st != MFX_OK || n == 0)
        return st;
    if (!x || !residual)
        return MFX_ERR_NULL;
    const int64_t xe = dtype_bytes(x_dt), re = dtype_bytes(res_dt);
    const int64_t xb = n * xe, rb = n * re, bb = cols * xe;
    if (overlaps(residual, rb, x, xb) || overlaps(bias, bb, x, xb))
        return MFX_ERR_ALIAS;
    return dispatch<false>(x_dt, res_dt, x, bias, residual, x, nullptr, n, cols, 0.0f, 0, 0, 0,
                           static_cast<cudaStream_t>(stream));
}

extern "C" int mfx_bias_dropout_add_bwd_dbias(int x_dt, int res_dt, int64_t rows, int64_t cols, const void* g,
                                              const uint8_t* keep_mask, float p, uint64_t seed, uint64_t offset,
                                              uint64_t elem_base, void* dx, void* dresidual, void* dbias,
                                              void* workspace, size_t* workspace_bytes, void* stream)
{
    using namespace mfx;
    int64_t n = 0;
    int st = check(x_dt, res_dt, rows, cols, p, &n);
    if (st != MFX_OK)
        return st;
    if (!workspace_bytes)
        return MFX_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t xe = dtype_bytes(x_dt);
    if (n == 0) {
        if (!workspace) {
            *workspace_bytes = 0;
            return MFX_OK;
        }
        if (cols == 0)
            return MFX_OK;
        if (!dbias)
            return MFX_ERR_NULL;
        return cudaMemsetAsync(dbias, 0, (size_t)(cols * xe), s) == cudaSuccess ? MFX_OK
                                                                               : cuda_failure(cudaGetLastError());
    }
    if (workspace) {
        st = bwd_check(x_dt, res_dt, n, g, keep_mask, elem_base, dx, dresidual, n);
        if (st != MFX_OK)
            return st;
        if (!dbias)
            return MFX_ERR_NULL;
        const int64_t xb = n * xe, re = dtype_bytes(res_dt), wsb = (int64_t)*workspace_bytes;
        if (overlaps(dbias, cols * xe, dx, xb) || overlaps(dbias, cols * xe, g, xb) ||
            overlaps(dbias, cols * xe, keep_mask, n) || overlaps(dbias, cols * xe, dresidual, n * re) ||
            overlaps(workspace, wsb, dx, xb) || overlaps(workspace, wsb, g, xb) || overlaps(workspace, wsb, keep_mask, n) ||
            overlaps(workspace, wsb, dresidual, n * re) || overlaps(workspace, wsb, dbias, cols * xe))
            return MFX_ERR_ALIAS;
    }
    void* dr = dresidual == g ? nullptr : dresidual;
    if (x_dt == MFX_BF16)
        return res_dt == MFX_BF16
                   ? launch_bwd_dbias<bf16, bf16>(g, keep_mask, dx, dr, dbias, rows, cols, p, seed, offset, elem_base,
                                                  workspace, workspace_bytes, s)
                   : launch_bwd_dbias<bf16, float>(g, keep_mask, dx, dr, dbias, rows, cols, p, seed, offset, elem_base,
                                                   workspace, workspace_bytes, s);
    return res_dt == MFX_BF16
               ? launch_bwd_dbias<float, bf16>(g, keep_mask, dx, dr, dbias, rows, cols, p, seed, offset, elem_base,
                                               workspace, workspace_bytes, s)
               : launch_bwd_dbias<float, float>(g, keep_mask, dx, dr, dbias, rows, cols, p, seed, offset, elem_base,
                                                workspace, workspace_bytes, s);
}
