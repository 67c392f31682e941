// mfx_device.cuh -- device helpers shared by the libmfx kernels: 16-byte
// streaming I/O, bf16 packing, the fp32 math of the activations, and the
// Philox4x32-10 counter-based generator.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

// Tuning knobs (compile-time; the defaults are the shipped configuration).
#ifndef MFX_PREFETCH_GELU
#define MFX_PREFETCH_GELU 1   // L2 bulk prefetch one unrolled iteration ahead
#endif
#ifndef MFX_PREFETCH_GLU_FWD
#define MFX_PREFETCH_GLU_FWD 1
#endif
#ifndef MFX_PREFETCH_GLU_BWD
#define MFX_PREFETCH_GLU_BWD 0  // measured: the 3-stream backward is faster without
#endif
#ifndef MFX_PREFETCH_WBWD
#define MFX_PREFETCH_WBWD 1     // weighted SwiGLU backward: next row to L2
#endif
#ifndef MFX_PREFETCH_WBWD_PART
#define MFX_PREFETCH_WBWD_PART 4  // eighths of the next row prefetched (measured best)
#endif
#ifndef MFX_UNROLL_WBWD
#define MFX_UNROLL_WBWD 2       // column units in flight, weighted SwiGLU backward (bf16)
#endif
#ifndef MFX_MINB_WBWD
#define MFX_MINB_WBWD 3
#endif
#ifndef MFX_UNROLL_GELU_PIPE
#define MFX_UNROLL_GELU_PIPE 4  // spans (units per consumer) per stage, bias-GeLU backward pipeline
#endif
#ifndef MFX_BDA_STAGE_KB
#define MFX_BDA_STAGE_KB 32    // bias-dropout-add training pipeline: stage size target (whole 256-unit spans)
#endif
#ifndef MFX_UNROLL_BDA_INF_PIPE
#define MFX_UNROLL_BDA_INF_PIPE 2  // the same for inference
#endif
#ifndef MFX_UNROLL_GLU_PIPE
#define MFX_UNROLL_GLU_PIPE 1  // spans (units per consumer) per stage, GLU pipeline
#endif
#ifndef MFX_UNROLL_GELU_FWD_PIPE
#define MFX_UNROLL_GELU_FWD_PIPE 8  // spans per stage, bias-GeLU forward pipeline
#endif
#ifndef MFX_UNROLL_GELU_DB_PIPE
#define MFX_UNROLL_GELU_DB_PIPE 4   // spans per stage (bf16; halved for fp32), bias-GeLU backward with the fused bias gradient
#endif
#ifndef MFX_RING_KB_GELU_DB
#define MFX_RING_KB_GELU_DB 96
#endif
#ifndef MFX_GELU_FWD_K_UNROLL
#define MFX_GELU_FWD_K_UNROLL 2     // unroll of its span loop
#endif
#ifndef MFX_UNROLL_SWIGLU_BWD_PIPE
#define MFX_UNROLL_SWIGLU_BWD_PIPE 1  // spans per stage, SwiGLU backward pipeline
#endif
#ifndef MFX_UNROLL_GEGLU_BWD_PIPE
#define MFX_UNROLL_GEGLU_BWD_PIPE 2  // the same for the GEGLU backward
#endif
#ifndef MFX_UNROLL_WBWD_PIPE
#define MFX_UNROLL_WBWD_PIPE 2  // units per consumer per stage, weighted SwiGLU backward pipeline
#endif
#ifndef MFX_RING_KB_SQRELU
#define MFX_RING_KB_SQRELU 64  // squared-ReLU backward ring (KB)
#endif
#ifndef MFX_PIPE_MINB_SQRELU
#define MFX_PIPE_MINB_SQRELU 3
#endif
#ifndef MFX_UNROLL_SQRELU_BWD
#define MFX_UNROLL_SQRELU_BWD 8  // units per consumer per stage, squared-ReLU backward (bf16)
#endif
#ifndef MFX_UNROLL_BDA_BWD
#define MFX_UNROLL_BDA_BWD 8  // 256-unit spans per stage, bias-dropout-add backward
#endif
#ifndef MFX_PREFETCH_BDA
#define MFX_PREFETCH_BDA 1
#endif
#ifndef MFX_UNROLL_GELU
#define MFX_UNROLL_GELU 4     // units in flight per thread, bias-GeLU
#endif
#ifndef MFX_UNROLL_GLU_FWD
#define MFX_UNROLL_GLU_FWD 2
#endif
#ifndef MFX_UNROLL_GLU_BWD
#define MFX_UNROLL_GLU_BWD 2
#endif
#ifndef MFX_UNROLL_BDA
#define MFX_UNROLL_BDA 4
#endif
#ifndef MFX_PIPE_GLU
#define MFX_PIPE_GLU 1        // GLU forward and unweighted backward through the pipeline
#endif
#ifndef MFX_PIPE_GELU
#define MFX_PIPE_GELU 1       // bias-GeLU through the pipeline
#endif
// Fast-tier reciprocal per forward kernel (see recip_1_2): 0 = the hardware
// approximation (one special-function op), 1 = quadratic start + one Newton
// step (four FMA ops), 3 = the cubic (three FMA ops).  Measured choices: the
// hardware op saves issue slots but doubles special-function use.  (The
// bias-GeLU forward takes the quadratic and one Newton step: gelu_fwd_fast.)
#ifndef MFX_RCP_GEGLU
#define MFX_RCP_GEGLU 0
#endif
#ifndef MFX_RCP_SWIGLU
#define MFX_RCP_SWIGLU 3
#endif
#ifndef MFX_RCP_SWIGLU_W
#define MFX_RCP_SWIGLU_W 0
#endif
// Backward factors (bias-GeLU, GEGLU, SwiGLU, weighted SwiGLU): 1 = hardware
// reciprocal (~1 ulp), 0 = two Newton steps (~1e-8).  Either is far inside
// the condition-scale bound the backward outputs are held to.
#ifndef MFX_HWRCP_BWD
#define MFX_HWRCP_BWD 0
#endif
#ifndef MFX_HWRCP_SWIGLU_BWD
#define MFX_HWRCP_SWIGLU_BWD 0 // SwiGLU backward (the GeLU and GEGLU ones follow MFX_HWRCP_BWD)
#endif
#ifndef MFX_HWRCP_WBWD
#define MFX_HWRCP_WBWD 1      // weighted SwiGLU backward (32 consumer warps per SM)
#endif
#ifndef MFX_PIPE_WBWD
#define MFX_PIPE_WBWD 1       // weighted SwiGLU backward through the pipeline
#endif
#ifndef MFX_RING_KB_WBWD
#define MFX_RING_KB_WBWD 96   // weighted SwiGLU backward
#endif
#ifndef MFX_PIPE_MINB_WBWD
#define MFX_PIPE_MINB_WBWD 2
#endif
#ifndef MFX_RING_KB_BDA
#define MFX_RING_KB_BDA 64    // bias-dropout-add training (two 24.6 KB stages)
#endif
#ifndef MFX_RING_KB_GELU
#define MFX_RING_KB_GELU 96   // bias-GeLU backward
#endif
#ifndef MFX_GELU_BWD_K_UNROLL
#define MFX_GELU_BWD_K_UNROLL 4   // unroll of the bias-GeLU backward pipeline's span loop
#endif
#ifndef MFX_SQRELU_BWD_K_UNROLL
#define MFX_SQRELU_BWD_K_UNROLL 8  // unroll of the squared-ReLU backward pipeline's chunk loop
#endif
#ifndef MFX_GEGLU_BWD_K_UNROLL
#define MFX_GEGLU_BWD_K_UNROLL 1  // unroll of the GEGLU backward pipeline's span loop
#endif
#ifndef MFX_SWIGLU_BWD_K_UNROLL
#define MFX_SWIGLU_BWD_K_UNROLL 1  // unroll of the SwiGLU backward pipeline's span loop
#endif
// Rings per pipeline (KB).  Fewer bytes in flight can be faster: with more
// stages than needed to cover the latency, the many concurrent bulk copies
// (hundreds of 4-8 KB streams over the GPU) cost DRAM efficiency (measured:
// SwiGLU backward 0.94 of the copy peak with 8 stages of 12 KB, 1.02 with 5).
#ifndef MFX_RING_KB_SWIGLU_BWD
#define MFX_RING_KB_SWIGLU_BWD 60
#endif
#ifndef MFX_RING_KB_GEGLU_BWD
#define MFX_RING_KB_GEGLU_BWD 96
#endif
#ifndef MFX_RING_KB_GLU_FWD
#define MFX_RING_KB_GLU_FWD 96     // GEGLU forward
#endif
#ifndef MFX_RING_KB_SWIGLU_FWD
#define MFX_RING_KB_SWIGLU_FWD 32  // SwiGLU forward, plain and weighted
#endif
#ifndef MFX_RING_KB_GELU_FWD
#define MFX_RING_KB_GELU_FWD 96
#endif
#ifndef MFX_RING_KB_BDA_INF
#define MFX_RING_KB_BDA_INF 50     // bias-dropout-add inference (two 24.6 KB stages)
#endif
#ifndef MFX_RING_KB_BDA_BWD
#define MFX_RING_KB_BDA_BWD 64     // two 32 KB stages (48 KB with the mask read)
#endif
#ifndef MFX_PIPE_MINB_BDA_BWD
#define MFX_PIPE_MINB_BDA_BWD 2
#endif
#ifndef MFX_WBWD_ROWS
#define MFX_WBWD_ROWS 1            // weighted SwiGLU backward, rows of <= 256 units: several rows per stage
#endif
#ifndef MFX_WBWD_RPIPE
#define MFX_WBWD_RPIPE 1           // weighted SwiGLU backward, any width: the realigning ring
#endif
#ifndef MFX_UNROLL_WBWD_RPIPE
#define MFX_UNROLL_WBWD_RPIPE 2    // ... units per consumer per stage
#endif
#ifndef MFX_RING_KB_WBWD_RPIPE
#define MFX_RING_KB_WBWD_RPIPE 96  // ... its ring
#endif
#ifndef MFX_WBWD_ANY_PF
#define MFX_WBWD_ANY_PF 1          // weighted SwiGLU backward, any width: next row to L2
#endif
#ifndef MFX_WBWD_ANY_BIASVEC
#define MFX_WBWD_ANY_BIASVEC 0     // ... its bias through realigned vectors (measured slower)
#endif
#ifndef MFX_MINB_WBWD_ANY
#define MFX_MINB_WBWD_ANY 3        // ... minimum resident blocks (caps registers)
#endif
#ifndef MFX_WBWD_ANY_U
#define MFX_WBWD_ANY_U 1           // ... units of a lane in flight
#endif
#ifndef MFX_WBWD_ANY_WORDST
#define MFX_WBWD_ANY_WORDST 1      // ... its bf16 outputs by word-granular stores
#endif
#ifndef MFX_BDA_PHASED_SHARE
#define MFX_BDA_PHASED_SHARE 1     // dropout training off a generator block: lanes share the blocks they draw
#endif
#ifndef MFX_BDA_BWD_BULK_ST
#define MFX_BDA_BWD_BULK_ST 1      // byte-mask backward: outputs through per-warp shared slots and bulk stores
#endif
#ifndef MFX_BDA_BWD_SLOTS
#define MFX_BDA_BWD_SLOTS 4        // output slots a warp cycles through
#endif
#ifndef MFX_RING_KB_SQRELU_FWD
#define MFX_RING_KB_SQRELU_FWD 96
#endif
#ifndef MFX_PIPE_MINB_SWIGLU_BWD
#define MFX_PIPE_MINB_SWIGLU_BWD 2
#endif
#ifndef MFX_PIPE_MINB_GLU
#define MFX_PIPE_MINB_GLU 2   // minimum resident pipeline blocks (caps registers)
#endif
// Bias-GeLU pipeline: test a unit's range by a per-stage span count (1) or
// by its 64-bit index (0); measured per direction.
#ifndef MFX_GELU_SPAN_COUNT_FWD
#define MFX_GELU_SPAN_COUNT_FWD 0
#endif
#ifndef MFX_GELU_SPAN_COUNT_BWD
#define MFX_GELU_SPAN_COUNT_BWD 1
#endif
#ifndef MFX_GLU_PTR_INC
#define MFX_GLU_PTR_INC 1  // SwiGLU forward pipeline: output pointer advanced per stage (0: recomputed per unit)
#endif
#ifndef MFX_PIPE_MINB_GELU_FWD
#define MFX_PIPE_MINB_GELU_FWD 2  // bias-GeLU forward pipeline
#endif
#ifndef MFX_PIPE_MINB_BDA_TRAIN
#define MFX_PIPE_MINB_BDA_TRAIN 2  // bias-dropout-add training pipeline
#endif
#ifndef MFX_PIPE_MINB_BDA
#define MFX_PIPE_MINB_BDA 3
#endif
#ifndef MFX_PIPE_MINB_GELU
#define MFX_PIPE_MINB_GELU 2
#endif
#ifndef MFX_PRECISE_RCP_GRAD
#define MFX_PRECISE_RCP_GRAD 1 // fp32 GeLU gradient factor: 1 / (1 + e) as hardware reciprocal + Newton step
#endif                         // (0: IEEE reciprocal; measured 0.86 -> 0.91, slower in the forwards)
#ifndef MFX_GLU_RPIPE
#define MFX_GLU_RPIPE 1        // GLU at any width/alignment (F >= 2048) through the bulk-copy ring
#endif
#ifndef MFX_GLU_RPIPE_WORD_ST
#define MFX_GLU_RPIPE_WORD_ST 1  // its bf16 backward's outputs by word-granular stores (0: assembled across the warp)
#endif
#ifndef MFX_RING_KB_GLU_RPIPE
#define MFX_RING_KB_GLU_RPIPE 96
#endif
#ifndef MFX_PIPE_MINB_GLU_RPIPE
#define MFX_PIPE_MINB_GLU_RPIPE 2  // minimum resident blocks of the GLU ring (caps registers)
#endif
#ifndef MFX_RING_KB_GLU_RPIPE_FWD16
#define MFX_RING_KB_GLU_RPIPE_FWD16 64  // its bf16 forward: a smaller ring, three blocks an SM
#endif
#ifndef MFX_PIPE_MINB_GLU_RPIPE_FWD16
#define MFX_PIPE_MINB_GLU_RPIPE_FWD16 3
#endif
#ifndef MFX_RING_KB_GLU_RPIPE_BWD16
#define MFX_RING_KB_GLU_RPIPE_BWD16 64  // its bf16 backward: the same (72 registers, no spills)
#endif
#ifndef MFX_PIPE_MINB_GLU_RPIPE_BWD16
#define MFX_PIPE_MINB_GLU_RPIPE_BWD16 3
#endif
#ifndef MFX_UNROLL_GLU_ANY
#define MFX_UNROLL_GLU_ANY 2   // units in flight per thread, GLU at any width/alignment
#endif
#ifndef MFX_GELU_FWD_PAIRED
#define MFX_GELU_FWD_PAIRED 0  // bias-GeLU forward pipeline (bf16): unit code on .f32x2 pairs (measured slower)
#endif
#ifndef MFX_GELU_FWD_EXPLICIT
#define MFX_GELU_FWD_EXPLICIT MFX_GELU_FWD_PAIRED  // its scalar forms as the same explicit steps
#endif
#ifndef MFX_BDA_PAIRED
#define MFX_BDA_PAIRED 0      // bias-dropout-add pipeline (bf16 x): arithmetic on .f32x2 pairs (measured slower)
#endif
#ifndef MFX_PHILOX_WIDE
#define MFX_PHILOX_WIDE 1     // Philox multiplies as one widening multiply each (0: low and high apart)
#endif
#ifndef MFX_PIPE_BDA
#define MFX_PIPE_BDA 1        // bias-dropout-add through the shared-memory bulk-copy pipeline
#endif
#ifndef MFX_MINB_GELU
#define MFX_MINB_GELU 1       // minimum resident blocks (caps registers)
#endif
#ifndef MFX_MINB_GLU
#define MFX_MINB_GLU 1
#endif
#ifndef MFX_MINB_BDA
#define MFX_MINB_BDA 1
#endif

namespace mfx {

constexpr int kThreadsPerBlock = 256;  // every kernel's block size

// Raw bf16 storage (the library never needs bf16 arithmetic: every value is
// widened to fp32 on load and rounded once on store).
struct bf16 {
    uint16_t bits;
};

template <typename T> struct DTypeInfo;
template <> struct DTypeInfo<float> { static constexpr int kBytes = 4; static constexpr bool kBf16 = false; };
template <> struct DTypeInfo<bf16> { static constexpr int kBytes = 2; static constexpr bool kBf16 = true; };

// The ABI dtype code of a storage type (0 = fp32, 1 = bf16).
template <typename T> constexpr int dtype_code() { return DTypeInfo<T>::kBf16 ? 1 : 0; }

// ---------------------------------------------------------------------------
// Memory: 16-byte coalesced streaming accesses.  Loads skip L1 allocation and
// ask L2 for 256-byte prefetch; stores are marked evict-first.  The loads are
// coherent (not .nc) so that in-place calls, where a thread reads a location
// and later writes it, stay within the PTX memory model.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Read-only cached 16-byte load for small re-read operands (the bias).
__device__ __forceinline__ uint4 ld16_ro(const void* p)
{
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

#ifndef MFX_ST_CS
#define MFX_ST_CS 1  // 1 = streaming (evict-first) stores, 0 = default write-back
#endif
#if MFX_ST_CS
#define MFX_ST_OP "st.global.cs"
#else
#define MFX_ST_OP "st.global"
#endif

__device__ __forceinline__ void st16(void* p, uint4 v)
{
    asm volatile(MFX_ST_OP ".v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st8(void* p, uint2 v)
{
    asm volatile(MFX_ST_OP ".v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel whose output feeds a second,
// dependent launch (the fused bias gradients' partials) lets that launch be
// scheduled once its main loop is done; the dependent kernel waits for this
// grid to complete, with its memory visible, before it reads.  Both are
// no-ops for a launch made without the programmatic-serialization attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// bf16 <-> fp32.  Widening is a shift; narrowing is the hardware's
// round-to-nearest-even conversion of two fp32 values at once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// lo -> bits [0, 16), hi -> bits [16, 32)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ float round_to_bf16(float v) { return bf16lo(pack_bf16x2(v, 0.0f)); }

__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const bf16* p) { return __uint_as_float((uint32_t)p->bits << 16); }
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(bf16* p, float v) { p->bits = (uint16_t)pack_bf16x2(v, 0.0f); }

// ---------------------------------------------------------------------------
// Pairs of fp32 values: the .f32x2 forms of add, mul and fma (one
// instruction for two lanes), each lane rounded exactly as the scalar
// operation would be.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 widen2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// Eight consecutive elements ("a group"): one 16-byte vector of bf16 or two
// of fp32.  `p` must be 16-byte aligned.
template <typename T> struct Raw8;
template <> struct Raw8<bf16> { uint4 v; };
template <> struct Raw8<float> { uint4 v[2]; };

__device__ __forceinline__ void ld8(const bf16* p, Raw8<bf16>& r) { r.v = ld16(p); }
__device__ __forceinline__ void ld8(const float* p, Raw8<float>& r)
{
    r.v[0] = ld16(p);
    r.v[1] = ld16(p + 4);
}
__device__ __forceinline__ void st8(bf16* p, const Raw8<bf16>& r) { st16(p, r.v); }
__device__ __forceinline__ void st8(float* p, const Raw8<float>& r)
{
    st16(p, r.v[0]);
    st16(p + 4, r.v[1]);
}

__device__ __forceinline__ void widen8(const Raw8<bf16>& r, float f[8])
{
    const uint32_t w[4] = {r.v.x, r.v.y, r.v.z, r.v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16lo(w[i]);
        f[2 * i + 1] = bf16hi(w[i]);
    }
}
__device__ __forceinline__ void widen8(const Raw8<float>& r, float f[8])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        f[4 * h + 0] = __uint_as_float(r.v[h].x);
        f[4 * h + 1] = __uint_as_float(r.v[h].y);
        f[4 * h + 2] = __uint_as_float(r.v[h].z);
        f[4 * h + 3] = __uint_as_float(r.v[h].w);
    }
}
__device__ __forceinline__ void narrow8(const float f[8], Raw8<bf16>& r)
{
    r.v = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                     pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ void narrow8(const float f[8], Raw8<float>& r)
{
#pragma unroll
    for (int h = 0; h < 2; ++h)
        r.v[h] = make_uint4(__float_as_uint(f[4 * h]), __float_as_uint(f[4 * h + 1]),
                            __float_as_uint(f[4 * h + 2]), __float_as_uint(f[4 * h + 3]));
}

// ---------------------------------------------------------------------------
// Runs of 8 elements at any element alignment, through aligned 16-byte
// vectors.  extract16 takes the 16 bytes at byte offset o (even) of a word
// array; ld8_any loads the run at p from the (one to three) aligned vectors
// that cover it.  Loads here are L1-cached: the neighbouring run reads the
// same vectors.
// ---------------------------------------------------------------------------
template <int NW>
__device__ __forceinline__ uint4 extract16(const uint32_t (&w)[NW], uint32_t o)
{
    const uint32_t h = (o & 3u) * 8u;
    uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0, a4 = 0;
    switch (o >> 2) {
#define MFX_PICK(Q)                                                                                             \
    case Q:                                                                                                     \
        if constexpr (Q + 4 < NW) {                                                                             \
            a0 = w[Q], a1 = w[Q + 1], a2 = w[Q + 2], a3 = w[Q + 3], a4 = w[Q + 4];                              \
        } else if constexpr (Q + 3 < NW) {                                                                      \
            a0 = w[Q], a1 = w[Q + 1], a2 = w[Q + 2], a3 = w[Q + 3];                                             \
        }                                                                                                       \
        break;
        MFX_PICK(0) MFX_PICK(1) MFX_PICK(2) MFX_PICK(3) MFX_PICK(4) MFX_PICK(5) MFX_PICK(6) MFX_PICK(7)
        MFX_PICK(8) MFX_PICK(9) MFX_PICK(10) MFX_PICK(11)
#undef MFX_PICK
    default: break;
    }
    return make_uint4(__funnelshift_r(a0, a1, h), __funnelshift_r(a1, a2, h), __funnelshift_r(a2, a3, h),
                      __funnelshift_r(a3, a4, h));
}

__device__ __forceinline__ uint4 ld16_ca(const void* p)
{
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// The run of 8 elements at p (any element alignment).  Every vector read
// lies inside [lo, hi) (the caller checks: in_vectors).
template <typename T>
__device__ __forceinline__ void ld8_any(const T* p, Raw8<T>& r)
{
    constexpr int NV = (int)sizeof(T) / 2 + 1;  // vectors covering a run: 2 (bf16), 3 (fp32)
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t phi = (uint32_t)(a & 15u);
    const char* v = reinterpret_cast<const char*>(a - phi);
    uint32_t w[4 * NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        uint4 q = make_uint4(0, 0, 0, 0);
        if (k < NV - 1 || phi != 0)
            q = ld16_ca(v + 16 * k);
        w[4 * k] = q.x, w[4 * k + 1] = q.y, w[4 * k + 2] = q.z, w[4 * k + 3] = q.w;
    }
    if constexpr (DTypeInfo<T>::kBf16) {
        r.v = extract16(w, phi);
    } else {
        r.v[0] = extract16(w, phi);
        r.v[1] = extract16(w, phi + 16u);
    }
}

// Whether the aligned vectors covering the run of 8 elements at p lie inside
// the byte range [lo, hi).
template <typename T>
__device__ __forceinline__ bool in_vectors(const T* p, uintptr_t lo, uintptr_t hi)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return (a & ~(uintptr_t)15) >= lo && ((a + 8 * sizeof(T) - 1) & ~(uintptr_t)15) + 16 <= hi;
}

// Ask L2 to fetch `bytes` (a multiple of 16) starting at 16-byte aligned `p`
// when `on` is nonzero (a bulk asynchronous prefetch: no registers, no
// completion to wait for).  Predicated rather than branched, so the hot loops
// keep straight-line code.
__device__ __forceinline__ void prefetch_l2_if(const void* p, uint32_t bytes, uint32_t on)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t"
                 "@q cp.async.bulk.prefetch.L2.global [%0], %1;\n\t}" ::"l"(p),
                 "r"(bytes), "r"(on));
}

// Block-cooperative L2 prefetch for grid-stride loops: lane 0 of a warp with
// `warp_on` asks L2 for the 256 units [first, first + 256) of a stream of
// `units` units of `unit_bytes` bytes (clipped to the stream).  Callers give
// warp k the block's k-th unrolled slice of the next iteration, so each warp
// spends one instruction and one address per stream per iteration.
template <bool ON>
__device__ __forceinline__ void prefetch_block_span(const void* base, int64_t first, int64_t units,
                                                    int unit_bytes, bool warp_on)
{
    if (ON) {
        const int64_t left = units - first;
        const uint32_t n = left < kThreadsPerBlock ? (uint32_t)(left > 0 ? left : 0) : kThreadsPerBlock;
        const uint32_t on = ((threadIdx.x & 31) == 0) & warp_on & (n > 0);
        prefetch_l2_if(static_cast<const char*>(base) + (on ? first * unit_bytes : 0), n * unit_bytes, on);
    }
}

// Eight bias values at a 16-byte aligned column (zeros without a bias).
template <typename T>
__device__ __forceinline__ void bias8(const T* bias, int64_t col, float b[8])
{
    if (!bias) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            b[k] = 0.0f;
        return;
    }
    Raw8<T> r;
    if constexpr (DTypeInfo<T>::kBf16) {
        r.v = ld16_ro(bias + col);
    } else {
        r.v[0] = ld16_ro(bias + col);
        r.v[1] = ld16_ro(bias + col + 4);
    }
    widen8(r, b);
}

// One bias value (0 without a bias).
template <typename T>
__device__ __forceinline__ float bias1(const T* bias, int64_t col)
{
    return bias ? load1(bias + col) : 0.0f;
}

// The bias of 8 consecutive elements whose first lies in column c0 (the
// columns wrap from cols - 1 to 0): one 16-byte load when the run is a
// 16-byte aligned run of one row, else element by element.
template <typename T>
__device__ __forceinline__ void bias8_at(const T* bias, int64_t c0, int64_t cols, float b[8])
{
    if (!bias || (cols % 8 == 0 && c0 % 8 == 0 && ((reinterpret_cast<uintptr_t>(bias) & 15u) == 0))) {
        bias8(bias, c0, b);
        return;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int64_t c = c0 + j;
        if (c >= cols)
            c -= cols;
        b[j] = load1(bias + (c < cols ? c : c % cols));
    }
}

// Vector or element-wise load of up to 8 elements into fp32 (missing ones 0).
template <typename T>
__device__ __forceinline__ void load8f(const T* p, bool vec, int n, float f[8])
{
    if (vec && n == 8) {
        Raw8<T> r;
        ld8(p, r);
        widen8(r, f);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            f[k] = k < n ? load1(p + k) : 0.0f;
    }
}

template <typename T>
__device__ __forceinline__ void store8f(T* p, bool vec, int n, const float f[8])
{
    if (vec && n == 8) {
        Raw8<T> r;
        narrow8(f, r);
        st8(p, r);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < n)
                store1(p + k, f[k]);
    }
}

// ---------------------------------------------------------------------------
// Activation math.  All of it is fp32.  Both tiers evaluate the logistic
// form of the tanh GeLU,
//     x * 0.5 * (1 + tanh u) = x * sigma(2u),   sigma(z) = 1 / (1 + e^-z),
// through e = exp(-|z|) in (0, 1] and q = 1 / (1 + e):
//     sigma(|z|) = q,  sigma(-|z|) = e q,  sigma(z) sigma(-z) = e q^2,
// which never subtracts nearly equal numbers, so the relative error stays at
// a few fp32 ulps for any sign of x (the printed form loses all relative
// precision when 1 + tanh u cancels for u << 0).
//
// Precise tier (fp32 outputs): libdevice expf and the IEEE reciprocal.
// Fast tier (bf16 outputs, whose 1-ulp budget is 2^-9 relative): the
// hardware 2^x approximation and a polynomial reciprocal on [1, 2], so the
// special-function unit does one operation per element.  A polynomial p of
// degree n with 1 - d p(d) = +-T_{n+1}(2d - 3) / |T_{n+1}(-3)| (T the
// Chebyshev polynomials; the constraint is the value 1 at d = 0) has the
// equioscillating minimum of the relative error on [1, 2]: 1/99 for the
// quadratic (210 - 144 d + 32 d^2) / 99, 1/577 for the cubic
// (1632 - 1696 d + 768 d^2 - 128 d^3) / 577.  Each forward kernel takes,
// as measured fastest for it (MFX_RCP_*): the cubic alone (1/577 = 1.73e-3
// = 0.89 of 2^-9; with the fp32 roundings and the exponential's 2^-22 the
// result stays within 1 ulp: 0.5 ulp rounding plus under 0.45 ulp), the
// quadratic and one Newton step ((1/99)^2 ~ 1.0e-4), or the hardware
// approximation.  The backward factors add sigma(z) sigma(-z) terms to
// sigma(z) and cancel near their roots, where that error would be amplified,
// so they take the quadratic and two Newton steps ((1/99)^4 ~ 1e-8).
// ---------------------------------------------------------------------------
constexpr double kGeluK0 = 0.79788456;   // sqrt(2/pi) as printed
constexpr double kGeluK1 = 0.044715;
constexpr double kGeluKD = 0.1070322243; // 3 * 0.79788456 * 0.044715 as printed
constexpr double kLog2e = 1.4426950408889634;

// 2^t for t <= 0 by the flush-to-zero hardware approximation, evaluated at
// t + 64 and scaled back by an exact 2^-64 so that results down to 2^-190
// (subnormal in fp32, still visible after a multiply by a large x) survive.
// `t64` is t + 64.
__device__ __forceinline__ float ex2_neg(float t64)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t64));
    return y * 5.421010862427522e-20f;  // 2^-64
}

// MODE 0: the hardware approximation (relative error ~1 ulp); 1, 2: the
// quadratic and one or two Newton steps; 3: the cubic alone.
template <int MODE>
__device__ __forceinline__ float recip_1_2(float d)
{
    static_assert(MODE >= 0 && MODE <= 3, "reciprocal mode");
    constexpr int STEPS = MODE;
    if (MODE == 0) {
        float r;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
        return r;
    }
    if (MODE == 3)
        return fmaf(fmaf(fmaf(-128.0f / 577.0f, d, 768.0f / 577.0f), d, -1696.0f / 577.0f), d, 1632.0f / 577.0f);
    float r = fmaf(fmaf(32.0f / 99.0f, d, -144.0f / 99.0f), d, 210.0f / 99.0f);
#pragma unroll
    for (int i = 0; i < STEPS; ++i) {
        const float t = fmaf(-d, r, 1.0f);
        r = fmaf(r, t, r);
    }
    return r;
}

// Logistic values of z: sp = sigma(|z|), sn = sigma(-|z|).  The precise tier
// takes z; the fast tier takes z log2(e).
struct Sig {
    float sp;
    float sn;
};

// Precise: sigma(|z|) = 1 - e r with r = 1/(1 + e) is formed by one fused
// multiply-add, so near 1 (large |z|, where outputs are largest) it carries a
// single rounding instead of the two of rounding 1 + e and then 1/(1 + e).
// Fast: `z` is z log2(e) (the callers fold log2(e) into their constants) and
// MODE picks the reciprocal (recip_1_2); the precise tier ignores MODE.
template <bool PRECISE, int MODE = 2, bool FAST_RCP = false>
__device__ __forceinline__ Sig sig_of(float z)
{
    if constexpr (PRECISE) {
        const float e = expf(-fabsf(z));
        const float d = 1.0f + e;
        float r;
        if (FAST_RCP) {
            // d in (1, 2]: no zero, subnormal or infinite case, so the hardware
            // reciprocal (about 1 ulp) and one Newton step give the reciprocal
            // to a fraction of an ulp without the IEEE division's slow path
            asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
            r = fmaf(r, fmaf(-d, r, 1.0f), r);
        } else {
            r = __frcp_rn(d);
        }
        return Sig{fmaf(-e, r, 1.0f), e * r};
    } else {
        const float e = ex2_neg(64.0f - fabsf(z));
        const float r = recip_1_2<MODE>(1.0f + e);
        return Sig{r, e * r};
    }
}

// Products of three or four factors.  Precise tier: the first pair (and the
// second) is split into its rounded product and exact error (the FMA
// two-product), so the whole product carries about one rounding.  A product
// that overflows skips the error term (inf - inf would be NaN).
__device__ __forceinline__ float two_prod_err(float a, float b, float p)
{
    return fabsf(p) < INFINITY ? fmaf(a, b, -p) : 0.0f;
}

template <bool PRECISE>
__device__ __forceinline__ float mul3(float a, float b, float c)
{
    if (PRECISE) {
        const float p = __fmul_rn(a, b);
        const float pe = two_prod_err(a, b, p);
        return fmaf(p, c, pe * c);
    }
    return a * b * c;
}

template <bool PRECISE>
__device__ __forceinline__ float mul4(float a, float b, float c, float d)
{
    if (PRECISE) {
        const float p1 = __fmul_rn(a, b), p2 = __fmul_rn(c, d);
        const float e1 = two_prod_err(a, b, p1), e2 = two_prod_err(c, d, p2);
        return fmaf(p1, p2, fmaf(p1, e2, e1 * p2));
    }
    return a * b * c * d;
}

// Logistic form of the tanh GeLU at x: returns sz = sigma(2u) =
// 0.5 (1 + tanh u), so gelu(x) = x sz; with GRAD also the backward factor
//   gelu'(x) = 0.5 x (1 - t^2)(k0 + kd x^2) + 0.5 (1 + t)
//            = x sigma(2u) sigma(-2u) (2 k0 + 2 kd x^2) + sigma(2u).
// x^2 is clamped so that for |x| > 1.8e19 (x^2 = inf) the vanishing first
// term stays 0 instead of 0 * inf.
template <bool PRECISE, bool GRAD, int RCP = 1>
__device__ __forceinline__ float gelu_sigma(float x, float* grad)
{
    const float x2 = x * x;
    // z = 2u = 2 * 0.79788456 * x * (1 + 0.044715 x^2), times log2(e) in the
    // fast tier: z' = x * (c0 + c1 x^2) with c0 = 2 k0 [log2 e], c1 = c0 k1.
    constexpr double c0 = PRECISE ? 2.0 * kGeluK0 : 2.0 * kGeluK0 * kLog2e;
    const float z = x * fmaf((float)(c0 * kGeluK1), x2, (float)c0);
    const Sig s = sig_of<PRECISE, GRAD ? (MFX_HWRCP_BWD ? 0 : 2) : RCP, GRAD && MFX_PRECISE_RCP_GRAD>(z);
    const float sz = z >= 0.0f ? s.sp : s.sn;
    if (GRAD) {
        const float poly2 = fmaf((float)(2.0 * kGeluKD), fminf(x2, 1.0e38f), (float)(2.0 * kGeluK0));
        *grad = fmaf(x * (s.sp * s.sn), poly2, sz);
    }
    return sz;
}

// The bias-GeLU forward of the fast tier, gelu(x) = x sigma(2u), as a fixed
// sequence of round-to-nearest fp32 steps: z = 2u log2(e) = x (c0 + c1 x^2);
// e = 2^-|z| (the hardware 2^x at 64 - |z|, scaled by 2^-64); r = 1 / (1 + e)
// by the quadratic start and one Newton step, written with nd = -(1 + e) so
// that every step is a plain multiply-add (no negated operand); sigma(2u) is
// r for z >= 0, else e r.  gelu_fwd_fast2 runs the same steps on two elements
// with the paired instructions (one issue for both), so the two forms give
// the same bits.
struct GeluFwdK {
    static constexpr float c0 = (float)(2.0 * kGeluK0 * kLog2e);
    static constexpr float c1 = (float)(2.0 * kGeluK0 * kLog2e * kGeluK1);
    static constexpr float r2 = 32.0f / 99.0f, r1 = 144.0f / 99.0f, r0 = 210.0f / 99.0f;
    static constexpr float two_m64 = 5.421010862427522e-20f;  // 2^-64
};

__device__ __forceinline__ float ex2_approx(float t)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
    return y;
}

__device__ __forceinline__ float gelu_fwd_fast(float x)
{
    using K = GeluFwdK;
    const float x2 = __fmul_rn(x, x);
    const float z = __fmul_rn(x, __fmaf_rn(K::c1, x2, K::c0));
    const float e = __fmul_rn(ex2_approx(__fadd_rn(64.0f, -fabsf(z))), K::two_m64);
    const float nd = __fmaf_rn(e, -1.0f, -1.0f);
    const float q = __fmaf_rn(K::r2, nd, K::r1);
    const float r = __fmaf_rn(q, nd, K::r0);
    const float t = __fmaf_rn(nd, r, 1.0f);
    const float rr = __fmaf_rn(r, t, r);
    return __fmul_rn(x, z >= 0.0f ? rr : __fmul_rn(e, rr));
}

__device__ __forceinline__ float2 gelu_fwd_fast2(float2 x)
{
    using K = GeluFwdK;
    const float2 z = mul2(x, fma2(f2(K::c1), mul2(x, x), f2(K::c0)));
    float2 e = make_float2(ex2_approx(__fadd_rn(64.0f, -fabsf(z.x))), ex2_approx(__fadd_rn(64.0f, -fabsf(z.y))));
    e = mul2(e, f2(K::two_m64));
    const float2 nd = fma2(e, f2(-1.0f), f2(-1.0f));
    const float2 r = fma2(fma2(f2(K::r2), nd, f2(K::r1)), nd, f2(K::r0));
    const float2 rr = fma2(r, fma2(nd, r, f2(1.0f)), r);
    const float2 sn = mul2(e, rr);
    return mul2(x, make_float2(z.x >= 0.0f ? rr.x : sn.x, z.y >= 0.0f ? rr.y : sn.y));
}

// SiLU pieces of a: sigma(a) and 1 - sigma(a) (silu(a) = a sigma(a)).
template <bool PRECISE, int STEPS>
__device__ __forceinline__ void silu_sigma(float a, float* sig, float* one_minus_sig)
{
    const Sig s = sig_of<PRECISE, STEPS>(PRECISE ? a : a * (float)kLog2e);
    const bool pos = a >= 0.0f;
    *sig = pos ? s.sp : s.sn;
    *one_minus_sig = pos ? s.sn : s.sp;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies, a word permutation and key xors; the key is bumped by
// the Weyl increments between rounds.
// ---------------------------------------------------------------------------
// The 64-bit product of two words as (lo, hi): MFX_PHILOX_WIDE = 1 forms it
// with one widening multiply, 0 with separate low and high multiplies.
__device__ __forceinline__ void mul_hilo(uint32_t a, uint32_t b, uint32_t& lo, uint32_t& hi)
{
#if MFX_PHILOX_WIDE
    const uint64_t p = (uint64_t)a * (uint64_t)b;
    lo = (uint32_t)p;
    hi = (uint32_t)(p >> 32);
#else
    lo = a * b;
    hi = __umulhi(a, b);
#endif
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint32_t lo0, hi0, lo1, hi1;
        mul_hilo(0xD2511F53u, c.x, lo0, hi0);
        mul_hilo(0xCD9E8D57u, c.z, lo1, hi1);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// The 128-bit block of mask block j: counter (lo j, hi j, lo offset, hi offset).
__device__ __forceinline__ uint4 mask_block(uint64_t j, uint64_t seed, uint64_t offset)
{
    return philox4x32_10(make_uint4((uint32_t)j, (uint32_t)(j >> 32), (uint32_t)offset,
                                    (uint32_t)(offset >> 32)),
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}

// The eight 16-bit words of elements [8j + o, 8j + o + 8) (o in 0..7, the
// same for every call of a launch): words o..7 of block j and 0..o-1 of
// block j + 1, as one 128-bit block (word k = element 8j + o + k), from the
// two blocks already drawn (mask_words_at) or drawing them (mask_block_at).
__device__ __forceinline__ uint4 mask_words_at(const uint4& a, const uint4& b, int o)
{
    if (o == 0)
        return a;
    const int h = (o & 1) * 16;
    uint32_t w[5];
    switch (o >> 1) {  // uniform across the launch
    case 0: w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x; break;
    case 1: w[0] = a.y, w[1] = a.z, w[2] = a.w, w[3] = b.x, w[4] = b.y; break;
    case 2: w[0] = a.z, w[1] = a.w, w[2] = b.x, w[3] = b.y, w[4] = b.z; break;
    default: w[0] = a.w, w[1] = b.x, w[2] = b.y, w[3] = b.z, w[4] = b.w; break;
    }
    return make_uint4(__funnelshift_r(w[0], w[1], h), __funnelshift_r(w[1], w[2], h),
                      __funnelshift_r(w[2], w[3], h), __funnelshift_r(w[3], w[4], h));
}

__device__ __forceinline__ uint4 mask_block_at(uint64_t j, int o, uint64_t seed, uint64_t offset)
{
    const uint4 a = mask_block(j, seed, offset);
    if (o == 0)
        return a;
    return mask_words_at(a, mask_block(j + 1, seed, offset), o);
}

// 16-bit word `lane` (0..7, little-endian) of a block.
__device__ __forceinline__ uint32_t word16(const uint4& b, int lane)
{
    const uint32_t w = (lane >> 1) == 0 ? b.x : (lane >> 1) == 1 ? b.y : (lane >> 1) == 2 ? b.z : b.w;
    return (lane & 1) ? (w >> 16) : (w & 0xFFFFu);
}

}  // namespace mfx
