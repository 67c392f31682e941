// mfx_pipe.cuh -- a warp-specialised bulk-copy pipeline for streaming
// kernels: one producer warp moves the block's next spans of every input
// stream into a ring of shared-memory stages with cp.async.bulk (the TMA
// engine's linear copy) and mbarrier transaction counts; eight consumer warps
// compute from shared memory and store their results straight to global
// memory.  Bytes in flight are bounded by the ring, not by registers.
//
// Every wait is bounded: after kWaitLimit polls it gives up, records the
// failure in the translation unit's device error word (read by
// mfx_device_error()) and the kernel returns without finishing; the producer
// first waits, again bounded, for the copies it issued.
#pragma once

#include <cstdint>

#include "mfx_device.cuh"

namespace mfx {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;    // = kThreadsPerBlock
constexpr int kPipeThreads = kConsumers + 32;     // + one producer warp
constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make the initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Poll the barrier until the phase of the given parity has completed;
// false after kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(bar), "r"(parity)
                     : "memory");
        if (done)
            return true;
    }
    return false;
}

// Linear bulk copy global -> this CTA's shared memory, completing `bytes`
// transactions on `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Stage bookkeeping shared by producer and consumers: use number n of stage
// s = it % NS is it / NS; `full[s]` completes once per use (parity n & 1),
// `empty[s]` completes when all consumer warps released use n.
struct Ring {
    uint32_t full0;   // address of full[0]; full[s] = full0 + 8 s
    uint32_t empty0;  // address of empty[0]
    __device__ __forceinline__ uint32_t full(int s) const { return full0 + 8u * s; }
    __device__ __forceinline__ uint32_t empty(int s) const { return empty0 + 8u * s; }
};

// Carve the ring's barriers from the start of dynamic shared memory and
// initialise them (thread 0), then make them visible block-wide.
template <int NS>
__device__ __forceinline__ Ring ring_setup(unsigned char* smem)
{
    static_assert(NS >= 2 && NS <= 8, "stages");
    Ring r{smem_addr(smem), smem_addr(smem) + 8u * NS};
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(r.full(s), 1);
            mbar_init(r.empty(s), kConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    return r;
}

constexpr int kRingHeader = 128;  // bytes reserved for up to 8 + 8 barriers

}  // namespace mfx
