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

// Linear bulk copy this CTA's shared memory -> global, tracked by the
// issuing thread's bulk async-groups.  Both addresses 16-byte aligned; bytes
// a multiple of 16.  Shared memory written by ordinary stores must be made
// visible to the copy engine first (fence_proxy_async by the writers, then a
// barrier among them).
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until at most N of this thread's committed groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Until every committed group of this thread has completed its writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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
constexpr size_t kMaxBlockSmem = 227 * 1024;  // dynamic shared memory a block may opt into

// Stages that fit a ring of `ring_bytes` at `stage_bytes` each, within [2, 8].
constexpr int ring_stages(int ring_bytes, int stage_bytes)
{
    return ring_bytes / stage_bytes < 2 ? 2 : (ring_bytes / stage_bytes > 8 ? 8 : ring_bytes / stage_bytes);
}

// Producer loop for streams laid out flat (unit i of every stream at byte
// i * unit_bytes[j] of its base): per iteration `it`, span k in [0, U)
// covers units [ub0 + (it*U + k)*S, +active) clipped to `units`, where
// `active` (<= 256) is the number of this block's consumer threads that own
// units; it lands at stage offset span_off[j] + k * 256 * unit_bytes[j].
// Run by one thread.
// A copy must be a multiple of 16 bytes, so a stream whose unit is smaller
// copies a multiple of 16 / gcd(unit bytes, 16) units (two for 8-byte
// units, sixteen for 1-byte units): the few units of a span's end past that
// are left for the consumers to read from global memory (copied_units).
// Returns false (after recording `err_flag` bits and draining the copies
// already issued) if a wait for a free stage ran out.
__device__ __forceinline__ uint32_t copied_units(uint32_t cnt, uint32_t unit_bytes)
{
    const uint32_t low = unit_bytes & (0u - unit_bytes);  // largest power of two dividing unit_bytes
    const uint32_t gran = low >= 16u ? 1u : 16u / low;
    return cnt - cnt % gran;
}

template <int NS, int U, int NSTREAMS>
__device__ __forceinline__ bool flat_producer(const Ring& ring, unsigned char* data, uint32_t stage_bytes,
                                              const void* const (&base)[NSTREAMS],
                                              const uint32_t (&unit_bytes)[NSTREAMS],
                                              const uint32_t (&span_off)[NSTREAMS], int64_t ub0, int64_t S,
                                              int64_t units, int64_t iters, unsigned* err_flag,
                                              uint32_t active = kConsumers)
{
    for (int64_t it = 0; it < iters; ++it) {
        const int s = (int)(it % NS);
        const int64_t n = it / NS;
        if (n > 0 && !mbar_wait(ring.empty(s), (uint32_t)((n - 1) & 1))) {
            atomicOr(err_flag, 2u);
            for (int64_t j = it - 1; j >= 0 && j > it - NS; --j)
                if (!mbar_wait(ring.full((int)(j % NS)), (uint32_t)((j / NS) & 1)))
                    atomicOr(err_flag, 4u);
            return false;
        }
        int64_t start[U];
        uint32_t cnt[U], total = 0;
#pragma unroll
        for (int k = 0; k < U; ++k) {
            start[k] = ub0 + (it * U + k) * S;
            const int64_t left = units - start[k];
            cnt[k] = left <= 0 ? 0u : (left < (int64_t)active ? (uint32_t)left : active);
#pragma unroll
            for (int j = 0; j < NSTREAMS; ++j)
                total += copied_units(cnt[k], unit_bytes[j]) * unit_bytes[j];
        }
        mbar_arrive_expect_tx(ring.full(s), total);
        unsigned char* st = data + (size_t)s * stage_bytes;
#pragma unroll
        for (int k = 0; k < U; ++k)
#pragma unroll
            for (int j = 0; j < NSTREAMS; ++j) {
                const uint32_t c = copied_units(cnt[k], unit_bytes[j]);
                if (c)
                    bulk_g2s(smem_addr(st + span_off[j] + k * kConsumers * unit_bytes[j]),
                             static_cast<const char*>(base[j]) + start[k] * unit_bytes[j], c * unit_bytes[j],
                             ring.full(s));
            }
    }
    return true;
}

// Consumer-side wait for stage s of iteration it (records err bit 1 on a
// timeout) and the release that follows the stage's use.
template <int NS>
__device__ __forceinline__ bool consumer_acquire(const Ring& ring, int64_t it, unsigned* err_flag)
{
    if (mbar_wait(ring.full((int)(it % NS)), (uint32_t)((it / NS) & 1)))
        return true;
    atomicOr(err_flag, 1u);
    return false;
}

template <int NS>
__device__ __forceinline__ void consumer_release(const Ring& ring, int64_t it)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(ring.empty((int)(it % NS)));
}

// Read one 8-element unit from shared memory.
__device__ __forceinline__ void lds8(const unsigned char* p, Raw8<bf16>& r) { r.v = *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void lds8(const unsigned char* p, Raw8<float>& r)
{
    r.v[0] = reinterpret_cast<const uint4*>(p)[0];
    r.v[1] = reinterpret_cast<const uint4*>(p)[1];
}

// Write one 8-element unit to shared memory (16-byte aligned).
__device__ __forceinline__ void stl8(unsigned char* p, const Raw8<bf16>& r) { *reinterpret_cast<uint4*>(p) = r.v; }
__device__ __forceinline__ void stl8(unsigned char* p, const Raw8<float>& r)
{
    reinterpret_cast<uint4*>(p)[0] = r.v[0];
    reinterpret_cast<uint4*>(p)[1] = r.v[1];
}

}  // namespace mfx
