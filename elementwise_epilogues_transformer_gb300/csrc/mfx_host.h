// mfx_host.h -- host-side helpers of libmfx: argument checks, alignment and
// overlap tests, and the grid plan every launch uses.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mfx.h"

namespace mfx {

constexpr int kThreads = 256;  // threads per block for every kernel (= kThreadsPerBlock)

// Records a CUDA error for mfx_last_cuda_error() and returns MFX_ERR_CUDA.
int cuda_failure(cudaError_t e);

// Status of the launch just issued.
inline int launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MFX_OK : cuda_failure(e);
}

inline bool valid_dtype(int dt) { return dt == MFX_F32 || dt == MFX_BF16; }
inline int64_t dtype_bytes(int dt) { return dt == MFX_BF16 ? 2 : 4; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// a * b without int64 overflow (a, b >= 0); false on overflow.
inline bool mul_ok(int64_t a, int64_t b, int64_t* out)
{
    if (a != 0 && b > INT64_MAX / a)
        return false;
    *out = a * b;
    return true;
}

// Do [a, a + na) and [b, b + nb) share a byte?  (NULL never overlaps.)
inline bool overlaps(const void* a, int64_t na, const void* b, int64_t nb)
{
    if (!a || !b || na <= 0 || nb <= 0)
        return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

// Overlap that is not the exact same buffer (allowed for element-wise
// in-place use: every element is read before the same thread writes it).
inline bool partial_overlap(const void* a, int64_t na, const void* b, int64_t nb)
{
    return overlaps(a, na, b, nb) && !(a == b && na == nb);
}

// Multiprocessor count of the current device.
int sm_count();

// Resident blocks of `kernel` per multiprocessor at kThreads threads.
int blocks_per_sm(const void* kernel);

// Resident blocks per multiprocessor at `block_threads` threads and `smem`
// bytes of dynamic shared memory (at least 1), cached per device, kernel and
// size; also raises the kernel's dynamic shared-memory limit to `smem` when
// it is above 48 KB and above every size set before.
int occupancy(const void* kernel, int block_threads, size_t smem);

// Launch geometry for a grid-stride loop over `units` work items of 8
// elements, one item per thread per iteration.
//
// In the fixed-column form the total thread count S is a multiple of
// `row_units` (items per row), so each thread keeps one column for the whole
// loop and holds that column's bias in registers.  S is the multiple of
// lcm(kThreads, row_units) nearest the device's resident-thread capacity
// (SMs x resident blocks x kThreads) from below (so that every block is
// resident at once), at least one, and no larger than the work needs.  When
// that multiple is more than 4x the capacity the fixed form is refused.
struct Grid {
    bool fixed = false;
    int64_t blocks = 0;
    int64_t S = 0;  // active unit-owning threads (plan_fixed_any; else blocks x kThreads)
};

Grid plan_grid(const void* kernel, int64_t units, int64_t row_units, bool want_fixed);

// The same plan for a kernel launched with `block_threads` threads of which
// `work_threads` (= kThreads) take units, and `smem` bytes of dynamic shared
// memory.  Sets the kernel's dynamic shared-memory limit on first use.
Grid plan_grid_ex(const void* kernel, int block_threads, size_t smem, int64_t units, int64_t row_units,
                  bool want_fixed);

// Fixed-column plan for any width: units are 8 consecutive elements of the
// flat tensor (unit u starts at element e0 + 8u for some fixed e0), so unit
// u's first column is (e0 + 8u) mod cols and units u and u + S start at the
// same column exactly when S is a multiple of P = cols / gcd(cols, 8).  S is
// the largest multiple of P within the resident-thread capacity (one wave of
// blocks; at least P, at most what the units need); it need not be a
// multiple of kThreads: the
// grid has ceil(S / kThreads) blocks and the last block's threads from
// S mod kThreads on take no units.  Refused (fixed = false) when P is more
// than 4x the capacity.
Grid plan_fixed_any(const void* kernel, int block_threads, size_t smem, int64_t units, int64_t cols);

// Fused bias gradients (see dbias.cu): lanes J of a fallback column-partial
// pass, the workspace protocol, the partial pass and the finishing sum.
constexpr int64_t kGenericLanes = 64;
int64_t dbias_generic_lanes(int64_t rows);
int dbias_workspace(int64_t J, int64_t W, void* workspace, size_t* workspace_bytes, bool* query);
int launch_column_partials(int dt, const void* src, int64_t rows, int64_t W, int64_t J, float* ws, cudaStream_t s);
int launch_dbias_finish(int dt, const float* ws, int64_t J, int64_t W, void* dbias, cudaStream_t s);

// Device error words of the translation units whose kernels have bounded
// waits: each returns its word (nonzero after a timed-out wait) and clears
// it.  0 when nothing failed.
unsigned take_device_error_dropout();
unsigned take_device_error_glu();
unsigned take_device_error_gelu();
unsigned take_device_error_sqrelu();
unsigned take_device_error_softmax();

}  // namespace mfx
