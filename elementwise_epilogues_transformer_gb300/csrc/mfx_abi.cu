// mfx_abi.cu -- status strings, the thread-local CUDA error, device queries
// and the launch-geometry plan shared by every entry point.
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>
#include <utility>

#include "mfx_host.h"

namespace mfx {

namespace {
thread_local int g_last_cuda_error = 0;

// Launch-geometry caches, shared by all host threads under one mutex:
// (device, kernel, block threads, dynamic shared memory) -> resident blocks
// per SM, and (device, kernel) -> the largest dynamic shared-memory limit set
// so far.  The limit only ever grows, so a launch planned with a cached
// occupancy always finds its shared memory allowed, whatever sizes other
// calls (or threads) launched the same kernel with in between.
struct OccKey {
    int device;
    const void* kernel;
    int threads;
    size_t smem;
    bool operator==(const OccKey& o) const
    {
        return device == o.device && kernel == o.kernel && threads == o.threads && smem == o.smem;
    }
};
struct OccHash {
    size_t operator()(const OccKey& k) const
    {
        size_t h = std::hash<const void*>()(k.kernel);
        h ^= (size_t)k.device * 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= (size_t)k.threads * 0xBF58476D1CE4E5B9ull + (h << 6) + (h >> 2);
        h ^= k.smem * 0x94D049BB133111EBull + (h << 6) + (h >> 2);
        return h;
    }
};
struct FnKeyHash {
    size_t operator()(const std::pair<int, const void*>& k) const
    {
        return std::hash<const void*>()(k.second) ^ ((size_t)k.first * 0x9E3779B97F4A7C15ull);
    }
};
std::mutex g_occ_mutex;
std::unordered_map<OccKey, int, OccHash> g_occ;
std::unordered_map<std::pair<int, const void*>, size_t, FnKeyHash> g_smem_limit;

constexpr int kMaxDevices = 64;
thread_local int g_sms[kMaxDevices] = {0};

int64_t gcd64(int64_t a, int64_t b)
{
    while (b) {
        int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}
}  // namespace

int cuda_failure(cudaError_t e)
{
    g_last_cuda_error = (int)e;
    return MFX_ERR_CUDA;
}

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    if (dev >= 0 && dev < kMaxDevices && g_sms[dev] > 0)
        return g_sms[dev];
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (dev >= 0 && dev < kMaxDevices)
        g_sms[dev] = n;
    return n;
}

int occupancy(const void* kernel, int block_threads, size_t smem)
{
    int dev = 0;
    cudaGetDevice(&dev);
    const OccKey key{dev, kernel, block_threads, smem};
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    auto it = g_occ.find(key);
    if (it != g_occ.end())
        return it->second;
    if (smem > 48 * 1024) {
        size_t& lim = g_smem_limit[{dev, kernel}];
        if (smem > lim && cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
                              cudaSuccess)
            lim = smem;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block_threads, smem) != cudaSuccess || n < 1)
        n = 1;
    g_occ.emplace(key, n);
    return n;
}

int blocks_per_sm(const void* kernel) { return occupancy(kernel, kThreads, 0); }

Grid plan_grid(const void* kernel, int64_t units, int64_t row_units, bool want_fixed)
{
    return plan_grid_ex(kernel, kThreads, 0, units, row_units, want_fixed);
}

Grid plan_grid_ex(const void* kernel, int block_threads, size_t smem, int64_t units, int64_t row_units,
                  bool want_fixed)
{
    Grid g;
    const int64_t capacity = (int64_t)sm_count() * occupancy(kernel, block_threads, smem) * kThreads;
    if (want_fixed && row_units > 0) {
        const int64_t L = kThreads / gcd64(kThreads, row_units) * row_units;  // lcm
        if (L <= 4 * capacity) {
            int64_t k = capacity / L;  // at most one wave of blocks
            if (k < 1)
                k = 1;
            const int64_t k_need = (units + L - 1) / L;
            if (k > k_need)
                k = k_need > 0 ? k_need : 1;
            g.fixed = true;
            g.blocks = k * L / kThreads;
            g.S = k * L;
            return g;
        }
    }
    int64_t need = (units + kThreads - 1) / kThreads;
    int64_t cap_blocks = capacity / kThreads;
    g.blocks = need < cap_blocks ? need : cap_blocks;
    if (g.blocks < 1)
        g.blocks = 1;
    g.S = g.blocks * kThreads;
    return g;
}

Grid plan_fixed_any(const void* kernel, int block_threads, size_t smem, int64_t units, int64_t cols)
{
    Grid g;
    const int64_t capacity = (int64_t)sm_count() * occupancy(kernel, block_threads, smem) * kThreads;
    const int64_t P = cols / gcd64(cols, 8);
    if (units < 1 || P > 4 * capacity)
        return g;
    // at most one wave: a block beyond the resident slots would run its whole
    // share after the others finish
    int64_t k = capacity / P;
    if (k < 1)
        k = 1;
    const int64_t k_need = (units + P - 1) / P;
    if (k > k_need)
        k = k_need;
    g.fixed = true;
    g.S = k * P;
    g.blocks = (g.S + kThreads - 1) / kThreads;
    return g;
}

}  // namespace mfx

extern "C" {

const char* mfx_status_string(int status)
{
    switch (status) {
    case MFX_OK: return "ok";
    case MFX_ERR_NULL: return "a required pointer is NULL";
    case MFX_ERR_SHAPE: return "negative or overflowing tensor sizes";
    case MFX_ERR_DTYPE: return "unknown dtype code";
    case MFX_ERR_PROB: return "dropout probability outside [0, 1)";
    case MFX_ERR_ALIAS: return "buffers overlap in a way the operation does not allow";
    case MFX_ERR_CUDA: return "CUDA launch failed (see mfx_last_cuda_error)";
    case MFX_ERR_DEVICE: return "a kernel gave up a bounded wait (see mfx_device_error)";
    case MFX_ERR_WORKSPACE: return "workspace too small or not 16-byte aligned";
    default: return "unknown status";
    }
}

int mfx_last_cuda_error(void) { return mfx::g_last_cuda_error; }

int mfx_device_error(unsigned* code)
{
    // one byte per source file: dropout, GLU, GeLU; the top byte holds the
    // squared ReLU's codes in its low nibble and the softmax's in its high one
    unsigned c = (mfx::take_device_error_dropout() & 0xFFu) | (mfx::take_device_error_glu() & 0xFFu) << 8 |
                 (mfx::take_device_error_gelu() & 0xFFu) << 16 | (mfx::take_device_error_sqrelu() & 0xFu) << 24 |
                 (mfx::take_device_error_softmax() & 0xFu) << 28;
    if (code)
        *code = c;
    return c ? MFX_ERR_DEVICE : MFX_OK;
}

int mfx_version(void) { return (1 << 16) | 3; }

}  // extern "C"
