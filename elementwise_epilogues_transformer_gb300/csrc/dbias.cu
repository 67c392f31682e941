// dbias.cu -- the deterministic second stage of the fused bias gradients,
// and the column-partial pass the unaligned fallbacks use.
//
// The page's backward returns one gradient tensor for the input and for the
// broadcast bias, and autograd sums it over the rows (Megatron-LM operator
// fusion walkthrough, www.wmrh.cn/news/51426, §4.3).  The fused kernels
// leave J partial sums per column in a workspace [J, W] (fp32); here each
// column's J partials are added in the fixed order j = 0 .. J-1 and the
// result is rounded once to the bias dtype.
#include "mfx_device.cuh"
#include "mfx_host.h"

namespace mfx {
namespace {

template <typename T>
__global__ void __launch_bounds__(kThreads)
dbias_finish(const float* __restrict__ ws, int64_t J, int64_t W, T* __restrict__ dbias)
{
    const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (c >= W)
        return;
    float s = 0.0f;
    for (int64_t j = 0; j < J; ++j)
        s += ws[j * W + c];
    store1(dbias + c, s);
}

// Partial column sums of a stored [rows, W] tensor: block (x, j) adds rows
// j, j + J, ... of columns [256 x, 256 x + 256) in row order.
template <typename T>
__global__ void __launch_bounds__(kThreads)
column_partials(const T* __restrict__ src, int64_t rows, int64_t W, int64_t J, float* __restrict__ ws)
{
    const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t j = blockIdx.y;
    if (c >= W)
        return;
    float s = 0.0f;
    for (int64_t r = j; r < rows; r += J)
        s += load1(src + r * W + c);
    ws[j * W + c] = s;
}

}  // namespace

int launch_dbias_finish(int dt, const float* ws, int64_t J, int64_t W, void* dbias, cudaStream_t s)
{
    const unsigned blocks = (unsigned)((W + kThreads - 1) / kThreads);
    if (dt == MFX_BF16)
        dbias_finish<bf16><<<blocks, kThreads, 0, s>>>(ws, J, W, static_cast<bf16*>(dbias));
    else
        dbias_finish<float><<<blocks, kThreads, 0, s>>>(ws, J, W, static_cast<float*>(dbias));
    return launch_status();
}

int launch_column_partials(int dt, const void* src, int64_t rows, int64_t W, int64_t J, float* ws, cudaStream_t s)
{
    const dim3 grid((unsigned)((W + kThreads - 1) / kThreads), (unsigned)J);
    if (dt == MFX_BF16)
        column_partials<bf16><<<grid, kThreads, 0, s>>>(static_cast<const bf16*>(src), rows, W, J, ws);
    else
        column_partials<float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(src), rows, W, J, ws);
    return launch_status();
}

int64_t dbias_generic_lanes(int64_t rows) { return rows < kGenericLanes ? (rows > 0 ? rows : 1) : kGenericLanes; }

// Workspace protocol shared by the *_dbias entry points.
int dbias_workspace(int64_t J, int64_t W, void* workspace, size_t* workspace_bytes, bool* query)
{
    *query = false;
    if (!workspace_bytes)
        return MFX_ERR_NULL;
    const size_t need = (size_t)J * (size_t)W * sizeof(float);
    if (!workspace) {
        *workspace_bytes = need;
        *query = true;
        return MFX_OK;
    }
    if (*workspace_bytes < need || !aligned16(workspace))
        return MFX_ERR_WORKSPACE;
    return MFX_OK;
}

}  // namespace mfx
