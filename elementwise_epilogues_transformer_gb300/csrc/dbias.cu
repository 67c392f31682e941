// dbias.cu -- the deterministic second stage of the fused bias gradients,
// and the column-partial pass the unaligned fallbacks use.
//
// The page's backward returns one gradient tensor for the input and for the
// broadcast bias, and autograd sums it over the rows (Megatron-LM operator
// fusion walkthrough, www.wmrh.cn/news/51426, §4.3).  The fused kernels
// leave J partial sums per column in a workspace [J, W] (fp32); here each
// column's J partials are added in a fixed tree order (the same on every
// run) and the result is rounded once to the bias dtype.
#include "mfx_device.cuh"
#include "mfx_host.h"

namespace mfx {
namespace {

// Block: 32 columns x kFinishWarps warps.  Warp w takes partials j = w,
// w + kFinishWarps, ... into 8 interleaved sums (eight independent loads in
// flight per lane), adds them pairwise, and the warp sums are added in warp
// order: a fixed tree.  The kernel is a programmatic dependent of the kernel
// that wrote the partials and waits for it before the first read.
constexpr int kFinishWarps = 32;

template <typename T>
__global__ void __launch_bounds__(32 * kFinishWarps)
dbias_finish(const float* __restrict__ ws, int64_t J, int64_t W, T* __restrict__ dbias)
{
    __shared__ float part[kFinishWarps][33];
    pdl_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t c = (int64_t)blockIdx.x * 32 + lane;
    float a[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        a[k] = 0.0f;
    if (c < W) {
        int64_t j = w;
        for (; j + 7 * kFinishWarps < J; j += 8 * kFinishWarps) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                a[k] += ws[(j + k * kFinishWarps) * W + c];
        }
#pragma unroll
        for (int k = 0; k < 7; ++k)
            if (j + k * kFinishWarps < J)
                a[k] += ws[(j + k * kFinishWarps) * W + c];
    }
    part[w][lane] = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
    __syncthreads();
    if (w == 0 && c < W) {
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < kFinishWarps; ++k)
            s[k & 3] += part[k][lane];
        store1(dbias + c, (s[0] + s[1]) + (s[2] + s[3]));
    }
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((W + 31) / 32));
    cfg.blockDim = dim3(32 * kFinishWarps);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        dt == MFX_BF16 ? cudaLaunchKernelEx(&cfg, dbias_finish<bf16>, ws, J, W, static_cast<bf16*>(dbias))
                       : cudaLaunchKernelEx(&cfg, dbias_finish<float>, ws, J, W, static_cast<float*>(dbias));
    return e == cudaSuccess ? launch_status() : cuda_failure(e);
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
