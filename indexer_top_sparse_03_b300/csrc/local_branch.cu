// The sliding-window local branch and its fusion with the sparse branch
// ("Sparse Attention and Hybrid Attention Architecture Design", branch
// fusion: a gate mixes the sparse branch with a local sliding-window branch,
// g * sparse + (1 - g) * local). The local branch is exact attention over the
// last W positions, run by the same attention kernels with a window index
// set; 1 - sigmoid(x) = sigmoid(-x), so the local branch uses the negated gate
// logits and the two gated outputs add up to the fused one.
#include "common.cuh"
#include "kernels.h"

namespace sa {
namespace {

__global__ void window_idx_kernel(int64_t t0, int rows, int W, int32_t* idx, int32_t* kept)
{
    const int64_t total = (int64_t)rows * W;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(x / W), i = (int)(x % W);
        const int64_t t = t0 + r;
        const int64_t first = t - W + 1 > 0 ? t - W + 1 : 0;
        const int64_t p = first + i;
        idx[x] = p <= t ? (int32_t)p : -1;
        if (i == 0) kept[r] = (int32_t)(t - first + 1);
    }
}

__global__ void negate_kernel(const float* x, float* neg, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        neg[i] = -x[i];
}

__global__ void add_bf16_kernel(uint32_t* out, const uint32_t* add, int64_t npairs)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npairs;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float2 a = bf16x2_to_f32x2(out[i]), b = bf16x2_to_f32x2(add[i]);
        out[i] = pack_bf16x2(a.x + b.x, a.y + b.y);
    }
}

unsigned grid_for(int64_t n) { return (unsigned)min64(8 * 148, (n + 255) / 256 > 0 ? (n + 255) / 256 : 1); }

}  // namespace

cudaError_t launch_window_idx(int64_t t0, int rows, int W, int32_t* idx, int32_t* kept, cudaStream_t s)
{
    if (rows <= 0) return cudaSuccess;
    window_idx_kernel<<<grid_for((int64_t)rows * W), 256, 0, s>>>(t0, rows, W, idx, kept);
    return cudaGetLastError();
}

cudaError_t launch_negate(const float* x, float* neg, int64_t n, cudaStream_t s)
{
    if (n <= 0) return cudaSuccess;
    negate_kernel<<<grid_for(n), 256, 0, s>>>(x, neg, n);
    return cudaGetLastError();
}

cudaError_t launch_add_bf16(void* out, const void* add, int64_t n, cudaStream_t s)
{
    if (n <= 0) return cudaSuccess;
    add_bf16_kernel<<<grid_for(n / 2), 256, 0, s>>>(static_cast<uint32_t*>(out), static_cast<const uint32_t*>(add),
                                                    n / 2);
    return cudaGetLastError();
}

}  // namespace sa
