// Block-granular selection: the indexer scores blocks of 2^lg consecutive
// positions through their mean-pooled key, Top-K keeps K / 2^lg blocks, and
// exact attention runs over every visible position of the kept blocks
// ("Sparse Attention and Hybrid Attention Architecture Design", block-level
// routing: keys pooled per block, blocks scored and selected, attention
// inside the selected blocks). The scoring, selection and attention kernels
// are the token-level ones; this file holds the three small steps around
// them: pooling, the per-row block count, and the block-to-position expansion.
#include "common.cuh"
#include "kernels.h"

namespace sa {
namespace {

// One thread per (block, column pair): the mean of the block's rows in fp32,
// rounded to bf16 (a block past N averages the rows it has).
__global__ void pool_keys_kernel(const bf16* k, int64_t N, int di, int lg, bf16* out, int64_t nb)
{
    const int64_t pairs = (int64_t)di / 2;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < nb * pairs;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = x / pairs;
        const int d = (int)(x % pairs) * 2;
        const int64_t j0 = b << lg;
        const int64_t j1 = min64(N, j0 + ((int64_t)1 << lg));
        float s0 = 0.0f, s1 = 0.0f;
        for (int64_t j = j0; j < j1; ++j) {
            const float2 f = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(k + j * di + d));
            s0 += f.x;
            s1 += f.y;
        }
        const float cnt = (float)(j1 - j0);
        *reinterpret_cast<uint32_t*>(out + b * di + d) = pack_bf16x2(s0 / cnt, s1 / cnt);
    }
}

__global__ void block_rowlen_kernel(int64_t t0, int rows, int lg, int32_t* row_len)
{
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < rows) row_len[r] = (int32_t)(((t0 + r) >> lg) + 1);
}

// One warp per row: kept block i (ascending) covers output slots
// [i 2^lg, (i+1) 2^lg); only the block holding t itself can be cut short, and
// it is the last kept block when kept, so the slots stay dense.
__global__ void expand_blocks_kernel(const int32_t* blk, int Kb, int64_t t0, int rows, int lg, int32_t* idx,
                                     int32_t* count)
{
    const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const int64_t t = t0 + r;
    const int B = 1 << lg;
    const int32_t* sel = blk + (int64_t)r * Kb;
    int32_t* out = idx + (int64_t)r * ((int64_t)Kb << lg);
    int nsel = 0;
    for (int i = 0; i < Kb; ++i) nsel += sel[i] >= 0 ? 1 : 0;     // -1 padding sits at the end
    int written = 0;
    for (int i = 0; i < nsel; ++i) {
        const int64_t p0 = (int64_t)sel[i] << lg;
        const int len = (int)min64(B, t - p0 + 1);                // positions <= t of this block
        for (int u = lane; u < B; u += 32) out[(int64_t)i * B + u] = u < len ? (int32_t)(p0 + u) : -1;
        written += len > 0 ? len : 0;
    }
    for (int64_t u = (int64_t)nsel * B + lane; u < ((int64_t)Kb << lg); u += 32) out[u] = -1;
    if (lane == 0) count[r] = written;
}

}  // namespace

cudaError_t launch_pool_keys(const void* k_idx, int64_t N, int di, int lg, void* pooled, cudaStream_t s)
{
    const int64_t nb = (N + ((int64_t)1 << lg) - 1) >> lg;
    if (nb <= 0) return cudaSuccess;
    const int64_t work = nb * (di / 2);
    const unsigned blocks = (unsigned)min64(4 * 148, (work + 255) / 256);
    pool_keys_kernel<<<blocks, 256, 0, s>>>(static_cast<const bf16*>(k_idx), N, di, lg, static_cast<bf16*>(pooled), nb);
    return cudaGetLastError();
}

cudaError_t launch_block_rowlen(int64_t t0, int rows, int lg, int32_t* row_len, cudaStream_t s)
{
    if (rows <= 0) return cudaSuccess;
    block_rowlen_kernel<<<(rows + 255) / 256, 256, 0, s>>>(t0, rows, lg, row_len);
    return cudaGetLastError();
}

cudaError_t launch_expand_blocks(const int32_t* blk, int Kb, int64_t t0, int rows, int lg, int32_t* idx,
                                 int32_t* count, cudaStream_t s)
{
    if (rows <= 0) return cudaSuccess;
    expand_blocks_kernel<<<(rows + 7) / 8, 256, 0, s>>>(blk, Kb, t0, rows, lg, idx, count);
    return cudaGetLastError();
}

}  // namespace sa
