// Indexer score on CUDA cores (fp32 FFMA), every input format.
//
//   s[t, j] = sum_h w[t,h] * max(0, q_idx[t,h,:] . k_idx[j,:])     (j < n_t)
//
// The relevance score of each query against each causal history position
// ("Hybrid Attention Architectures...", section 3.1, indexing stage). This
// kernel is the general path: fp32 inputs, and any shape the tensor-core
// kernel does not cover. One thread owns one key; a CTA covers TQ queries x
// 128 keys; q for the TQ queries sits in shared memory as fp32 with its FP8
// scale already applied, the key scale multiplies the finished dot product
// (a positive factor commutes with the ReLU).
#include "common.cuh"
#include "kernels.h"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int KEYS_PER_CTA = 128;

template <int HP>   // heads padded to a power of two; TQ * HP == 32
__global__ void __launch_bounds__(KEYS_PER_CTA)
indexer_simt_kernel(IndexerArgs a)
{
    constexpr int TQ = 32 / HP;
    extern __shared__ float qs[];           // [TQ][HP][di]
    const int di = a.di, Hi = a.Hi;
    const int t0 = a.t_begin + blockIdx.x * TQ;
    const int j0 = blockIdx.y * KEYS_PER_CTA;
    const int t_last = min(t0 + TQ, a.T) - 1;
    const int64_t n_last = indexer_row_n(a, t_last);
    if (j0 >= n_last) return;               // the whole tile is beyond every row's history

    for (int i = threadIdx.x; i < TQ * HP * di; i += blockDim.x) {
        const int d = i % di, h = (i / di) % HP, tq = i / (di * HP);
        const int t = t0 + tq;
        float v = 0.0f;
        if (t < a.T && h < Hi) {
            const int64_t e = ((int64_t)t * Hi + h) * di + d;
            if (a.dtype == SA_F32) v = static_cast<const float*>(a.q_idx)[e];
            else if (a.dtype == SA_BF16) v = to_f32(static_cast<const bf16*>(a.q_idx)[e]);
            else v = e4m3_to_f32(static_cast<const uint8_t*>(a.q_idx)[e]) * a.q_scale[(int64_t)t * Hi + h];
        }
        qs[i] = v;
    }
    __syncthreads();

    const int j = j0 + threadIdx.x;
    const bool jv = j < a.N;
    float acc[32];
#pragma unroll
    for (int p = 0; p < 32; ++p) acc[p] = 0.0f;

    for (int d0 = 0; d0 < di; d0 += 8) {
        float kv[8];
        if (a.dtype == SA_F32) {
            const float4* kp = reinterpret_cast<const float4*>(static_cast<const float*>(a.k_idx) + (int64_t)j * di + d0);
            float4 x = jv ? kp[0] : make_float4(0, 0, 0, 0);
            float4 y = jv ? kp[1] : make_float4(0, 0, 0, 0);
            kv[0] = x.x; kv[1] = x.y; kv[2] = x.z; kv[3] = x.w;
            kv[4] = y.x; kv[5] = y.y; kv[6] = y.z; kv[7] = y.w;
        } else if (a.dtype == SA_BF16) {
            uint4 x = jv ? *reinterpret_cast<const uint4*>(static_cast<const bf16*>(a.k_idx) + (int64_t)j * di + d0)
                         : make_uint4(0, 0, 0, 0);
            float2 f;
            f = bf16x2_to_f32x2(x.x); kv[0] = f.x; kv[1] = f.y;
            f = bf16x2_to_f32x2(x.y); kv[2] = f.x; kv[3] = f.y;
            f = bf16x2_to_f32x2(x.z); kv[4] = f.x; kv[5] = f.y;
            f = bf16x2_to_f32x2(x.w); kv[6] = f.x; kv[7] = f.y;
        } else {
            uint2 x = jv ? *reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(a.k_idx) + (int64_t)j * di + d0)
                         : make_uint2(0, 0);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kv[e] = e4m3_to_f32((x.x >> (8 * e)) & 0xff);
                kv[4 + e] = e4m3_to_f32((x.y >> (8 * e)) & 0xff);
            }
        }
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            const float4 q0 = *reinterpret_cast<const float4*>(&qs[p * di + d0]);
            const float4 q1 = *reinterpret_cast<const float4*>(&qs[p * di + d0 + 4]);
            float s = acc[p];
            s = fmaf(q0.x, kv[0], s); s = fmaf(q0.y, kv[1], s);
            s = fmaf(q0.z, kv[2], s); s = fmaf(q0.w, kv[3], s);
            s = fmaf(q1.x, kv[4], s); s = fmaf(q1.y, kv[5], s);
            s = fmaf(q1.z, kv[6], s); s = fmaf(q1.w, kv[7], s);
            acc[p] = s;
        }
    }

    if (!jv) return;
    const float ks = (a.dtype == SA_FP8_E4M3) ? a.k_scale[j] : 1.0f;
#pragma unroll
    for (int tq = 0; tq < TQ; ++tq) {
        const int t = t0 + tq;
        if (t >= a.T) break;
        const int64_t n_t = indexer_row_n(a, t);
        if (j >= n_t) continue;
        float s = 0.0f;
#pragma unroll
        for (int h = 0; h < HP; ++h) {
            if (h < Hi) s = fmaf(a.w[(int64_t)t * Hi + h], fmaxf(acc[tq * HP + h] * ks, 0.0f), s);
        }
        a.scores[(int64_t)(t - a.t_begin) * a.ld_s + j] = s;
    }
}

template <int HP>
cudaError_t launch_hp(const IndexerArgs& a, cudaStream_t s)
{
    constexpr int TQ = 32 / HP;
    const int rows = a.T - a.t_begin;
    dim3 grid((rows + TQ - 1) / TQ, (a.N + KEYS_PER_CTA - 1) / KEYS_PER_CTA);
    const size_t smem = sizeof(float) * TQ * HP * a.di;
    indexer_simt_kernel<HP><<<grid, KEYS_PER_CTA, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_simt(const IndexerArgs& a, cudaStream_t s)
{
    if (a.thr) return cudaErrorNotSupported;                 // filter mode is tensor-core only
    if (a.T - a.t_begin <= 0 || a.N <= 0) return cudaSuccess;
    if (a.Hi <= 1) return launch_hp<1>(a, s);
    if (a.Hi <= 2) return launch_hp<2>(a, s);
    if (a.Hi <= 4) return launch_hp<4>(a, s);
    if (a.Hi <= 8) return launch_hp<8>(a, s);
    if (a.Hi <= 16) return launch_hp<16>(a, s);
    return launch_hp<32>(a, s);
}

cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s)
{
    if (indexer_tc_supported(a)) {
        const cudaError_t e = launch_indexer_tc(a, s);
        if (e != cudaErrorNotSupported) return e;
    }
    return launch_indexer_simt(a, s);
}

}  // namespace sa
