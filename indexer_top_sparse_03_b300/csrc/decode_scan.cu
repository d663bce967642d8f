// Decode indexer scan: the score of each sequence's new query against every
// cached indexer key of that sequence ("Hybrid Attention Architectures...",
// section 3.1, indexing stage; the scan is the bandwidth-bound part of a
// decode step, "Sparse Attention and Hybrid Attention Architecture Design",
// section 1: decoding is memory-bandwidth bound).
//
//   s[b, j] = sum_h w[b,h] * max(0, q_idx[b,h,:] . k_idx[seq_start[b] + j,:])
//
// Keys are the M side of an m16n8k16 MMA (16 keys per warp step), indexer
// heads the N side (8 per n-tile, zero-padded). The dot product does not care
// in which order the dimensions are summed, so the k-slots of the MMA are
// mapped to physical dimensions such that every lane's A fragment for two
// k-steps is one contiguous 16-byte piece of a key row: lanes load their
// fragments straight from global memory (fully used 32-byte sectors), with
// no shared-memory staging, and q's B fragments use the same mapping.
//   k-step kk, fragment column c  ->  dim 32*(kk/2) + 8*((c%8)/2)
//                                        + 4*(kk%2) + 2*(c/8) + c%2
#include "common.cuh"
#include "kernels.h"

namespace sa {
namespace {

constexpr int SCAN_THREADS = 256;           // 8 warps
constexpr int SCAN_CHUNK = 4096;            // keys per CTA
constexpr int SCAN_UNROLL = 4;              // 16-key groups in flight per warp

template <int DI, int NTH>
__global__ void __launch_bounds__(SCAN_THREADS)
decode_scan_kernel(DecodeScanArgs a)
{
    constexpr int KS = DI / 16;              // k-steps
    constexpr int VM = DI / 32;              // 16-byte pieces per key row per lane
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    int64_t n = a.ctx_len[b];
    n = n < 0 ? 0 : (n > a.max_ctx ? a.max_ctx : n);
    const int64_t j0 = (int64_t)blockIdx.x * SCAN_CHUNK;
    if (j0 >= n) return;
    const int cnt = (int)min64(SCAN_CHUNK, n - j0);

    // q fragments (B operand) and head weights held by this lane
    const bf16* q = static_cast<const bf16*>(a.q_idx) + (int64_t)b * a.Hi * DI;
    uint32_t bq[KS][NTH][2];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
            const int h = nt * 8 + g;
            const int d = 32 * (kk >> 1) + 8 * t4 + 4 * (kk & 1);
            uint2 v = make_uint2(0, 0);
            if (h < a.Hi) v = *reinterpret_cast<const uint2*>(q + h * DI + d);
            bq[kk][nt][0] = v.x;
            bq[kk][nt][1] = v.y;
        }
    }
    float wl[NTH][2];
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = nt * 8 + 2 * t4 + e;
            wl[nt][e] = h < a.Hi ? a.w[(int64_t)b * a.Hi + h] : 0.0f;
        }
    }

    const bf16* kb = static_cast<const bf16*>(a.k_idx) + (a.seq_start[b] + j0) * DI;
    float* sc = a.scores + (int64_t)b * a.max_ctx + j0;
    constexpr int STEP = 8 * 16 * SCAN_UNROLL;   // keys per CTA iteration

    for (int base = warp * 16; base < cnt; base += STEP) {
        uint4 va[SCAN_UNROLL][VM], vb[SCAN_UNROLL][VM];
#pragma unroll
        for (int u = 0; u < SCAN_UNROLL; ++u) {
            const int k0 = base + u * 8 * 16 + g, k1 = k0 + 8;
#pragma unroll
            for (int m = 0; m < VM; ++m) {
                va[u][m] = k0 < cnt ? ldg_stream16(kb + (int64_t)k0 * DI + 32 * m + 8 * t4) : make_uint4(0, 0, 0, 0);
                vb[u][m] = k1 < cnt ? ldg_stream16(kb + (int64_t)k1 * DI + 32 * m + 8 * t4) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < SCAN_UNROLL; ++u) {
            float acc[NTH][4];
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const int m = kk >> 1;
                uint32_t af[4];
                af[0] = (kk & 1) ? va[u][m].z : va[u][m].x;
                af[2] = (kk & 1) ? va[u][m].w : va[u][m].y;
                af[1] = (kk & 1) ? vb[u][m].z : vb[u][m].x;
                af[3] = (kk & 1) ? vb[u][m].w : vb[u][m].y;
#pragma unroll
                for (int nt = 0; nt < NTH; ++nt) mma_16816(acc[nt], af, bq[kk][nt][0], bq[kk][nt][1]);
            }
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) {
                s0 = fmaf(wl[nt][0], fmaxf(acc[nt][0], 0.0f), s0);
                s0 = fmaf(wl[nt][1], fmaxf(acc[nt][1], 0.0f), s0);
                s1 = fmaf(wl[nt][0], fmaxf(acc[nt][2], 0.0f), s1);
                s1 = fmaf(wl[nt][1], fmaxf(acc[nt][3], 0.0f), s1);
            }
            s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
            s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            const int k0 = base + u * 8 * 16 + g, k1 = k0 + 8;
            if (t4 == 0) {
                if (k0 < cnt) sc[k0] = s0;
                if (k1 < cnt) sc[k1] = s1;
            }
        }
    }
}

template <int DI>
cudaError_t launch_di(const DecodeScanArgs& a, cudaStream_t s)
{
    dim3 grid((unsigned)((a.max_ctx + SCAN_CHUNK - 1) / SCAN_CHUNK), a.B);
    if (a.Hi <= 8) decode_scan_kernel<DI, 1><<<grid, SCAN_THREADS, 0, s>>>(a);
    else if (a.Hi <= 16) decode_scan_kernel<DI, 2><<<grid, SCAN_THREADS, 0, s>>>(a);
    else decode_scan_kernel<DI, 4><<<grid, SCAN_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_scan(const DecodeScanArgs& a, cudaStream_t s)
{
    if (a.B <= 0 || a.max_ctx <= 0) return cudaSuccess;
    switch (a.di) {
    case 32: return launch_di<32>(a, s);
    case 64: return launch_di<64>(a, s);
    case 128: return launch_di<128>(a, s);
    case 256: return launch_di<256>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sa
