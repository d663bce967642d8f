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
// FP8-e4m3 keys (one fp32 scale per cached row) run the m16n8k32 e4m3 shape
// with the same byte mapping (a lane's 16-byte piece again feeds two
// k-steps, now of 32 codes each), which halves the bytes the scan streams.
// As in the prefill indexer, the query-row scale is folded into the head
// weight and the key scale multiplies the finished head sum (a positive
// factor commutes with the ReLU):
//   s[b, j] = sk[j] * sum_h (w[b,h] sq[b,h]) * max(0, q8[b,h,:] . k8[j,:])
//
// Work split: every row is cut into chunks of 1024 keys, and the grid (two
// CTAs per SM) splits the concatenated chunks of all rows into equal
// contiguous ranges, so that ragged batches (a few long rows, many short
// ones) keep every SM streaming; a CTA's chunks of one row are consecutive.
//
// Every CTA also counts its scores into a 4096-bin histogram of the top 12
// bits of their order-preserving keys (shared-memory atomics), and adds the
// non-zero bins to the sequence's histogram in global memory once per row it
// touched: the Top-K step reads that histogram to find the bin of the K-th
// best score without another pass over the scores.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "topk_core.cuh"

namespace sa {
namespace {

constexpr int SCAN_THREADS = 256;           // 8 warps
constexpr int SCAN_CHUNK = 1024;            // keys per chunk; a CTA takes a contiguous run of chunks
constexpr int SCAN_MAX_B = 2048;            // rows per launch (larger batches take several launches)
// 16-key groups in flight per warp: about 8 KB of key rows per warp
__host__ __device__ constexpr int scan_unroll(int row_bytes) { return row_bytes <= 128 ? 4 : (row_bytes == 256 ? 2 : 1); }

template <int DI, int NTH, bool FP8>
__device__ __forceinline__ void decode_scan_body(const DecodeScanArgs& a)
{
    constexpr int RB = FP8 ? DI : 2 * DI;    // bytes per key row
    constexpr int KS = FP8 ? DI / 32 : DI / 16;   // k-steps
    constexpr int VM = RB / 64;              // 16-byte pieces per key row per lane
    constexpr int SCAN_UNROLL_DI = FP8 ? 2 * scan_unroll(2 * DI) : scan_unroll(RB);
    griddep_wait();                          // the zeroed histogram and tickets
    griddep_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    __shared__ unsigned sh_hist[HBINS];
    __shared__ int sh_prefix[SCAN_MAX_B + 1];  // chunks of the launch's rows before row b
    __shared__ unsigned warp_tot[32];
    __shared__ int sh_last;
    __shared__ BinSplit split;
    auto row_len = [&](int b) -> int64_t {
        const int64_t n = a.ctx_len[a.b_begin + b];
        return n < 0 ? 0 : (n > a.max_ctx ? a.max_ctx : n);
    };
    for (int i = tid; i < HBINS; i += SCAN_THREADS) sh_hist[i] = 0;
    if (tid == 0) sh_prefix[0] = 0;
    int carry = 0;
    for (int b0 = 0; b0 < a.nb; b0 += SCAN_THREADS) {
        const int b = b0 + tid;
        const unsigned c = b < a.nb ? (unsigned)((row_len(b) + a.chunk - 1) / a.chunk) : 0u;
        unsigned total;
        const unsigned incl = block_scan_incl(c, warp_tot, &total);
        if (b < a.nb) sh_prefix[b + 1] = carry + (int)incl;
        carry += (int)total;
    }
    __syncthreads();
    // this CTA's contiguous range of the launch's chunks (consecutive chunks
    // of one row stay in one CTA, so its histogram is flushed once per row)
    const int64_t total = sh_prefix[a.nb];
    const int c_begin = (int)((int64_t)blockIdx.x * total / gridDim.x);
    const int c_end = (int)((int64_t)(blockIdx.x + 1) * total / gridDim.x);
    if (c_begin >= c_end) return;
    int b = 0;
    {
        int hi = a.nb;                       // sh_prefix[b] <= c_begin < sh_prefix[hi]
        while (hi - b > 1) {
            const int mid = (b + hi) >> 1;
            if (sh_prefix[mid] <= c_begin) b = mid; else hi = mid;
        }
    }

    uint32_t bq[KS][NTH][2];
    float wl[NTH][2];
    using QT = typename std::conditional<FP8, uint8_t, bf16>::type;
    constexpr int QPE = 16 / (int)sizeof(QT);  // elements per 16-byte piece
    auto load_query = [&](int bl) {
        const int bg = a.b_begin + bl;
        const QT* q = static_cast<const QT*>(a.q_idx) + (int64_t)bg * a.Hi * DI;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) {
                const int h = nt * 8 + g;
                const int d = 4 * QPE * (kk >> 1) + QPE * t4 + (QPE / 2) * (kk & 1);
                uint2 v = make_uint2(0, 0);
                if (h < a.Hi) v = *reinterpret_cast<const uint2*>(q + h * DI + d);
                bq[kk][nt][0] = v.x;
                bq[kk][nt][1] = v.y;
            }
        }
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = nt * 8 + 2 * t4 + e;
                float wv = 0.0f;
                if (h < a.Hi) {
                    wv = a.w[(int64_t)bg * a.Hi + h];
                    if constexpr (FP8) wv *= a.q_scale[(int64_t)bg * a.Hi + h];
                }
                wl[nt][e] = wv;
            }
        }
    };
    // the row's counts go to its global histogram; the CTA that completes the
    // row's last chunk (atomic count, nothing waits) finds the bin of the
    // K-th best score once, for the Top-K step
    auto finish_row = [&](int bl, int done) {
        const int bg = a.b_begin + bl;
        __syncthreads();
        unsigned* gh = a.hist + (int64_t)bg * HBINS;
        for (int i = tid; i < HBINS; i += SCAN_THREADS) {
            const unsigned c = sh_hist[i];
            if (c) atomicAdd(gh + i, c);
            sh_hist[i] = 0;
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const unsigned chunks = (unsigned)(sh_prefix[bl + 1] - sh_prefix[bl]);
            sh_last = atomicAdd(a.row_tickets + bg, (unsigned)done) + (unsigned)done == chunks;
        }
        __syncthreads();
        if (sh_last) {
            __threadfence();
            stage_hist(sh_hist, gh);
            const BinSplit bs = find_bin(sh_hist, (unsigned)a.K, warp_tot, &split);
            if (tid == 0) a.split[bg] = bs;
            for (int i = tid; i < HBINS; i += SCAN_THREADS) sh_hist[i] = 0;
            __syncthreads();
        }
    };

    load_query(b);
    int done = 0;
    const uint64_t pol = l2_evict_first_policy();
    for (int c = c_begin; c < c_end; ++c) {
        if (c >= sh_prefix[b + 1]) {         // the next row (rows without chunks are skipped)
            finish_row(b, done);
            done = 0;
            do { ++b; } while (c >= sh_prefix[b + 1]);
            load_query(b);
        }
        const int bg = a.b_begin + b;
        const int64_t j0 = (int64_t)(c - sh_prefix[b]) * a.chunk;
        const int cnt = (int)min64(a.chunk, row_len(b) - j0);
        // key rows in elements of their storage type (bf16, or one e4m3 byte)
        using KT = typename std::conditional<FP8, uint8_t, bf16>::type;
        const KT* kb = static_cast<const KT*>(a.k_idx) + (a.seq_start[bg] + j0) * DI;
        constexpr int PE = 16 / (int)sizeof(KT);     // elements per 16-byte piece
        const float* ksc = nullptr;
        if constexpr (FP8) ksc = a.k_scale + a.seq_start[bg] + j0;
        float* sc = a.scores + (int64_t)bg * a.ld_s + j0;
        constexpr int STEP = 8 * 16 * SCAN_UNROLL_DI;   // keys per CTA iteration
        for (int base = warp * 16; base < cnt; base += STEP) {
            uint4 va[SCAN_UNROLL_DI][VM], vb[SCAN_UNROLL_DI][VM];
            float sa0[FP8 ? SCAN_UNROLL_DI : 1], sa1[FP8 ? SCAN_UNROLL_DI : 1];   // FP8 key scales (lanes with t4 == 0)
#pragma unroll
            for (int u = 0; u < SCAN_UNROLL_DI; ++u) {
                const int k0 = base + u * 8 * 16 + g, k1 = k0 + 8;
#pragma unroll
                for (int m = 0; m < VM; ++m) {
                    va[u][m] = k0 < cnt ? ldg_stream16_hint(kb + (int64_t)k0 * DI + 4 * PE * m + PE * t4, pol) : make_uint4(0, 0, 0, 0);
                    vb[u][m] = k1 < cnt ? ldg_stream16_hint(kb + (int64_t)k1 * DI + 4 * PE * m + PE * t4, pol) : make_uint4(0, 0, 0, 0);
                }
                if constexpr (FP8) {
                    sa0[u] = (t4 == 0 && k0 < cnt) ? __ldg(ksc + k0) : 0.0f;
                    sa1[u] = (t4 == 0 && k1 < cnt) ? __ldg(ksc + k1) : 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < SCAN_UNROLL_DI; ++u) {
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
                    for (int nt = 0; nt < NTH; ++nt) {
                        if constexpr (FP8) mma_16832_e4m3(acc[nt], af, bq[kk][nt][0], bq[kk][nt][1]);
                        else mma_16816(acc[nt], af, bq[kk][nt][0], bq[kk][nt][1]);
                    }
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
                if constexpr (FP8) {
                    s0 *= sa0[u];
                    s1 *= sa1[u];
                }
                if (t4 == 0) {
                    if (k0 < cnt) { sc[k0] = s0; atomicAdd(&sh_hist[key_bin(score_key(s0))], 1u); }
                    if (k1 < cnt) { sc[k1] = s1; atomicAdd(&sh_hist[key_bin(score_key(s1))], 1u); }
                }
            }
        }
        ++done;
    }
    finish_row(b, done);
}

template <int DI, int NTH>
__global__ void __launch_bounds__(SCAN_THREADS)
decode_scan_kernel(DecodeScanArgs a)
{
    decode_scan_body<DI, NTH, false>(a);
}

// FP8 keys: two CTAs per SM are kept for the single n-tile shape (its twice
// deeper unroll would otherwise take more than half the register file)
template <int DI, int NTH>
__global__ void __launch_bounds__(SCAN_THREADS, NTH == 1 ? 2 : 1)
decode_scan_fp8_kernel(DecodeScanArgs a)
{
    decode_scan_body<DI, NTH, true>(a);
}

__global__ void __launch_bounds__(256)
zero_kernel(uint4* p, size_t n16)
{
    griddep_launch();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_uint4(0, 0, 0, 0);
}

template <int DI>
cudaError_t launch_di(const DecodeScanArgs& a, cudaStream_t s)
{
    // about two CTAs per SM, each with an equal share of the rows' chunks
    const int64_t chunks_max = (int64_t)a.nb * ((a.max_ctx + a.chunk - 1) / a.chunk);
    const dim3 grid((unsigned)min64(chunks_max, 2 * (int64_t)device_sm_count()));
    if (a.fp8) {
        if constexpr (DI % 64 == 0) {
            if (a.Hi <= 8) return launch_kernel(decode_scan_fp8_kernel<DI, 1>, grid, dim3(SCAN_THREADS), 0, s, true, a);
            if (a.Hi <= 16) return launch_kernel(decode_scan_fp8_kernel<DI, 2>, grid, dim3(SCAN_THREADS), 0, s, true, a);
            return launch_kernel(decode_scan_fp8_kernel<DI, 4>, grid, dim3(SCAN_THREADS), 0, s, true, a);
        }
        return cudaErrorInvalidValue;
    }
    if (a.Hi <= 8) return launch_kernel(decode_scan_kernel<DI, 1>, grid, dim3(SCAN_THREADS), 0, s, true, a);
    if (a.Hi <= 16) return launch_kernel(decode_scan_kernel<DI, 2>, grid, dim3(SCAN_THREADS), 0, s, true, a);
    return launch_kernel(decode_scan_kernel<DI, 4>, grid, dim3(SCAN_THREADS), 0, s, true, a);
}

}  // namespace

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s)
{
    const size_t n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)min64(1184, (int64_t)((n16 + 255) / 256));
    zero_kernel<<<blocks, 256, 0, s>>>(static_cast<uint4*>(p), n16);
    return cudaGetLastError();
}

cudaError_t launch_decode_scan(const DecodeScanArgs& args, cudaStream_t s)
{
    if (args.B <= 0 || args.max_ctx <= 0) return cudaSuccess;
    DecodeScanArgs a = args;
    a.chunk = SCAN_CHUNK;
    for (a.b_begin = 0; a.b_begin < a.B; a.b_begin += SCAN_MAX_B) {
        a.nb = a.B - a.b_begin < SCAN_MAX_B ? a.B - a.b_begin : SCAN_MAX_B;
        cudaError_t e;
        switch (a.di) {
        case 32: e = launch_di<32>(a, s); break;
        case 64: e = launch_di<64>(a, s); break;
        case 128: e = launch_di<128>(a, s); break;
        case 256: e = launch_di<256>(a, s); break;
        default: e = cudaErrorInvalidValue; break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sa
