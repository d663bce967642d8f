// Exact per-row Top-K ("Hybrid Attention Architectures...", section 3.1,
// filtering stage: keep the K highest-scoring positions; an exact tie goes to
// the lower position). Used by topk_select and by the prefill path.
//
// One CTA per row, scores compared through order-preserving 32-bit keys.
//   n <= K        every position is kept.
//   n <= 16384    the row's keys are staged in shared memory once, then an
//                 MSB-first radix select (8-bit digits) finds the K-th key and
//                 one ordered pass emits the kept positions.
//   longer rows   a sample guides one streaming pass:
//     1. a strided sample of ~n/16 keys (blocks of 8 consecutive keys, one
//        32-byte sector each) is counted into a 4096-bin histogram of the
//        keys' top 12 bits, then the samples of the bin holding the k'-th
//        best (k' = the sample's share of K plus a six-sigma margin) into a
//        histogram of the next 12 bits; the resulting 24-bit prefix is a
//        lower bound T_lo that at least K keys of the row reach almost
//        surely, while only a few thousand do;
//     2. one pass over the row keeps the positions with key >= T_lo, in
//        ascending order (block prefix sums), as (key << 32 | ~position)
//        composites;
//     3. a 4096-bin histogram over equal slices of [T_lo, max candidate key]
//        gives the slice of the K-th best; a radix search over the
//        candidates of that slice alone finds the exact boundary (by key,
//        then by lower position);
//     4. the kept candidates are emitted in their (ascending) order.
//   If fewer than K or more than the list holds reach T_lo, or the boundary
//   bin is too crowded, the row falls back to the radix select over the whole
//   row, so the result is exact in every case.
// The output lists min(K, n) positions in ascending order, then -1 padding.
#include "common.cuh"
#include "kernels.h"
#include "topk_core.cuh"

namespace sa {
namespace {

constexpr int TK_THREADS = 512;
constexpr int STAGE_MAX = 16384;             // keys staged in shared memory (64 KB)
constexpr int SAMPLE_BLOCKS = 1024;          // sampled 8-key blocks at most
constexpr int CAND_CAP = 5120;               // candidate composites (40 KB)
constexpr int BIN_CAP = 1024;                // composites of the boundary bin (8 KB)
constexpr int PER_THREAD = 16;               // consecutive positions per thread per pass step
constexpr int SAMPLE_MAX = SAMPLE_BLOCKS * 8;     // sampled keys kept in shared memory (32 KB)
constexpr size_t TK_SMEM_LONG = HBINS * 4 + SAMPLE_MAX * 4 + CAND_CAP * 8 + BIN_CAP * 8;
constexpr size_t TK_SMEM = STAGE_MAX * 4 > TK_SMEM_LONG ? STAGE_MAX * 4 : TK_SMEM_LONG;

SA_DEVINL int64_t topk_row_len(const TopkArgs& a, int r)
{
    int64_t n = a.row_len ? (int64_t)a.row_len[r] : a.causal_first + r + 1;
    return n < 0 ? 0 : (n > a.n_cap ? a.n_cap : n);
}

// 16 consecutive scores from position j0 as keys; positions >= n give 0
// (below every score's key). Vector loads when the run is aligned and whole.
SA_DEVINL void load16(const float* row, int64_t j0, int64_t n, bool aligned, uint32_t (&k)[PER_THREAD])
{
    if (aligned && j0 + PER_THREAD <= n) {
        const float4* p = reinterpret_cast<const float4*>(row + j0);
#pragma unroll
        for (int i = 0; i < PER_THREAD / 4; ++i) {
            const float4 v = __ldcs(p + i);
            k[4 * i] = score_key(v.x); k[4 * i + 1] = score_key(v.y);
            k[4 * i + 2] = score_key(v.z); k[4 * i + 3] = score_key(v.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < PER_THREAD; ++i) k[i] = j0 + i < n ? score_key(__ldcs(row + j0 + i)) : 0u;
    }
}

// Sample-guided selection of a long row (n > STAGE_MAX). Returns false if the
// sample's bound did not isolate between K and CAND_CAP candidates, or the
// boundary bin holds more than BIN_CAP of them.
__device__ bool sampled_select(const float* row, int64_t n, int K, int32_t* out, unsigned* hist,
                               uint32_t* samp, unsigned long long* cand, unsigned long long* bcand,
                               RadixShared& sh, BinSplit* split)
{
    const int tid = threadIdx.x;
    const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    // 1. sample histogram: blocks of 8 consecutive keys, one every S positions
    const int64_t S = max64(16, ((n + SAMPLE_BLOCKS - 1) / SAMPLE_BLOCKS + 7) / 8 * 8);
    const int nblk = (int)((n + S - 1) / S);
    for (int i = tid; i < HBINS; i += TK_THREADS) hist[i] = 0;
    __syncthreads();
    // warp-uniform trip count, so that the whole warp meets the match below
    for (int b0 = tid & ~31; b0 < nblk; b0 += TK_THREADS) {
        const int b = b0 + (tid & 31);
        const int64_t j0 = (int64_t)b * S;
        uint32_t k[8];
        if (b >= nblk) {
#pragma unroll
            for (int i = 0; i < 8; ++i) k[i] = 0u;
        } else if (aligned && j0 + 8 <= n) {
            const float4 v0 = __ldcs(reinterpret_cast<const float4*>(row + j0));
            const float4 v1 = __ldcs(reinterpret_cast<const float4*>(row + j0) + 1);
            k[0] = score_key(v0.x); k[1] = score_key(v0.y); k[2] = score_key(v0.z); k[3] = score_key(v0.w);
            k[4] = score_key(v1.x); k[5] = score_key(v1.y); k[6] = score_key(v1.z); k[7] = score_key(v1.w);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) k[i] = j0 + i < n ? score_key(__ldcs(row + j0 + i)) : 0u;
        }
        // samples crowd into few bins: one atomic per distinct bin per warp
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool valid = b < nblk && j0 + i < n;
            if (b < nblk) samp[b * 8 + i] = valid ? k[i] : 0u;
            const uint32_t bin = valid ? key_bin(k[i]) : (uint32_t)HBINS;
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, bin);
            if (bin < (uint32_t)HBINS && (threadIdx.x & 31) == __ffs(peers) - 1)
                atomicAdd(&hist[bin], (unsigned)__popc(peers));
        }
    }
    const int64_t tail = n - (int64_t)(nblk - 1) * S;
    const int m = (nblk - 1) * 8 + (int)min64(8, tail);          // valid samples
    const double share = (double)K * (double)m / (double)n;
    const double kq_d = ceil(share + 6.0 * sqrt(share) + 16.0);
    __syncthreads();
    if (kq_d >= (double)m) return false;
    const BinSplit sb = find_bin(hist, (unsigned)kq_d, sh.warp_tot, split);
    // refine inside that bin with the next 12 key bits, so that the bound sits
    // just below the sample's k'-th best key rather than a whole bin lower
    for (int i = tid; i < HBINS; i += TK_THREADS) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < nblk * 8; i += TK_THREADS) {
        const uint32_t k = samp[i];
        if (key_bin(k) == (uint32_t)sb.bin && k != 0u) atomicAdd(&hist[(k >> (HSHIFT - HBITS)) & (HBINS - 1)], 1u);
    }
    __syncthreads();
    const BinSplit sb2 = find_bin(hist, (unsigned)kq_d - sb.above, sh.warp_tot, split);
    const uint32_t lo = ((uint32_t)sb.bin << HSHIFT) | ((uint32_t)sb2.bin << (HSHIFT - HBITS));

    // 2. one pass over the row: positions with key >= lo, in ascending order;
    //    the next step's loads are issued before this step's prefix sum
    unsigned written = 0;
    uint32_t kmax = lo;
    uint32_t kc[PER_THREAD], kn[PER_THREAD];
    const int64_t step = (int64_t)TK_THREADS * PER_THREAD;
    load16(row, (int64_t)tid * PER_THREAD, n, aligned, kn);
    for (int64_t base = 0; base < n; base += step) {
#pragma unroll
        for (int i = 0; i < PER_THREAD; ++i) kc[i] = kn[i];
        const int64_t j0 = base + (int64_t)tid * PER_THREAD;
        if (base + step < n) load16(row, j0 + step, n, aligned, kn);
        unsigned c = 0;
#pragma unroll
        for (int i = 0; i < PER_THREAD; ++i) c += (j0 + i < n && kc[i] >= lo) ? 1u : 0u;
        unsigned total;
        const unsigned incl = block_scan_incl(c, sh.warp_tot, &total);
        unsigned pos = written + incl - c;
#pragma unroll
        for (int i = 0; i < PER_THREAD; ++i) {
            if (j0 + i < n && kc[i] >= lo) {
                kmax = max(kmax, kc[i]);
                if (pos < (unsigned)CAND_CAP)
                    cand[pos] = ((unsigned long long)kc[i] << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)(j0 + i));
                ++pos;
            }
        }
        written += total;
    }
    kmax = block_max_u32(kmax, sh.warp_tot);
    if (written < (unsigned)K || written > (unsigned)CAND_CAP) return false;

    // 3. the exact boundary among the candidates
    CandBoundary cb;
    if (!cand_boundary(cand, written, lo, kmax, (unsigned)K, hist, bcand, BIN_CAP, sh, split, cb)) return false;

    // 4. emit the kept candidates in their ascending order
    unsigned emitted = 0;
    for (unsigned i0 = 0; i0 < written; i0 += TK_THREADS) {
        const unsigned i = i0 + tid;
        bool keep = false;
        unsigned long long c = 0;
        if (i < written) {
            c = cand[i];
            keep = cand_keep(c, cb);
        }
        unsigned total;
        const unsigned incl = block_scan_incl(keep ? 1u : 0u, sh.warp_tot, &total);
        if (keep && emitted + incl - 1 < (unsigned)K) out[emitted + incl - 1] = (int32_t)(0xFFFFFFFFu - (uint32_t)c);
        emitted += total;
    }
    return true;
}

__global__ void __launch_bounds__(TK_THREADS, 2)
topk_rows_kernel(TopkArgs a)
{
    __shared__ RadixShared sh;
    __shared__ BinSplit split;
    extern __shared__ __align__(16) unsigned char tk_smem[];
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t n = topk_row_len(a, r);
    const int K = a.K;
    int32_t* out = a.idx + (int64_t)r * a.ld_idx;
    const float* row = a.scores + (int64_t)r * a.ld_s;

    if (n <= K) {                            // keep everything, in order
        for (int i = tid; i < K; i += TK_THREADS) out[i] = i < n ? i : -1;
        return;
    }
    if (n <= STAGE_MAX) {
        uint32_t* keys = reinterpret_cast<uint32_t*>(tk_smem);
        for (int64_t j = tid; j < n; j += TK_THREADS) keys[j] = score_key(row[j]);
        __syncthreads();
        radix_select_row([&](int64_t j) { return keys[j]; }, n, K, out, sh, keys);
        return;
    }
    unsigned* hist = reinterpret_cast<unsigned*>(tk_smem);
    uint32_t* samp = reinterpret_cast<uint32_t*>(tk_smem + HBINS * 4);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(tk_smem + HBINS * 4 + SAMPLE_MAX * 4);
    unsigned long long* bcand = cand + CAND_CAP;
    if (!sampled_select(row, n, K, out, hist, samp, cand, bcand, sh, &split)) {
        __syncthreads();
        radix_select_row([&](int64_t j) { return score_key(__ldcg(row + j)); }, n, K, out, sh);
    }
}

// Rows that all fit the stage (n_cap <= STAGE_MAX): small CTAs, so that many
// rows are in flight per SM (one row's radix passes are short and end in
// block barriers), and shared memory sized to the longest row.
template <int NT>
__global__ void __launch_bounds__(NT)
topk_short_kernel(TopkArgs a)
{
    __shared__ RadixShared sh;
    extern __shared__ __align__(16) unsigned char tk_smem[];
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t n = topk_row_len(a, r);
    const int K = a.K;
    int32_t* out = a.idx + (int64_t)r * a.ld_idx;
    const float* row = a.scores + (int64_t)r * a.ld_s;
    if (n <= K) {
        for (int i = tid; i < K; i += NT) out[i] = i < n ? i : -1;
        return;
    }
    // stage the row's keys and count their top digits (the radix select's
    // first pass) on the way
    uint32_t* keys = reinterpret_cast<uint32_t*>(tk_smem);
    for (int i = tid; i < RADIX; i += NT) sh.hist[i] = 0;
    __syncthreads();
    int64_t j_tail = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
        const int64_t n4 = n / 4;
        const float4* r4 = reinterpret_cast<const float4*>(row);
        uint4* k4 = reinterpret_cast<uint4*>(keys);
#pragma unroll 4
        for (int64_t i = tid; i < n4; i += NT) {
            const float4 v = __ldcs(r4 + i);
            const uint4 k = make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
            k4[i] = k;
            atomicAdd(&sh.hist[k.x >> 24], 1u); atomicAdd(&sh.hist[k.y >> 24], 1u);
            atomicAdd(&sh.hist[k.z >> 24], 1u); atomicAdd(&sh.hist[k.w >> 24], 1u);
        }
        j_tail = n4 * 4;
    }
    for (int64_t j = j_tail + tid; j < n; j += NT) {
        const uint32_t k = score_key(__ldcs(row + j));
        keys[j] = k;
        atomicAdd(&sh.hist[k >> 24], 1u);
    }
    __syncthreads();
    radix_select_row<true>([&](int64_t j) { return keys[j]; }, n, K, out, sh, keys);
}

constexpr int TK_SHORT_THREADS = 128;

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
    if (a.n_cap > a.K && a.n_cap <= STAGE_MAX) {
        const size_t ssm = ((size_t)a.n_cap * 4 + 15) / 16 * 16;
        cudaError_t e = cudaFuncSetAttribute(topk_short_kernel<TK_SHORT_THREADS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        topk_short_kernel<TK_SHORT_THREADS><<<a.rows, TK_SHORT_THREADS, ssm, s>>>(a);
        return cudaGetLastError();
    }
    const size_t smem = a.n_cap <= a.K ? 0 : TK_SMEM;
    if (smem) {
        cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
    }
    topk_rows_kernel<<<a.rows, TK_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sa
