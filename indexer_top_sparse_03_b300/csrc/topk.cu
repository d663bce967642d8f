// Exact per-row Top-K ("Hybrid Attention Architectures...", section 3.1,
// filtering stage: keep the K highest-scoring positions; an exact tie goes to
// the lower position). Used by topk_select and by the prefill path.
//
// One CTA per row, scores compared through order-preserving 32-bit keys.
//   n <= K        every position is kept.
//   n <= 16384    the row's keys are staged in shared memory once, then an
//                 MSB-first radix select (8-bit digits) finds the K-th key and
//                 one ordered pass emits the kept positions.
//   longer rows   a sample guides one streaming pass. A strided sample of
//                 ~n/16 keys (8-key blocks, one 32-byte sector each) gives a
//                 lower bound T_lo: the k'-th best sampled key, with k' the
//                 sample's expected share of K plus a six-sigma margin, so
//                 that almost surely at least K keys of the row reach T_lo
//                 while only a few thousand do. The pass over the row keeps
//                 the positions with key >= T_lo, in ascending order (block
//                 prefix sums), as (key << 32 | ~position) composites; an exact
//                 radix search over those composites then picks the K best and
//                 they are emitted in order. If fewer than K or more than the
//                 list holds reach T_lo, the row falls back to the radix select
//                 over the whole row, so the result is exact in every case.
// The output lists min(K, n) positions in ascending order, then -1 padding.
#include "common.cuh"
#include "kernels.h"
#include "topk_core.cuh"

namespace sa {
namespace {

constexpr int TK_THREADS = 512;
constexpr int STAGE_MAX = 16384;             // keys staged in shared memory (64 KB)
constexpr int SAMPLE_MAX = 8192;             // sampled keys (32 KB)
constexpr int CAND_CAP = 8192;               // candidate composites (64 KB)
constexpr int PER_THREAD = 16;               // consecutive positions per thread per pass step
constexpr size_t TK_SMEM = (STAGE_MAX * 4 > SAMPLE_MAX * 4 + CAND_CAP * 8) ? STAGE_MAX * 4
                                                                          : SAMPLE_MAX * 4 + CAND_CAP * 8;

SA_DEVINL int64_t topk_row_len(const TopkArgs& a, int r)
{
    int64_t n = a.row_len ? (int64_t)a.row_len[r] : a.causal_first + r + 1;
    return n < 0 ? 0 : (n > a.n_cap ? a.n_cap : n);
}

// Sample-guided selection of a long row (n > STAGE_MAX). Returns false if the
// sample's bound did not isolate between K and CAND_CAP candidates.
__device__ bool sampled_select(const float* row, int64_t n, int K, int32_t* out, uint32_t* samp,
                               unsigned long long* cand, RadixShared& sh)
{
    const int tid = threadIdx.x;
    // 1. sample: blocks of 8 consecutive keys, one every S positions
    const int64_t nblk_max = SAMPLE_MAX / 8;
    const int64_t S = max64(16, ((n + nblk_max - 1) / nblk_max + 7) / 8 * 8);
    const int nblk = (int)((n + S - 1) / S);
    const int slots = nblk * 8;
    for (int e = tid; e < slots; e += TK_THREADS) {
        const int64_t j = (int64_t)(e >> 3) * S + (e & 7);
        samp[e] = j < n ? score_key(__ldcg(row + j)) : 0u;      // 0 is below every score's key
    }
    const int64_t tail = n - (int64_t)(nblk - 1) * S;
    const int m = (nblk - 1) * 8 + (int)min64(8, tail);          // valid samples
    const double share = (double)K * (double)m / (double)n;
    const double kq_d = ceil(share + 6.0 * sqrt(share) + 16.0);
    if (kq_d >= (double)m) return false;
    __syncthreads();
    uint32_t t_lo, t_mask;
    radix_kth<uint32_t>(samp, (unsigned)slots, (unsigned)kq_d, sh, t_lo, t_mask);

    // 2. one pass over the row: positions with key >= t_lo, in ascending order
    const uint32_t lo = t_lo;
    unsigned written = 0;
    for (int64_t base = 0; base < n; base += (int64_t)TK_THREADS * PER_THREAD) {
        const int64_t j0 = base + (int64_t)tid * PER_THREAD;
        uint32_t keys[PER_THREAD];
        unsigned c = 0;
#pragma unroll
        for (int u = 0; u < PER_THREAD; ++u) {
            const int64_t j = j0 + u;
            keys[u] = j < n ? score_key(__ldg(row + j)) : 0u;
            c += (j < n && keys[u] >= lo) ? 1u : 0u;
        }
        unsigned total;
        const unsigned incl = block_scan_incl(c, sh.warp_tot, &total);
        unsigned pos = written + incl - c;
#pragma unroll
        for (int u = 0; u < PER_THREAD; ++u) {
            const int64_t j = j0 + u;
            if (j < n && keys[u] >= lo) {
                if (pos < (unsigned)CAND_CAP)
                    cand[pos] = ((unsigned long long)keys[u] << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)j);
                ++pos;
            }
        }
        written += total;
    }
    if (written < (unsigned)K || written > (unsigned)CAND_CAP) return false;
    __syncthreads();

    // 3. the K best candidates (composites are distinct), emitted in order
    unsigned long long prefix, mask;
    radix_kth<unsigned long long>(cand, written, (unsigned)K, sh, prefix, mask);
    unsigned emitted = 0;
    for (unsigned i0 = 0; i0 < written; i0 += TK_THREADS) {
        const unsigned i = i0 + tid;
        const bool keep = i < written && (cand[i] & mask) >= prefix;
        unsigned total;
        const unsigned incl = block_scan_incl(keep ? 1u : 0u, sh.warp_tot, &total);
        if (keep && emitted + incl - 1 < (unsigned)K)
            out[emitted + incl - 1] = (int32_t)(0xFFFFFFFFu - (uint32_t)cand[i]);
        emitted += total;
    }
    return true;
}

__global__ void __launch_bounds__(TK_THREADS, 2)
topk_rows_kernel(TopkArgs a)
{
    __shared__ RadixShared sh;
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
        radix_select_row([&](int64_t j) { return keys[j]; }, n, K, out, sh);
        return;
    }
    uint32_t* samp = reinterpret_cast<uint32_t*>(tk_smem);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(tk_smem + SAMPLE_MAX * 4);
    if (!sampled_select(row, n, K, out, samp, cand, sh)) {
        __syncthreads();
        radix_select_row([&](int64_t j) { return score_key(__ldcg(row + j)); }, n, K, out, sh);
    }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
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
