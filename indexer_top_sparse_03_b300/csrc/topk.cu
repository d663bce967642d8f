// Exact per-row Top-K by radix select ("Hybrid Attention Architectures...",
// section 3.1, filtering stage: keep the K highest-scoring positions).
//
// One CTA per row. Scores are mapped to order-preserving 32-bit keys; an
// MSB-first radix select with 8-bit digits (shared-memory histograms, warp
// match-aggregated atomics, a one-warp suffix scan to find the threshold
// digit) narrows down the key of the K-th best score. A single ordered pass
// then emits, in ascending position order, every position whose key is above
// the threshold plus the lowest-position ones that equal it: this is the
// "ties go to the lower position" rule, and it makes the output deterministic.
// Rows short enough are staged once in shared memory; longer rows are re-read
// from global memory (L2) on every pass. No sort is ever materialised.
#include "common.cuh"
#include "kernels.h"

namespace sa {
namespace {

constexpr int TK_THREADS = 1024;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int RADIX = 256;
constexpr int SMEM_KEYS = 12288;     // 48 KB of keys staged per row

struct TopkShared {
    unsigned hist[RADIX];
    unsigned warp_tot[TK_WARPS];
    int digit, above, cnt;
};

SA_DEVINL int64_t topk_row_len(const TopkArgs& a, int r)
{
    int64_t n = a.row_len ? (int64_t)a.row_len[r] : a.causal_first + r + 1;
    return n < 0 ? 0 : (n > a.n_cap ? a.n_cap : n);
}

// Finds the digit d* with  count(digit > d*) < need <= count(digit >= d*).
// Called by warp 0 only; results land in sh.digit / sh.above / sh.cnt.
SA_DEVINL void find_digit(TopkShared& sh, unsigned need)
{
    const int lane = threadIdx.x & 31;
    // lane l owns digits 255-8l .. 248-8l (descending)
    unsigned own = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) own += sh.hist[255 - 8 * lane - i];
    unsigned incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const unsigned excl = incl - own;
    if (excl < need && need <= incl) {
        unsigned run = excl;
        for (int i = 0; i < 8; ++i) {
            const int d = 255 - 8 * lane - i;
            const unsigned c = sh.hist[d];
            if (run + c >= need) {
                sh.digit = d; sh.above = (int)run; sh.cnt = (int)c;
                break;
            }
            run += c;
        }
    }
}

template <bool STAGED>
__global__ void __launch_bounds__(TK_THREADS)
topk_rows_kernel(TopkArgs a)
{
    __shared__ TopkShared sh;
    extern __shared__ uint32_t keys[];      // [SMEM_KEYS] when STAGED
    const int r = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n = topk_row_len(a, r);
    const int K = a.K;
    int32_t* out = a.idx + (int64_t)r * a.ld_idx;
    const float* row = a.scores + (int64_t)r * a.ld_s;

    if (n <= K) {                            // keep everything, in order
        for (int i = tid; i < K; i += TK_THREADS) out[i] = i < n ? i : -1;
        return;
    }
    if (STAGED) {
        for (int64_t j = tid; j < n; j += TK_THREADS) keys[j] = score_key(row[j]);
        __syncthreads();
    }
    auto key_at = [&](int64_t j) -> uint32_t {
        return STAGED ? keys[j] : score_key(__ldcg(row + j));
    };

    uint32_t prefix = 0, mask = 0;
    unsigned need = (unsigned)K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < RADIX; i += TK_THREADS) sh.hist[i] = 0;
        __syncthreads();
        for (int64_t j0 = 0; j0 < n; j0 += TK_THREADS) {
            const int64_t j = j0 + tid;
            int bin = RADIX;                         // "no bin"
            if (j < n) {
                const uint32_t u = key_at(j);
                if ((u & mask) == prefix) bin = (u >> shift) & (RADIX - 1);
            }
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (bin < RADIX && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bin], __popc(peers));
        }
        __syncthreads();
        if (warp == 0) find_digit(sh, need);
        __syncthreads();
        prefix |= (uint32_t)sh.digit << shift;
        mask |= (uint32_t)(RADIX - 1) << shift;
        need -= (unsigned)sh.above;
        const bool done = need == (unsigned)sh.cnt;   // the whole bucket is kept
        __syncthreads();
        if (done) break;
    }

    // ordered emission: keys above the threshold, plus the first `need`
    // (lowest positions) of those equal to it
    const uint32_t lanemask_lt = (1u << lane) - 1u;
    unsigned written = 0, eq_before = 0;
    for (int64_t j0 = 0; j0 < n; j0 += TK_THREADS) {
        const int64_t j = j0 + tid;
        bool gt = false, eq = false;
        if (j < n) {
            const uint32_t u = key_at(j) & mask;
            gt = u > prefix;
            eq = u == prefix;
        }
        const unsigned bgt = __ballot_sync(0xffffffffu, gt);
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) sh.warp_tot[warp] = __popc(bgt) | (__popc(beq) << 16);
        __syncthreads();
        unsigned wpre = 0, tot = 0;
        for (int w = 0; w < TK_WARPS; ++w) {
            const unsigned v = sh.warp_tot[w];
            wpre += (w < warp) ? v : 0u;
            tot += v;
        }
        const unsigned gt_ex = (wpre & 0xffff) + __popc(bgt & lanemask_lt);
        const unsigned eq_ex = (wpre >> 16) + __popc(beq & lanemask_lt);
        const unsigned eq_quota = need > eq_before ? need - eq_before : 0u;
        if (gt || (eq && eq_ex < eq_quota)) {
            const unsigned pos = written + gt_ex + min(eq_ex, eq_quota);
            if (pos < (unsigned)K) out[pos] = (int32_t)j;
        }
        written += (tot & 0xffff) + min(tot >> 16, eq_quota);
        eq_before += tot >> 16;
        __syncthreads();
    }
    for (int i = (int)written + tid; i < K; i += TK_THREADS) out[i] = -1;
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
    if (a.n_cap <= SMEM_KEYS) {
        const size_t smem = sizeof(uint32_t) * (size_t)SMEM_KEYS;
        cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        topk_rows_kernel<true><<<a.rows, TK_THREADS, smem, s>>>(a);
    } else {
        topk_rows_kernel<false><<<a.rows, TK_THREADS, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace sa
