// Decode Top-K: the K best positions of each sequence's score row
// ("Hybrid Attention Architectures...", section 3.1, filtering stage; an
// exact tie goes to the lower position), for rows far longer than K.
//
// The scan has already counted, per sequence, the top 12 bits of every
// score's order-preserving key into a 4096-bin histogram, and its last CTA
// has found the bin b* that holds the K-th best score. Every position in a
// higher bin
// is kept, and only the positions inside b* (a few hundred to a few thousand
// for continuous scores) need an exact ranking. Two launches:
//
//   1. bitmap pass, grid (slices, B): each thread reads 32 consecutive scores
//      of one row (L2-resident: the scan wrote them just before), writes one
//      bitmap word (bit set: the position's bin is above b*), and
//      appends the positions of bin b* to a per-row candidate list as 64-bit
//      composites (key << 32 | ~position: a larger composite means a better
//      score, then a lower position).
//   2. finish pass, one CTA per row: stages the row's bitmap and candidates in
//      shared memory, radix-selects the K - above best composites among the
//      candidates, sets their bits, then emits the kept positions in
//      ascending order by a prefix count over the bitmap words.
// A row whose candidates overflow the list (huge runs of equal scores) is
// instead selected by the block-wide radix select over the whole row. Rows
// with n <= K keep every position.
#include "common.cuh"
#include "kernels.h"
#include "topk_core.cuh"

namespace sa {
namespace {

constexpr int BM_THREADS = 256;
constexpr int BM_SLICE = 32 * BM_THREADS;    // positions per bitmap CTA: one bitmap word per thread
constexpr int FIN_THREADS = 512;
constexpr int FIN_WORDS = 16384;             // shared-memory bitmap: rows up to 524288 positions

SA_DEVINL int64_t row_len(const DecodeSelectArgs& a, int b)
{
    int64_t n = a.ctx_len[b];
    return n < 0 ? 0 : (n > a.max_ctx ? a.max_ctx : n);
}

// four CTAs per SM (at most 64 registers): the 512 CTAs of a 32 x 131072
// batch then run in one wave instead of two
__global__ void __launch_bounds__(BM_THREADS, 4)
decode_bitmap_kernel(DecodeSelectArgs a)
{
    griddep_wait();                          // scores, bins and counters of the scan
    griddep_launch();
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int64_t n = row_len(a, b);
    const int64_t w = (int64_t)blockIdx.x * BM_THREADS + threadIdx.x;   // this thread's bitmap word
    const int64_t j0 = w << 5;
    if (n <= a.K || j0 >= n) return;

    const float* row = a.scores + (int64_t)b * a.ld_s;
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldcg(reinterpret_cast<const float4*>(row + j0) + i);
    const BinSplit bs = a.split[b];
    const bool take_bin = bs.above + bs.in_bin == (unsigned)a.K;     // the whole bin is kept
    const uint32_t bstar = (uint32_t)bs.bin;

    uint32_t keep = 0, maybe = 0, keys[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float x = (&v[i >> 2].x)[i & 3];
        keys[i] = score_key(x);
        const uint32_t bin = key_bin(keys[i]);
        const bool valid = j0 + i < n;
        if (valid && (bin > bstar || (take_bin && bin == bstar))) keep |= 1u << i;
        if (valid && !take_bin && bin == bstar) maybe |= 1u << i;
    }
    a.bitmap[(int64_t)b * a.ld_w + w] = keep;

    // candidates of bin b*: warp-aggregated slot reservation. Threads past
    // the row's end have returned; they are the warp's highest lanes.
    const unsigned am = __activemask();
    const int last = 31 - __clz(am);
    const unsigned c = __popc(maybe);
    unsigned incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned u = __shfl_up_sync(am, incl, o);
        if (lane >= o) incl += u;
    }
    const unsigned wtot = __shfl_sync(am, incl, last);
    if (wtot == 0) return;
    unsigned base = 0;
    if (lane == 0) base = atomicAdd(a.cand_cnt + b, wtot);
    base = __shfl_sync(am, base, 0);
    unsigned pos = base + incl - c;
    unsigned long long* cand = a.cand + (int64_t)b * a.cand_cap;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if ((maybe >> i) & 1u) {
            if (pos < (unsigned)a.cand_cap)
                cand[pos] = ((unsigned long long)keys[i] << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)(j0 + i));
            ++pos;
        }
    }
}

__global__ void __launch_bounds__(FIN_THREADS)
decode_finish_kernel(DecodeSelectArgs a)
{
    extern __shared__ __align__(16) unsigned long long fin_smem[];
    unsigned long long* cs = fin_smem;                                       // [cand_cap]
    uint32_t* bits = reinterpret_cast<uint32_t*>(fin_smem + a.cand_cap);     // [FIN_WORDS]
    __shared__ RadixShared sh;
    griddep_wait();                          // bitmaps and candidates
    griddep_launch();
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t n = row_len(a, b);
    const int K = a.K;
    int32_t* out = a.idx + (int64_t)b * K;
    if (n <= K) {
        for (int i = tid; i < K; i += FIN_THREADS) out[i] = i < n ? i : -1;
        return;
    }
    const float* row = a.scores + (int64_t)b * a.ld_s;
    const BinSplit bs = a.split[b];
    const bool take_bin = bs.above + bs.in_bin == (unsigned)K;
    const unsigned cnt = take_bin ? 0u : __ldcg(a.cand_cnt + b);
    const int64_t words = (n + 31) >> 5;
    if (words > FIN_WORDS || cnt > (unsigned)a.cand_cap || (!take_bin && cnt != bs.in_bin)) {
        // too long for the shared-memory bitmap, or too many candidates for
        // the list: exact radix select over the row
        radix_select_row([&](int64_t j) { return score_key(__ldcg(row + j)); }, n, K, out, sh);
        return;
    }
    // the kept-position bits of the higher bins, and the candidates of bin b*
    const uint4* gb = reinterpret_cast<const uint4*>(a.bitmap + (int64_t)b * a.ld_w);
    for (int64_t i = tid; i < (words + 3) / 4; i += FIN_THREADS) reinterpret_cast<uint4*>(bits)[i] = __ldcg(gb + i);
    const unsigned long long* cg = a.cand + (int64_t)b * a.cand_cap;
    for (unsigned i = tid; i < cnt; i += FIN_THREADS) cs[i] = __ldcg(cg + i);
    __syncthreads();
    if (!take_bin) {
        // the (K - above)-th largest composite (all distinct); the top 12 bits
        // of every candidate's key are the bin itself, so the search starts
        // at the digit of bits 48..55 (its top half is still the bin, equal
        // for every candidate) and its 8-bit digits end exactly at bit 0: the
        // low bits of the position decide ties of equal keys
        unsigned long long prefix, mask;
        radix_kth<unsigned long long>(cs, cnt, (unsigned)K - bs.above, sh, prefix, mask, 48);
        prefix |= (unsigned long long)bs.bin << (64 - HBITS);
        mask |= ~0ull << (64 - HBITS);
        for (unsigned i = tid; i < cnt; i += FIN_THREADS) {
            const unsigned long long c = cs[i];
            if ((c & mask) >= prefix) {
                const uint32_t j = 0xFFFFFFFFu - (uint32_t)c;
                atomicOr(bits + (j >> 5), 1u << (j & 31));
            }
        }
        __syncthreads();
    }

    // ordered emission: thread t owns a contiguous run of bitmap words
    const int64_t per = (words + FIN_THREADS - 1) / FIN_THREADS;
    const int64_t w_lo = min64(words, (int64_t)tid * per), w_hi = min64(words, w_lo + per);
    unsigned c = 0;
    for (int64_t w = w_lo; w < w_hi; ++w) c += __popc(bits[w]);
    unsigned total;
    const unsigned incl = block_scan_incl(c, sh.warp_tot, &total);
    unsigned pos = incl - c;
    for (int64_t w = w_lo; w < w_hi; ++w) {
        uint32_t word = bits[w];
        while (word) {
            const int bit = __ffs(word) - 1;
            if (pos < (unsigned)K) out[pos] = (int32_t)((w << 5) + bit);
            ++pos;
            word &= word - 1;
        }
    }
    for (int i = (int)total + tid; i < K; i += FIN_THREADS) out[i] = -1;
}

}  // namespace

cudaError_t launch_decode_select(const DecodeSelectArgs& a, cudaStream_t s)
{
    if (a.B <= 0) return cudaSuccess;
    if (a.max_ctx > a.K) {
        dim3 grid((unsigned)((a.max_ctx + BM_SLICE - 1) / BM_SLICE), a.B);
        cudaError_t e = launch_kernel(decode_bitmap_kernel, grid, dim3(BM_THREADS), 0, s, true, a);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(unsigned long long) * (size_t)a.cand_cap + sizeof(uint32_t) * FIN_WORDS;
    cudaError_t e = cudaFuncSetAttribute(decode_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
    }
    return launch_kernel(decode_finish_kernel, dim3(a.B), dim3(FIN_THREADS), smem, s, true, a);
}

}  // namespace sa
