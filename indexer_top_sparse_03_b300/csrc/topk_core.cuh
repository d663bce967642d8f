// Device pieces of the exact Top-K ("Hybrid Attention Architectures...",
// section 3.1, filtering stage: keep the K highest-scoring positions; an
// exact tie goes to the lower position).
//
// Scores are compared through order-preserving 32-bit keys (score_key). Two
// selection schemes share these pieces:
//   - a block-wide MSB-first radix select over one row (8-bit digits), used
//     for short rows staged in shared memory and as the general fallback;
//   - a threshold-bin scheme for long rows: a 4096-bin histogram of the key's
//     top 12 bits gives the bin holding the K-th best score, every position in
//     a higher bin is kept, and only the positions inside that bin are ranked
//     exactly (by key, then by lower position).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace sa {

constexpr int RADIX = 256;
constexpr int HBITS = 12;                       // bits of the threshold-bin histogram
constexpr int HBINS = 1 << HBITS;
constexpr int HSHIFT = 32 - HBITS;

SA_DEVINL uint32_t key_bin(uint32_t key) { return key >> HSHIFT; }

// Inclusive prefix sum over the threads of the block (any multiple of 32 up
// to 1024 threads); `warp_tot` is 32 words of shared scratch. Contains two
// __syncthreads.
SA_DEVINL unsigned block_scan_incl(unsigned v, unsigned* warp_tot, unsigned* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    unsigned before = 0, all = 0;
    for (int w = 0; w < nw; ++w) {
        const unsigned t = warp_tot[w];
        before += (w < warp) ? t : 0u;
        all += t;
    }
    __syncthreads();
    if (total) *total = all;
    return v + before;
}

// Copies a 4096-bin histogram from global memory into shared memory with
// 16-byte loads (whole block; ends with __syncthreads).
SA_DEVINL void stage_hist(unsigned* dst, const unsigned* src)
{
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = threadIdx.x; i < HBINS / 4; i += blockDim.x) d4[i] = __ldcg(s4 + i);
    __syncthreads();
}

// The bin holding the K-th largest key of a 4096-bin shared-memory histogram
// with at least K entries (bins counted from the top). `out` is shared
// scratch that receives the answer. Whole block.
SA_DEVINL BinSplit find_bin(const unsigned* hist, unsigned K, unsigned* warp_tot, BinSplit* out)
{
    if (threadIdx.x == 0) { out->bin = 0; out->above = 0; out->in_bin = 0; }
    const int per = HBINS / blockDim.x;            // bins per thread (4 .. 16)
    const int top = HBINS - 1 - threadIdx.x * per; // this thread's bins: top, top-1, ...
    unsigned own = 0;
    for (int i = 0; i < per; ++i) own += hist[top - i];
    const unsigned incl = block_scan_incl(own, warp_tot, nullptr);
    const unsigned excl = incl - own;
    if (excl < K && K <= incl) {
        unsigned run = excl;
        for (int i = 0; i < per; ++i) {
            const unsigned c = hist[top - i];
            if (run + c >= K) {
                out->bin = top - i; out->above = run; out->in_bin = c;
                break;
            }
            run += c;
        }
    }
    __syncthreads();
    const BinSplit r = *out;
    __syncthreads();
    return r;
}

// ---------------------------------------------------------------------------
// block-wide radix select over one row (8-bit digits, MSB first) + ordered
// emission of the kept positions into out[0 .. K-1]
// ---------------------------------------------------------------------------
struct RadixShared {
    unsigned hist[RADIX];
    unsigned warp_tot[32];
    int digit, above, cnt;
};

// Finds d* with count(digit > d*) < need <= count(digit >= d*). Warp 0 only.
SA_DEVINL void radix_find_digit(RadixShared& sh, unsigned need)
{
    const int lane = threadIdx.x & 31;
    unsigned own = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) own += sh.hist[255 - 8 * lane - i];
    unsigned incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
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

// MSB-first radix search over cnt values v[0..cnt) in shared memory (8-bit
// digits): on return, the values v with (v & mask) >= prefix number at least
// `need`, and exactly `need` when the values are distinct. Whole block.
// `start_shift` is the lowest bit of the first digit examined, a multiple of
// 8 (the digits then end exactly at bit 0): callers that know the values share
// their top bits start below them (and must then merge those bits into prefix
// and mask themselves).
template <typename T>
__device__ void radix_kth(const T* v, unsigned cnt, unsigned need, RadixShared& sh, T& prefix_out, T& mask_out,
                          int start_shift = (int)sizeof(T) * 8 - 8)
{
    const int tid = threadIdx.x, nth = blockDim.x;
    T prefix = 0, mask = 0;
    start_shift = (start_shift + 7) & ~7;    // whole digits down to bit 0
    for (int shift = start_shift; shift >= 0; shift -= 8) {
        for (int i = tid; i < RADIX; i += nth) sh.hist[i] = 0;
        __syncthreads();
        for (unsigned i = tid; i < cnt; i += nth) {
            const T x = v[i];
            if ((x & mask) == prefix) atomicAdd(&sh.hist[(unsigned)(x >> shift) & (RADIX - 1)], 1u);
        }
        __syncthreads();
        if (tid < 32) radix_find_digit(sh, need);
        __syncthreads();
        prefix |= (T)sh.digit << shift;
        mask |= (T)(RADIX - 1) << shift;
        need -= (unsigned)sh.above;
        const bool done = need == (unsigned)sh.cnt;     // the whole bucket is kept
        __syncthreads();
        if (done) break;
    }
    prefix_out = prefix;
    mask_out = mask;
}

// ---------------------------------------------------------------------------
// exact boundary inside a candidate list
// ---------------------------------------------------------------------------
// Candidates are composites c = (key << 32) | ~position (distinct, and the
// larger composite is the better one: higher key, then lower position), all
// with key >= lo. Relative to lo, rel(c) = c - (lo << 32); the 4096 bins are
// equal slices of [lo, kmax], 2^bsh keys wide. A candidate is kept iff its
// bin is above the boundary bin, or it is in that bin with
// (rel & mask) >= prefix.
struct CandBoundary {
    uint32_t lo;
    int bsh;
    unsigned bin;
    unsigned long long prefix, mask;
};
SA_DEVINL unsigned long long cand_rel(unsigned long long c, uint32_t lo)
{
    return c - ((unsigned long long)lo << 32);
}
SA_DEVINL uint32_t cand_bin(unsigned long long c, const CandBoundary& b)
{
    return (uint32_t)(cand_rel(c, b.lo) >> (32 + b.bsh));
}
SA_DEVINL bool cand_keep(unsigned long long c, const CandBoundary& b)
{
    const uint32_t bin = cand_bin(c, b);
    return bin > b.bin || (bin == b.bin && (cand_rel(c, b.lo) & b.mask) >= b.prefix);
}

// Finds the boundary that keeps exactly K of the cnt >= K candidates cand[]
// (shared or global memory). hist is 4096 words of shared scratch, bcand
// room for bin_cap composites. Returns false (nothing decided) when the
// boundary bin holds more than bin_cap candidates. Whole block.
SA_DEVINL bool cand_boundary(const unsigned long long* cand, unsigned cnt, uint32_t lo, uint32_t kmax,
                             unsigned K, unsigned* hist, unsigned long long* bcand, unsigned bin_cap,
                             RadixShared& sh, BinSplit* split, CandBoundary& out)
{
    const int tid = threadIdx.x, nth = blockDim.x;
    CandBoundary b;
    b.lo = lo;
    b.bsh = max(0, 32 - __clz((int)((kmax - lo) | 1u)) - HBITS);
    for (int i = tid; i < HBINS; i += nth) hist[i] = 0;
    __syncthreads();
    for (unsigned i = tid; i < cnt; i += nth) atomicAdd(&hist[cand_bin(cand[i], b)], 1u);
    __syncthreads();
    const BinSplit cb = find_bin(hist, K, sh.warp_tot, split);
    if (cb.in_bin > bin_cap) return false;
    b.bin = (unsigned)cb.bin;
    // gather the boundary bin (any order: the search is order-free)
    if (tid == 0) sh.cnt = 0;
    __syncthreads();
    for (unsigned i = tid; i < cnt; i += nth) {
        const unsigned long long c = cand[i];
        if (cand_bin(c, b) == b.bin) bcand[atomicAdd(&sh.cnt, 1)] = cand_rel(c, lo);
    }
    __syncthreads();
    // one bin's rel values agree above bit 32 + bsh: search from the digit
    // holding bit 31 + bsh down (digits are 8 bits, ending at bit 0)
    radix_kth<unsigned long long>(bcand, cb.in_bin, K - cb.above, sh, b.prefix, b.mask, (31 + b.bsh) / 8 * 8);
    out = b;
    return true;
}

// Block-wide maximum of one value per thread (shared scratch: 32 words).
SA_DEVINL uint32_t block_max_u32(uint32_t v, unsigned* warp_tot)
{
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) warp_tot[warp] = v;
    __syncthreads();
    uint32_t m = 0;
    for (int w = 0; w < nw; ++w) m = max(m, (uint32_t)warp_tot[w]);
    __syncthreads();
    return m;
}

// Keeps the K best of the n keys given by key_at(j) (n > K) and writes their
// positions in ascending order to out[0 .. K-1]. Whole block, blockDim.x a
// multiple of 32.
// With HIST0 the caller has already counted the top digits (key >> 24) of
// all n keys into sh.hist (and synchronised), so the first pass is skipped.
// `staged`, when given, holds the same n keys in 16-byte-aligned shared
// memory: the counting passes (which do not depend on the order of the keys)
// then read four keys per load.
template <bool HIST0 = false, typename KeyAt>
__device__ void radix_select_row(KeyAt key_at, int64_t n, int K, int32_t* out, RadixShared& sh,
                                 const uint32_t* staged = nullptr)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nth = blockDim.x;
    uint32_t prefix = 0, mask = 0;
    unsigned need = (unsigned)K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (!HIST0 || shift != 24) {
            for (int i = tid; i < RADIX; i += nth) sh.hist[i] = 0;
            __syncthreads();
            auto count = [&](uint32_t u) {
                if ((u & mask) == prefix) atomicAdd(&sh.hist[(u >> shift) & (RADIX - 1)], 1u);
            };
            int64_t j_tail = 0;
            if (staged) {                    // 16-byte-aligned keys in shared memory: four per load
                const int64_t n4 = n >> 2;
                const uint4* s4 = reinterpret_cast<const uint4*>(staged);
                for (int64_t i = tid; i < n4; i += nth) {
                    const uint4 u = s4[i];
                    count(u.x); count(u.y); count(u.z); count(u.w);
                }
                j_tail = n4 << 2;
            }
            for (int64_t j = j_tail + tid; j < n; j += nth) count(key_at(j));
            __syncthreads();
        }
        if (warp == 0) radix_find_digit(sh, need);
        __syncthreads();
        prefix |= (uint32_t)sh.digit << shift;
        mask |= (uint32_t)(RADIX - 1) << shift;
        need -= (unsigned)sh.above;
        const bool done = need == (unsigned)sh.cnt;   // the whole bucket is kept
        __syncthreads();
        if (done) break;
    }

    // ordered emission: keys above the threshold, plus the first `need`
    // (lowest positions) of those equal to it. Each warp takes 32 x EMIT_STEPS
    // consecutive positions per round (32 per step, one ballot pair per step),
    // so a round of the block covers nth x EMIT_STEPS positions with one
    // exchange of warp totals.
    constexpr int EMIT_STEPS = 8;
    const uint32_t lanemask_lt = (1u << lane) - 1u;
    const int nw = nth >> 5;
    unsigned written = 0, eq_before = 0;
    for (int64_t j0 = 0; j0 < n; j0 += (int64_t)nth * EMIT_STEPS) {
        const int64_t wb = j0 + (int64_t)warp * 32 * EMIT_STEPS;
        unsigned bgt[EMIT_STEPS], beq[EMIT_STEPS];
        unsigned cgt = 0, ceq = 0;
#pragma unroll
        for (int i = 0; i < EMIT_STEPS; ++i) {
            const int64_t j = wb + i * 32 + lane;
            bool gt = false, eq = false;
            if (j < n) {
                const uint32_t u = key_at(j) & mask;
                gt = u > prefix;
                eq = u == prefix;
            }
            bgt[i] = __ballot_sync(0xffffffffu, gt);
            beq[i] = __ballot_sync(0xffffffffu, eq);
            cgt += __popc(bgt[i]);
            ceq += __popc(beq[i]);
        }
        if (lane == 0) sh.warp_tot[warp] = cgt | (ceq << 16);
        __syncthreads();
        unsigned wpre = 0, tot = 0;
        for (int w = 0; w < nw; ++w) {
            const unsigned v = sh.warp_tot[w];
            wpre += (w < warp) ? v : 0u;
            tot += v;
        }
        const unsigned eq_quota = need > eq_before ? need - eq_before : 0u;
        unsigned gt_run = wpre & 0xffff, eq_run = wpre >> 16;
#pragma unroll
        for (int i = 0; i < EMIT_STEPS; ++i) {
            const unsigned gt_ex = gt_run + __popc(bgt[i] & lanemask_lt);
            const unsigned eq_ex = eq_run + __popc(beq[i] & lanemask_lt);
            const bool gt = (bgt[i] >> lane) & 1u, eq = (beq[i] >> lane) & 1u;
            if (gt || (eq && eq_ex < eq_quota)) {
                const unsigned pos = written + gt_ex + min(eq_ex, eq_quota);
                if (pos < (unsigned)K) out[pos] = (int32_t)(wb + i * 32 + lane);
            }
            gt_run += __popc(bgt[i]);
            eq_run += __popc(beq[i]);
        }
        written += (tot & 0xffff) + min(tot >> 16, eq_quota);
        eq_before += tot >> 16;
        __syncthreads();
    }
}

}  // namespace sa
