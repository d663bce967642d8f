// Indexer fused with Top-K for long causal rows ("Hybrid Attention
// Architectures...", section 3.1: the indexing stage scores every history
// position, the filtering stage keeps the K best; an exact tie goes to the
// lower position). Here the score rows never reach memory:
//
//   1. sample: one key per stratum of 16 consecutive positions (stratified,
//      pseudo-random offset inside each stratum) is gathered into a compact
//      key matrix, and the tensor-core indexer scores every query of the pass
//      against the sampled keys of its history (about n/16 of them);
//   2. threshold: per query row, the k'-th best sampled key, k' being the
//      sample's share of K plus a six-sigma margin, is a lower bound that at
//      least K of the row's n keys reach almost surely, while only a few
//      thousand do;
//   3. filter: the tensor-core indexer scores the full history and keeps, per
//      work item, the (key, position) pairs at or above the row's threshold
//      (indexer_tc.cu, filter mode);
//   4. select (this file): per row, the kept pairs of all its work items are
//      gathered into shared memory, the exact K-th best is found among them
//      (slices of [threshold, max key], then a radix search inside the
//      boundary slice) and the kept positions are emitted in ascending order
//      through a shared-memory bitmap;
//   5. fallback: a row whose threshold kept fewer than K pairs, or more than
//      the lists hold, is scored again on CUDA cores into a scratch row and
//      selected by the block-wide radix select, so every row is exact.
#include "common.cuh"
#include "kernels.h"
#include "topk_core.cuh"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int TH_THREADS = 256;
constexpr int FS_THREADS = 512;
constexpr int FS_BIN_CAP = 1024;
constexpr int FB_THREADS = 512;

// ---------------------------------------------------------------------------
// 1. the stratified key sample
// ---------------------------------------------------------------------------
__global__ void sample_gather_kernel(const uint4* k_idx, int chunks, const float* k_scale, int64_t ns, int lg,
                                     uint4* ksamp, float* ksamp_scale)
{
    const int64_t total = ns * chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / chunks;
        const int c = (int)(i - row * chunks);
        const int64_t p = sample_pos(row, lg);
        ksamp[i] = __ldg(k_idx + p * chunks + c);
        if (c == 0 && k_scale) ksamp_scale[row] = k_scale[p];
    }
}

// ---------------------------------------------------------------------------
// 2. per-row threshold from the sampled scores
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(TH_THREADS)
sample_threshold_kernel(FusedSelectArgs a, const float* ssc, int64_t ld_ssc)
{
    extern __shared__ __align__(16) uint32_t th_keys[];
    __shared__ RadixShared sh;
    const int r = blockIdx.x;
    const int64_t t = a.t_begin + r;
    const int64_t n = t + 1 < a.N ? t + 1 : a.N;
    const int64_t c = sample_count(t, a.sample_log2) < a.ns ? sample_count(t, a.sample_log2) : a.ns;
    const double share = (double)a.K * (double)c / (double)n;
    const double kq = ceil(share + 6.0 * sqrt(share) + 16.0);
    if (kq >= (double)c) {                   // too few samples: keep everything (the row falls back)
        if (threadIdx.x == 0) a.thr[r] = 0u;
        return;
    }
    const float* row = ssc + (int64_t)r * ld_ssc;
    for (int64_t i = threadIdx.x; i < c; i += TH_THREADS) th_keys[i] = score_key(__ldcg(row + i));
    __syncthreads();
    uint32_t prefix, mask;
    // an early stop leaves the low digits zero: a lower bound, still valid
    radix_kth<uint32_t>(th_keys, (unsigned)c, (unsigned)kq, sh, prefix, mask);
    if (threadIdx.x == 0) a.thr[r] = prefix;
}

// ---------------------------------------------------------------------------
// 4. exact selection among the kept pairs
// ---------------------------------------------------------------------------
SA_DEVINL int row_segments(const FusedSelectArgs& a, int r)
{
    const int qi = r / a.tq;
    const int64_t t_last = min64(a.t_begin + (int64_t)(qi + 1) * a.tq, a.t_begin + a.rows) - 1;
    const int64_t n_last = min64(a.N, t_last + 1);
    const int64_t tiles = (n_last + 127) / 128;
    return (int)((tiles + a.group - 1) / a.group);
}

__global__ void __launch_bounds__(FS_THREADS)
fused_select_kernel(FusedSelectArgs a)
{
    extern __shared__ __align__(16) unsigned long long fs_smem[];
    unsigned long long* cand = fs_smem;                                          // [cand_cap]
    unsigned long long* bcand = cand + a.cand_cap;                               // [FS_BIN_CAP]
    unsigned* hist = reinterpret_cast<unsigned*>(bcand + FS_BIN_CAP);            // [HBINS]
    uint32_t* bits = hist + HBINS;                                               // [words]
    unsigned* offs = bits + a.words;                                             // [nseg + 1]
    __shared__ RadixShared sh;
    __shared__ BinSplit split;
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t t = a.t_begin + r;
    const int64_t n = t + 1 < a.N ? t + 1 : a.N;
    const int K = a.K;
    int32_t* out = a.idx + (int64_t)r * a.ld_idx;
    const int nseg = row_segments(a, r);
    const unsigned* cnt = a.seg_cnt + (int64_t)r * a.nseg;

    // segment counts -> offsets (one segment per thread and round)
    bool bad = false;
    unsigned base = 0;
    for (int g0 = 0; g0 < nseg; g0 += FS_THREADS) {
        const int g = g0 + tid;
        const unsigned c = g < nseg ? __ldcg(cnt + g) : 0u;
        bad = bad || c > (unsigned)a.cap_seg;        // the segment lost pairs
        unsigned total;
        const unsigned incl = block_scan_incl(c, sh.warp_tot, &total);
        if (g < nseg) offs[g] = base + incl - c;
        base += total;
    }
    bad = __syncthreads_or(bad) != 0;
    const unsigned total = base;
    if (bad || total < (unsigned)K || total > (unsigned)a.cand_cap || n <= K) {
        if (tid == 0) a.fail_list[atomicAdd(a.fail_cnt, 1u)] = r;
        return;
    }
    // gather the pairs (one warp per segment); the filter pass stores the
    // score's bits, made the order-preserving key here
    const int warp = tid >> 5, lane = tid & 31;
    for (int g = warp; g < nseg; g += FS_THREADS / 32) {
        const unsigned c = __ldcg(cnt + g);
        const unsigned long long* src = a.seg_cand + ((int64_t)r * a.nseg + g) * a.cap_seg;
        for (unsigned k = lane; k < c; k += 32) {
            const unsigned long long v = __ldcg(src + k);
            cand[offs[g] + k] = ((unsigned long long)score_key(__uint_as_float((uint32_t)(v >> 32))) << 32) |
                                (v & 0xFFFFFFFFull);
        }
    }
    uint32_t kmax = 0;
    __syncthreads();
    for (unsigned i = tid; i < total; i += FS_THREADS) kmax = max(kmax, (uint32_t)(cand[i] >> 32));
    kmax = block_max_u32(kmax, sh.warp_tot);
    const uint32_t lo = a.thr[r];
    CandBoundary cb;
    if (!cand_boundary(cand, total, lo, kmax, (unsigned)K, hist, bcand, FS_BIN_CAP, sh, &split, cb)) {
        if (tid == 0) a.fail_list[atomicAdd(a.fail_cnt, 1u)] = r;
        return;
    }
    // kept positions into the bitmap, then ascending emission
    const int64_t words = (n + 31) >> 5;
    for (int64_t i = tid; i < words; i += FS_THREADS) bits[i] = 0u;
    __syncthreads();
    for (unsigned i = tid; i < total; i += FS_THREADS) {
        const unsigned long long c = cand[i];
        if (cand_keep(c, cb)) {
            const uint32_t j = 0xFFFFFFFFu - (uint32_t)c;
            atomicOr(bits + (j >> 5), 1u << (j & 31));
        }
    }
    __syncthreads();
    const int64_t per = (words + FS_THREADS - 1) / FS_THREADS;
    const int64_t w_lo = min64(words, (int64_t)tid * per), w_hi = min64(words, w_lo + per);
    unsigned c = 0;
    for (int64_t w = w_lo; w < w_hi; ++w) c += __popc(bits[w]);
    unsigned kept;
    const unsigned incl = block_scan_incl(c, sh.warp_tot, &kept);
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
}

// ---------------------------------------------------------------------------
// 5. fallback rows: CUDA-core scores into a scratch row, then radix select
// ---------------------------------------------------------------------------
SA_DEVINL float key_elem(const IndexerArgs& ia, int64_t j, int d)
{
    const int64_t e = j * ia.di + d;
    if (ia.dtype == SA_BF16) return to_f32(static_cast<const bf16*>(ia.k_idx)[e]);
    if (ia.dtype == SA_FP8_E4M3) return e4m3_to_f32(static_cast<const uint8_t*>(ia.k_idx)[e]);
    return static_cast<const float*>(ia.k_idx)[e];
}

__global__ void __launch_bounds__(FB_THREADS)
fused_fallback_kernel(FusedSelectArgs a)
{
    extern __shared__ __align__(16) float fb_q[];                    // [Hi][di] then [Hi] weights
    __shared__ RadixShared sh;
    const IndexerArgs& ia = a.ia;
    const unsigned nfail = *reinterpret_cast<volatile unsigned*>(a.fail_cnt);
    const int Hi = ia.Hi, di = ia.di;
    float* wq = fb_q + Hi * di;
    for (unsigned f = blockIdx.x; f < nfail; f += gridDim.x) {
        const int r = a.fail_list[f];
        const int64_t t = a.t_begin + r;
        const int64_t n = t + 1 < a.N ? t + 1 : a.N;
        int32_t* out = a.idx + (int64_t)r * a.ld_idx;
        __syncthreads();                                             // fb_q of the previous row is free
        if (n <= a.K) {
            for (int i = threadIdx.x; i < a.K; i += FB_THREADS) out[i] = i < n ? i : -1;
            continue;
        }
        for (int i = threadIdx.x; i < Hi * di; i += FB_THREADS) {
            const int64_t e = t * Hi * di + i;
            float v;
            if (ia.dtype == SA_BF16) v = to_f32(static_cast<const bf16*>(ia.q_idx)[e]);
            else if (ia.dtype == SA_FP8_E4M3) v = e4m3_to_f32(static_cast<const uint8_t*>(ia.q_idx)[e]);
            else v = static_cast<const float*>(ia.q_idx)[e];
            fb_q[i] = v;
        }
        for (int h = threadIdx.x; h < Hi; h += FB_THREADS) {
            float wv = ia.w[t * Hi + h];
            if (ia.dtype == SA_FP8_E4M3) wv *= ia.q_scale[t * Hi + h];
            wq[h] = wv;
        }
        __syncthreads();
        float* row = a.scratch + (int64_t)r * a.ld_scratch;
        for (int64_t j = threadIdx.x; j < n; j += FB_THREADS) {
            float s = 0.0f;
            for (int h = 0; h < Hi; ++h) {
                float acc = 0.0f;
                for (int d = 0; d < di; ++d) acc = fmaf(fb_q[h * di + d], key_elem(ia, j, d), acc);
                s = fmaf(wq[h], fmaxf(acc, 0.0f), s);
            }
            if (ia.dtype == SA_FP8_E4M3) s *= ia.k_scale[j];
            row[j] = s;
        }
        __syncthreads();
        radix_select_row([&](int64_t j) { return score_key(__ldcg(row + j)); }, n, a.K, out, sh);
    }
}

}  // namespace

cudaError_t launch_sample_gather(const void* k_idx, int row_bytes, const float* k_scale, int64_t ns, int lg,
                                 void* ksamp, float* ksamp_scale, cudaStream_t s)
{
    if (ns <= 0) return cudaSuccess;
    const int chunks = row_bytes / 16;
    const int64_t total = ns * chunks;
    const unsigned blocks = (unsigned)min64(4 * 148, (total + 255) / 256);
    sample_gather_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(k_idx), chunks, k_scale, ns, lg,
                                                static_cast<uint4*>(ksamp), ksamp_scale);
    return cudaGetLastError();
}

size_t fused_threshold_smem(int64_t max_samples) { return sizeof(uint32_t) * (size_t)max_samples; }

cudaError_t launch_sample_threshold(const FusedSelectArgs& a, const float* ssc, int64_t ld_ssc, int64_t max_samples,
                                    cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
    const size_t smem = fused_threshold_smem(max_samples);
    cudaError_t e = cudaFuncSetAttribute(sample_threshold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    sample_threshold_kernel<<<a.rows, TH_THREADS, smem, s>>>(a, ssc, ld_ssc);
    return cudaGetLastError();
}

size_t fused_select_smem(const FusedSelectArgs& a)
{
    return sizeof(unsigned long long) * ((size_t)a.cand_cap + FS_BIN_CAP) + sizeof(unsigned) * HBINS +
           sizeof(uint32_t) * (size_t)a.words + sizeof(unsigned) * ((size_t)a.nseg + 1);
}

cudaError_t launch_fused_select(const FusedSelectArgs& a, cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
    const size_t smem = fused_select_smem(a);
    cudaError_t e = cudaFuncSetAttribute(fused_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fused_select_kernel<<<a.rows, FS_THREADS, smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t fb_smem = sizeof(float) * ((size_t)a.ia.Hi * a.ia.di + a.ia.Hi);
    e = cudaFuncSetAttribute(fused_fallback_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fb_smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)min64(a.rows, device_sm_count());
    fused_fallback_kernel<<<grid, FB_THREADS, fb_smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sa
