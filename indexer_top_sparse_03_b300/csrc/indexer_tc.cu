// Indexer score on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   s[t, j] = sum_h w[t,h] * max(0, q_idx[t,h,:] . k_idx[j,:])     (j < n_t)
//
// The light relevance score of every query against every causal history
// position ("Hybrid Attention Architectures...", section 3.1, indexing stage;
// no positional encoding, "From Full Attention to Sparsity", indexer
// paragraph). For FP8 inputs each stored row carries a positive fp32 scale;
// the query scale is folded into the head weight and the key scale multiplies
// the finished head sum (a positive factor commutes with the ReLU).
//
// Tile = 128 keys (the MMA's M side, one TMEM lane per key) x 256 (query,
// head) pairs (the N side: q_idx viewed as a [T*Hi, di] matrix already lists
// the pairs of consecutive queries). With this orientation the head sum of a
// (key, query) score lies in the registers of the one thread that owns the
// key's TMEM lane, so the epilogue needs no cross-thread reduction, and its
// stores are coalesced (a warp writes 32 consecutive keys of one query).
//
// Persistent CTAs, one per SM, each walking a static stride of work items
// (query tile, group of up to 8 key tiles; key tiles wholly outside the
// causal window are never visited). Warp roles:
//   warp 0      TMA producer: query tile once per item, key tiles through a
//               ring of shared-memory stages (128-byte-swizzled K-major tiles)
//   warp 1      TMEM owner (512 columns = two 128x256 fp32 accumulators) and
//               MMA issuer (one thread, kind::f16 or kind::f8f6f4)
//   warps 2-17  epilogue: TMEM -> registers, ReLU, weighted head sum, causal
//               mask, fp32 store; four warps per TMEM sub-partition, each
//               taking a quarter of the 256 columns
// Accumulators are double-buffered so that the epilogue of one key tile
// overlaps the MMAs of the next. Every wait is bounded (see tc.cuh).
//
// Filter mode (the indexer fused with the first step of Top-K): instead of
// storing every score, the epilogue keeps the (key, query) pairs whose score
// reaches the query's threshold, collects them per query in shared memory
// over a work item, and writes them out as that item's segment; nothing of
// the score matrix reaches memory.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "../../include/sparse_attn.h"

namespace sa {

// error word of the bounded waits (read back by sa_device_errors)
__device__ unsigned g_tc_error = 0;

namespace {

constexpr int TC_BM = 128;                 // keys per tile (MMA M)
constexpr int TC_BN = 256;                 // (query, head) pairs per tile (MMA N)
constexpr int TC_ACC = 512 / TC_BN;        // TMEM accumulator buffers (all 512 columns)
constexpr int TC_GROUP = INDEXER_GROUP;    // key tiles per work item
constexpr int TC_EPI_WARPS = 16;                          // four per TMEM sub-partition
constexpr int TC_THREADS = 32 * (2 + TC_EPI_WARPS);
constexpr int TC_EPI_COLS = TC_BN * 4 / TC_EPI_WARPS;     // accumulator columns per epilogue thread

template <int ES, int DI, int HI, bool FILTER = false>
struct TcCfg {
    static constexpr int TQ = TC_BN / HI;                  // queries per tile
    static constexpr int ROWB = DI * ES;                   // bytes per operand row
    static constexpr int KB = ROWB < 128 ? ROWB : 128;     // K-block bytes = swizzle span
    static constexpr int NKB = ROWB / KB;
    static constexpr int KSTEPS = KB / 32;                 // MMAs per K-block (K = 32 bytes)
    static constexpr int A_BYTES = TC_BM * ROWB;
    static constexpr int B_BYTES = TC_BN * ROWB;
    static constexpr int STAGES = (A_BYTES <= 16384) ? 4 : 3;
    static constexpr int B_BUFS = (STAGES * A_BYTES + 2 * B_BYTES <= 160 * 1024) ? 2 : 1;
    static constexpr int OFF_B = STAGES * A_BYTES;
    static constexpr int OFF_W = OFF_B + B_BUFS * B_BYTES;
    static constexpr int OFF_THR = OFF_W + TC_BN * 4;          // filter: TQ thresholds
    static constexpr int OFF_CNT = OFF_THR + TQ * 4;           // filter: [TQ][4] local counts
    // filter mode: the local candidate lists
    static constexpr int OFF_C = (OFF_CNT + TQ * 16 + 1023) / 1024 * 1024;
    static constexpr int BAR_BYTES = 8 * (2 * STAGES + 4 + 2 * TC_ACC) + 16;
    static constexpr int SMEM_MAX = 227 * 1024 - 1024;         // opt-in maximum less the alignment slack
    // candidates per query and work item kept in shared memory (filter mode)
    static constexpr int LCAP_FIT = (SMEM_MAX - OFF_C - BAR_BYTES) / (TQ * 8);
    // a query's list is four sub-lists, one per TMEM sub-partition (each
    // filled by the one warp that owns those 32 keys of the tile)
    static constexpr int LCAP = (LCAP_FIT > 1024 ? 1024 : (LCAP_FIT < 4 ? 4 : LCAP_FIT)) / 4 * 4;
    static constexpr int SUBCAP = LCAP / 4;
    static constexpr bool FILTER_OK = LCAP_FIT >= 64;          // else filter mode is not offered
    static constexpr int L_BYTES = FILTER && FILTER_OK ? TQ * LCAP * 8 : 0;
    static constexpr int OFF_BAR = OFF_C + L_BYTES;
    // never less than 116 KB, so that two CTAs cannot share an SM (each holds
    // all 512 TMEM columns)
    static constexpr int SMEM_NEED = OFF_BAR + BAR_BYTES + 1024;
    static constexpr int SMEM = SMEM_NEED > 116 * 1024 ? SMEM_NEED : 116 * 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(SUBCAP * 4 == LCAP, "four whole sub-lists per query");
    static constexpr uint32_t IDESC = mma_idesc(ES == 2 ? 1u : 0u, TC_BM, TC_BN);
    static_assert(ROWB % KB == 0 && KB >= 32, "operand rows must be 32, 64 or a multiple of 128 bytes");
};

// Work items: query tile qi (TQ queries from t_begin + qi*TQ) x group g of
// TC_GROUP key tiles (only tiles inside the causal window exist). The host
// cuts the item sequence, in (qi, g) order, into one contiguous range per CTA
// with about equal key-tile counts, and passes each CTA's first item; a CTA
// then steps through its range item by item.
constexpr int TC_MAX_CTAS = 256;

struct TcSchedule {
    int qi[TC_MAX_CTAS + 1];                // first item of CTA c is (qi[c], g[c]);
    int g[TC_MAX_CTAS + 1];                 // entry gridDim.x is the end of the last range
};

// key tiles of query tile qi: those below the last row's history end (row
// lengths never decrease with t)
template <int TQ>
__host__ __device__ inline int item_tiles_total(const IndexerArgs& a, int qi)
{
    const int64_t t0 = (int64_t)a.t_begin + (int64_t)qi * TQ;
    const int64_t t_last = min64(t0 + TQ, a.T) - 1;
    return (int)((indexer_row_n(a, t_last) + TC_BM - 1) / TC_BM);
}

struct ItemWalk {
    int qi, g, ng;                          // current item and its query tile's group count
    int end_qi, end_g;
    SA_DEVINL bool valid() const { return qi < end_qi || (qi == end_qi && g < end_g); }
};

template <int TQ>
SA_DEVINL void item_next(const IndexerArgs& a, ItemWalk& w)
{
    if (++w.g < w.ng) return;
    w.g = 0;
    ++w.qi;
    w.ng = (item_tiles_total<TQ>(a, w.qi) + TC_GROUP - 1) / TC_GROUP;
}

// Weighted ReLU head sum of one (key, query) score from its HI accumulator
// columns; w holds the query's HI head weights (16-byte aligned). With four or
// more heads the sum runs on packed fp32x2 lanes (two heads per instruction).
template <int HI>
SA_DEVINL float head_sum(const uint32_t* r, const float* w)
{
    if constexpr (HI >= 4) {
        unsigned long long acc2 = 0ull;
#pragma unroll
        for (int h4 = 0; h4 < HI; h4 += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(w + h4);
            acc2 = f32x2_fma(f32x2_pack(fmaxf(__uint_as_float(r[h4]), 0.0f), fmaxf(__uint_as_float(r[h4 + 1]), 0.0f)),
                             f32x2_pack(w4.x, w4.y), acc2);
            acc2 = f32x2_fma(f32x2_pack(fmaxf(__uint_as_float(r[h4 + 2]), 0.0f), fmaxf(__uint_as_float(r[h4 + 3]), 0.0f)),
                             f32x2_pack(w4.z, w4.w), acc2);
        }
        const float2 s2 = f32x2_unpack(acc2);
        return s2.x + s2.y;
    } else {
        float s = 0.0f;
#pragma unroll
        for (int h = 0; h < HI; ++h) s = fmaf(w[h], fmaxf(__uint_as_float(r[h]), 0.0f), s);
        return s;
    }
}

// Epilogue of one accumulator tile for one thread: TC_EPI_COLS columns of its
// key (TC_EPI_COLS / HI queries). All of them are loaded from TMEM first and
// the accumulator is released (one arrival per warp) before any arithmetic,
// so the next MMA into this buffer overlaps the head sums and stores. FULL
// tiles lie inside every query's causal window; the others test each
// (query, key) pair: store iff t < T and j < n_t.
template <int HI, bool FULL, bool FP8>
SA_DEVINL void epi_tile(uint32_t taddr, const float* w, float ks, float* p, int64_t ld_s, int64_t j,
                        int t_first, const IndexerArgs& a, uint64_t* empty_bar)
{
    constexpr int QPC = 32 / HI;                       // queries per 32 columns
    constexpr int CH = TC_EPI_COLS / 32;
    uint32_t r[CH][32];
#pragma unroll
    for (int c = 0; c < CH; ++c) tmem_ld32(taddr + c * 32, r[c]);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
#pragma unroll
        for (int qq = 0; qq < QPC; ++qq) {
            float s = head_sum<HI>(&r[c][qq * HI], w + (c * QPC + qq) * HI);
            if (FP8) s *= ks;
            if (FULL) {
                *p = s;
            } else {
                const int t = t_first + c * QPC + qq;
                if (t < a.T && j < indexer_row_n(a, t)) *p = s;
            }
            p += ld_s;
        }
    }
}

// Filter-mode epilogue of one accumulator tile for one thread (one key j,
// TC_EPI_COLS / HI queries): a pair is kept iff it is inside the query's
// history and score_key(s) >= thr[q]. The warp ballots its 32 keys per query
// and appends the kept ones to its own sub-list of the query (no other warp
// writes there, so the count needs no atomic); counts keep growing past
// subcap (the overflow is detected when the item is written out).
template <int HI, bool FULL, bool FP8>
SA_DEVINL void epi_filter(uint32_t taddr, const float* w, float ks, int64_t j, int t_first,
                          const IndexerArgs& a, const uint32_t* thr, unsigned* cnt4,
                          unsigned long long* lsub, int subcap, uint64_t* empty_bar)
{
    constexpr int QPC = 32 / HI;
    constexpr int CH = TC_EPI_COLS / 32;
    uint32_t r[CH][32];
#pragma unroll
    for (int c = 0; c < CH; ++c) tmem_ld32(taddr + c * 32, r[c]);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    const int lane = threadIdx.x & 31;
    if (lane == 0) mbar_arrive(empty_bar);
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
#pragma unroll
        for (int qq = 0; qq < QPC; ++qq) {
            const int q = c * QPC + qq;
            float s = head_sum<HI>(&r[c][qq * HI], w + q * HI);
            if (FP8) s *= ks;
            const uint32_t key = score_key(s);
            bool pass = key >= thr[q];
            if (!FULL) {
                const int t = t_first + q;
                pass = pass && t < a.T && j < indexer_row_n(a, t);
            }
            const unsigned m = __ballot_sync(0xFFFFFFFFu, pass);
            if (m) {                                   // warp-uniform
                const unsigned base = cnt4[q * 4];     // this warp's count for query q
                const unsigned slot = base + (unsigned)__popc(m & below);
                if (pass && slot < (unsigned)subcap)
                    lsub[(size_t)q * 4 * subcap + slot] =
                        ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)j);
                __syncwarp();
                if (lane == 0) cnt4[q * 4] = base + (unsigned)__popc(m);
            }
        }
    }
}


template <int ES, int DI, int HI, bool FILTER>
__global__ void __launch_bounds__(TC_THREADS, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  IndexerArgs a, const __grid_constant__ TcSchedule sched)
{
    using C = TcCfg<ES, DI, HI, FILTER>;
    constexpr int TQ = C::TQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::OFF_B;
    float* sW = reinterpret_cast<float*>(smem + C::OFF_W);
    uint32_t* sThr = reinterpret_cast<uint32_t*>(smem + C::OFF_THR);
    unsigned* sCnt = reinterpret_cast<unsigned*>(smem + C::OFF_CNT);
    unsigned long long* sL = reinterpret_cast<unsigned long long*>(smem + C::OFF_C);   // [TQ][LCAP], filter mode
    constexpr bool filter = FILTER && C::FILTER_OK;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* a_full = bars;                       // [STAGES]
    uint64_t* a_empty = bars + C::STAGES;          // [STAGES]
    uint64_t* b_full = bars + 2 * C::STAGES;       // [2]
    uint64_t* b_empty = b_full + 2;                // [2]
    uint64_t* acc_full = b_empty + 2;              // [TC_ACC]
    uint64_t* acc_empty = acc_full + TC_ACC;       // [TC_ACC]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + TC_ACC);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) { mbar_init(&a_full[i], 1); mbar_init(&a_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&b_full[i], 1); mbar_init(&b_empty[i], 1); }
        for (int i = 0; i < TC_ACC; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], TC_EPI_WARPS); }
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    ItemWalk it;
    it.qi = sched.qi[blockIdx.x];
    it.g = sched.g[blockIdx.x];
    it.ng = (item_tiles_total<TQ>(a, it.qi) + TC_GROUP - 1) / TC_GROUP;
    it.end_qi = sched.qi[blockIdx.x + 1];
    it.end_g = sched.g[blockIdx.x + 1];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0, bb = 0;
            uint32_t aph = 0, bph = 0;
            for (; it.valid(); item_next<TQ>(a, it)) {
                const int t0 = a.t_begin + it.qi * TQ;
                const int ntiles = item_tiles_total<TQ>(a, it.qi);
                const int k_begin = it.g * TC_GROUP, k_end = min(ntiles, k_begin + TC_GROUP);
                if (!mbar_wait(&b_empty[bb], bph ^ 1, &g_tc_error)) break;
                mbar_arrive_expect_tx(&b_full[bb], C::B_BYTES);
                uint8_t* bdst = sB + (C::B_BUFS == 2 ? bb : 0) * C::B_BYTES;
                for (int kb = 0; kb < C::NKB; ++kb)
                    tma_load_2d(bdst + kb * TC_BN * C::KB, &tm_q, kb * (C::KB / ES), t0 * HI, &b_full[bb]);
                bool ok = true;
                for (int kt = k_begin; kt < k_end; ++kt) {
                    if (!mbar_wait(&a_empty[s], aph ^ 1, &g_tc_error)) { ok = false; break; }
                    mbar_arrive_expect_tx(&a_full[s], C::A_BYTES);
                    uint8_t* adst = sA + s * C::A_BYTES;
                    for (int kb = 0; kb < C::NKB; ++kb)
                        tma_load_2d(adst + kb * TC_BM * C::KB, &tm_k, kb * (C::KB / ES), kt * TC_BM, &a_full[s]);
                    if (++s == C::STAGES) { s = 0; aph ^= 1; }
                }
                if (!ok) break;
                if (C::B_BUFS == 2) { bb ^= 1; if (bb == 0) bph ^= 1; } else { bph ^= 1; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0, bb = 0, ab = 0;
            uint32_t aph = 0, bph = 0, acph = 0;
            for (; it.valid(); item_next<TQ>(a, it)) {
                const int ntiles = item_tiles_total<TQ>(a, it.qi);
                const int k_begin = it.g * TC_GROUP, k_end = min(ntiles, k_begin + TC_GROUP);
                if (!mbar_wait(&b_full[bb], bph, &g_tc_error)) break;
                tc_fence_after();
                const uint32_t b_base = smem_u32(sB + (C::B_BUFS == 2 ? bb : 0) * C::B_BYTES);
                bool ok = true;
                for (int kt = k_begin; kt < k_end; ++kt) {
                    if (!mbar_wait(&a_full[s], aph, &g_tc_error) || !mbar_wait(&acc_empty[ab], acph ^ 1, &g_tc_error)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + s * C::A_BYTES);
                    const uint32_t d = tmem + (uint32_t)(ab * TC_BN);
#pragma unroll
                    for (int kb = 0; kb < C::NKB; ++kb) {
#pragma unroll
                        for (int ks = 0; ks < C::KSTEPS; ++ks) {
                            const uint64_t ad = smem_desc_kmajor(a_base + kb * TC_BM * C::KB + ks * 32, C::KB);
                            const uint64_t bd = smem_desc_kmajor(b_base + kb * TC_BN * C::KB + ks * 32, C::KB);
                            const uint32_t acc = (kb | ks) != 0;
                            if (ES == 2) tc_mma_f16(d, ad, bd, C::IDESC, acc);
                            else tc_mma_f8(d, ad, bd, C::IDESC, acc);
                        }
                    }
                    tc_commit(&a_empty[s]);          // smem stage free once these MMAs finish
                    tc_commit(&acc_full[ab]);        // accumulator ready for the epilogue
                    if (++s == C::STAGES) { s = 0; aph ^= 1; }
                    if (++ab == TC_ACC) { ab = 0; acph ^= 1; }
                }
                if (!ok) break;
                tc_commit(&b_empty[bb]);
                if (C::B_BUFS == 2) { bb ^= 1; if (bb == 0) bph ^= 1; } else { bph ^= 1; }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = threadIdx.x - 64;                 // 0 .. 32 * TC_EPI_WARPS - 1
        const int sub = warp & 3;                       // TMEM sub-partition of this warp
        const int half = (warp - 2) >> 2;               // which TC_EPI_COLS columns
        const int row = sub * 32 + lane;                // TMEM lane = key within the tile
        const bool fp8 = (ES == 1);
        int ab = 0;
        uint32_t acph = 0;
        bool ok = true;
        // After a timed-out wait the loop keeps its shape (same named-barrier
        // count in every epilogue warp) but touches neither TMEM nor memory.
        for (; it.valid(); item_next<TQ>(a, it)) {
            const int t0 = a.t_begin + it.qi * TQ;
            const int ntiles = item_tiles_total<TQ>(a, it.qi);
            const int k_begin = it.g * TC_GROUP, k_end = min(ntiles, k_begin + TC_GROUP);
            // head weights of this query tile (FP8: times the query-row scale)
            asm volatile("bar.sync 1, %0;" :: "r"(TC_EPI_WARPS * 32) : "memory");
            for (int i = e; i < TC_BN; i += TC_EPI_WARPS * 32) {
                const int t = t0 + i / HI;
                float wv = 0.0f;
                if (t < a.T) {
                    wv = a.w[(int64_t)t * HI + (i % HI)];
                    if (fp8) wv *= a.q_scale[(int64_t)t * HI + (i % HI)];
                }
                sW[i] = wv;
            }
            if (filter && e < TQ) {
                const int t = t0 + e;
                sThr[e] = t < a.T ? a.thr[t - a.t_begin] : 0xFFFFFFFFu;
                reinterpret_cast<uint4*>(sCnt)[e] = make_uint4(0u, 0u, 0u, 0u);
            }
            asm volatile("bar.sync 1, %0;" :: "r"(TC_EPI_WARPS * 32) : "memory");

            // tiles whose every key is visible to every query of the tile
            // skip the per-query causal mask
            const int64_t n_first = indexer_row_n(a, t0);
            const bool rows_full = t0 + TQ <= a.T;
            const int tq_first = half * (TC_EPI_COLS / HI);
            // FP8 key scales are loaded one tile ahead
            auto key_scale = [&](int kt) -> float {
                const int64_t jj = (int64_t)kt * TC_BM + row;
                return (fp8 && jj < a.N) ? __ldg(a.k_scale + jj) : 1.0f;
            };
            float ks_next = key_scale(k_begin);
            for (int kt = k_begin; kt < k_end; ++kt) {
                const int64_t j = (int64_t)kt * TC_BM + row;
                const float ks = ks_next;
                if (fp8 && kt + 1 < k_end) ks_next = key_scale(kt + 1);
                const bool full = rows_full && (int64_t)kt * TC_BM + TC_BM <= n_first;
                if (ok) ok = mbar_wait(&acc_full[ab], acph, &g_tc_error);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
                    const uint32_t taddr = tmem + ((uint32_t)(sub * 32) << 16) + (uint32_t)(ab * TC_BN + half * TC_EPI_COLS);
                    const float* w_half = sW + tq_first * HI;
                    if constexpr (filter) {
                        // query q's sub-list `sub` starts at sL + (q * 4 + sub) * SUBCAP
                        unsigned long long* lc = sL + ((size_t)tq_first * 4 + sub) * C::SUBCAP;
                        unsigned* c4 = sCnt + tq_first * 4 + sub;
                        if (full)
                            epi_filter<HI, true, ES == 1>(taddr, w_half, ks, j, t0 + tq_first, a, sThr + tq_first,
                                                          c4, lc, C::SUBCAP, &acc_empty[ab]);
                        else
                            epi_filter<HI, false, ES == 1>(taddr, w_half, ks, j, t0 + tq_first, a, sThr + tq_first,
                                                           c4, lc, C::SUBCAP, &acc_empty[ab]);
                    } else {
                        float* p = a.scores + (int64_t)(t0 + tq_first - a.t_begin) * a.ld_s + j;
                        if (full)
                            epi_tile<HI, true, ES == 1>(taddr, w_half, ks, p, a.ld_s, j, 0, a, &acc_empty[ab]);
                        else
                            epi_tile<HI, false, ES == 1>(taddr, w_half, ks, p, a.ld_s, j, t0 + tq_first, a,
                                                         &acc_empty[ab]);
                    }
                }
                if (++ab == TC_ACC) { ab = 0; acph ^= 1; }
            }
            if constexpr (filter) {
                // the item's segment: query t0 + q of this item goes to
                // segment it.g of its row; the count is the true one
                asm volatile("bar.sync 1, %0;" :: "r"(TC_EPI_WARPS * 32) : "memory");
                constexpr int TPQ = TC_EPI_WARPS * 32 / TQ;           // threads per query
                const int q = e / TPQ, k0 = e % TPQ;
                const int t = t0 + q;
                if (ok && t < a.T) {
                    const uint4 c4 = reinterpret_cast<const uint4*>(sCnt)[q];
                    const unsigned cs[4] = {c4.x, c4.y, c4.z, c4.w};
                    const unsigned cnt = c4.x + c4.y + c4.z + c4.w;
                    const bool lost = c4.x > (unsigned)C::SUBCAP || c4.y > (unsigned)C::SUBCAP ||
                                      c4.z > (unsigned)C::SUBCAP || c4.w > (unsigned)C::SUBCAP;
                    const int64_t seg = (int64_t)(t - a.t_begin) * a.nseg + it.g;
                    unsigned long long* dst = a.seg_cand + seg * a.cap_seg;
                    if (!lost && cnt <= (unsigned)a.cap_seg) {
                        unsigned off = 0;
#pragma unroll
                        for (int sb = 0; sb < 4; ++sb) {
                            const unsigned long long* src = sL + ((size_t)q * 4 + sb) * C::SUBCAP;
                            for (unsigned k = k0; k < cs[sb]; k += TPQ) dst[off + k] = src[k];
                            off += cs[sb];
                        }
                    }
                    // a sub-list that lost pairs makes the segment count as overflowed
                    if (k0 == 0) a.seg_cnt[seg] = lost ? (unsigned)a.cap_seg + 1u : cnt;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int ES, int DI, int HI, bool FILTER>
cudaError_t launch_tc_mode(const IndexerArgs& a, cudaStream_t s)
{
    using C = TcCfg<ES, DI, HI, FILTER>;
    CUtensorMap tk, tq;
    if (!make_tensor_map_2d(&tk, a.k_idx, ES, a.N, DI, DI, C::KB / ES, TC_BM) ||
        !make_tensor_map_2d(&tq, a.q_idx, ES, (int64_t)a.T * HI, DI, DI, C::KB / ES, TC_BN))
        return cudaErrorNotSupported;
    // items in (qi, g) order, cut into contiguous ranges of about equal tiles
    const int nq = (a.T - a.t_begin + C::TQ - 1) / C::TQ;
    int64_t tiles = 0, items = 0;
    for (int qi = 0; qi < nq; ++qi) {
        const int nt = item_tiles_total<C::TQ>(a, qi);
        tiles += nt;
        items += (nt + TC_GROUP - 1) / TC_GROUP;
    }
    if (items == 0) return cudaSuccess;
    const int grid = (int)min64(min64(items, device_sm_count()), TC_MAX_CTAS);
    TcSchedule sched;
    int c = 0;
    int64_t done = 0;
    sched.qi[0] = 0;
    sched.g[0] = 0;
    for (int qi = 0; qi < nq && c + 1 < grid; ++qi) {
        const int nt = item_tiles_total<C::TQ>(a, qi);
        const int ng = (nt + TC_GROUP - 1) / TC_GROUP;
        for (int g = 0; g < ng && c + 1 < grid; ++g) {
            // start CTA c + 1 here once CTA c has its share of the tiles
            if (done * grid >= tiles * (int64_t)(c + 1)) {
                ++c;
                sched.qi[c] = qi;
                sched.g[c] = g;
            }
            done += min(TC_GROUP, nt - g * TC_GROUP);
        }
    }
    for (int k = c + 1; k <= grid; ++k) {    // unused CTAs (and the end marker): past the last item
        sched.qi[k] = nq;
        sched.g[k] = 0;
    }
    cudaError_t e = cudaFuncSetAttribute(indexer_tc_kernel<ES, DI, HI, FILTER>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
    }
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, indexer_tc_kernel<ES, DI, HI, FILTER>) != cudaSuccess || fa.maxThreadsPerBlock < TC_THREADS) {
        (void)cudaGetLastError();
        return cudaErrorNotSupported;        // the caller falls back to the CUDA-core kernel
    }
    indexer_tc_kernel<ES, DI, HI, FILTER><<<grid, TC_THREADS, C::SMEM, s>>>(tk, tq, a, sched);
    return cudaGetLastError();
}

template <int ES, int DI, int HI>
cudaError_t launch_tc(const IndexerArgs& a, cudaStream_t s)
{
    if (!a.thr) return launch_tc_mode<ES, DI, HI, false>(a, s);
    if constexpr (TcCfg<ES, DI, HI, false>::FILTER_OK) return launch_tc_mode<ES, DI, HI, true>(a, s);
    return cudaErrorNotSupported;
}

template <int ES, int DI>
cudaError_t launch_tc_hi(const IndexerArgs& a, cudaStream_t s)
{
    switch (a.Hi) {
    case 1: return launch_tc<ES, DI, 1>(a, s);
    case 2: return launch_tc<ES, DI, 2>(a, s);
    case 4: return launch_tc<ES, DI, 4>(a, s);
    case 8: return launch_tc<ES, DI, 8>(a, s);
    case 16: return launch_tc<ES, DI, 16>(a, s);
    case 32: return launch_tc<ES, DI, 32>(a, s);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// host helpers shared with the other TMA kernels
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        (void)cudaGetLastError();
    });
    return fn;
}

bool make_tensor_map_2d(CUtensorMap* m, const void* base, int elem_bytes, int64_t rows, int64_t cols,
                        int64_t row_stride_elems, int box_cols, int box_rows, bool swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride_elems * elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const int span = box_cols * elem_bytes;
    const CUtensorMapSwizzle sw = !swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE
                                : span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : span == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 148;
    }
    return n;
}

template <int ES, int DI>
int filter_lcap_hi(int Hi)
{
    switch (Hi) {
    case 1: return TcCfg<ES, DI, 1>::FILTER_OK ? TcCfg<ES, DI, 1>::LCAP : 0;
    case 2: return TcCfg<ES, DI, 2>::FILTER_OK ? TcCfg<ES, DI, 2>::LCAP : 0;
    case 4: return TcCfg<ES, DI, 4>::FILTER_OK ? TcCfg<ES, DI, 4>::LCAP : 0;
    case 8: return TcCfg<ES, DI, 8>::FILTER_OK ? TcCfg<ES, DI, 8>::LCAP : 0;
    case 16: return TcCfg<ES, DI, 16>::FILTER_OK ? TcCfg<ES, DI, 16>::LCAP : 0;
    case 32: return TcCfg<ES, DI, 32>::FILTER_OK ? TcCfg<ES, DI, 32>::LCAP : 0;
    default: return 0;
    }
}

int indexer_filter_lcap(const IndexerArgs& a)
{
    if (!indexer_tc_supported(a)) return 0;
    if (a.dtype == SA_BF16) {
        switch (a.di) {
        case 16: return filter_lcap_hi<2, 16>(a.Hi);
        case 32: return filter_lcap_hi<2, 32>(a.Hi);
        case 64: return filter_lcap_hi<2, 64>(a.Hi);
        case 128: return filter_lcap_hi<2, 128>(a.Hi);
        default: return 0;
        }
    }
    switch (a.di) {
    case 32: return filter_lcap_hi<1, 32>(a.Hi);
    case 64: return filter_lcap_hi<1, 64>(a.Hi);
    case 128: return filter_lcap_hi<1, 128>(a.Hi);
    case 256: return filter_lcap_hi<1, 256>(a.Hi);
    default: return 0;
    }
}

int indexer_query_tile(const IndexerArgs& a) { return a.Hi > 0 ? TC_BN / a.Hi : 0; }

cudaError_t indexer_device_errors(unsigned* bits, bool reset)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, g_tc_error, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(unsigned));
    }
    return e;
}

bool indexer_tc_supported(const IndexerArgs& a)
{
    const bool hi_ok = a.Hi == 1 || a.Hi == 2 || a.Hi == 4 || a.Hi == 8 || a.Hi == 16 || a.Hi == 32;
    if (!hi_ok) return false;
    if (a.dtype == SA_BF16) return a.di == 16 || a.di == 32 || a.di == 64 || a.di == 128;
    if (a.dtype == SA_FP8_E4M3) return a.di == 32 || a.di == 64 || a.di == 128 || a.di == 256;
    return false;
}

cudaError_t launch_indexer_tc(const IndexerArgs& a, cudaStream_t s)
{
    if (a.T - a.t_begin <= 0 || a.N <= 0) return cudaSuccess;
    if (a.thr && indexer_filter_lcap(a) < a.cap_seg) return cudaErrorNotSupported;
    if (a.dtype == SA_BF16) {
        switch (a.di) {
        case 16: return launch_tc_hi<2, 16>(a, s);
        case 32: return launch_tc_hi<2, 32>(a, s);
        case 64: return launch_tc_hi<2, 64>(a, s);
        case 128: return launch_tc_hi<2, 128>(a, s);
        default: break;
        }
    } else if (a.dtype == SA_FP8_E4M3) {
        switch (a.di) {
        case 32: return launch_tc_hi<1, 32>(a, s);
        case 64: return launch_tc_hi<1, 64>(a, s);
        case 128: return launch_tc_hi<1, 128>(a, s);
        case 256: return launch_tc_hi<1, 256>(a, s);
        default: break;
        }
    }
    return cudaErrorNotSupported;
}

}  // namespace sa
