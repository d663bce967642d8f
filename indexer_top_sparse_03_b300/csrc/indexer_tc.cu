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
// Persistent CTAs, one per SM, each walking a contiguous range of work items
// (query tile, group of up to 8 key tiles; key tiles wholly outside the
// causal window are never visited) that the host cuts so that every CTA gets
// about the same number of key tiles. The key tiles of an item alternate
// between two independent pipelines (even / odd tiles), each with its own
// stage ring, MMA thread, 128x256 fp32 accumulator (2 x 256 = all 512 TMEM
// columns) and eight epilogue warps, so that one pipeline's epilogue runs
// while the other's MMAs fill its accumulator. Warp roles:
//   warps 0, 2  TMA producers of pipelines 0 / 1: the item's query tile
//               (shared, double-buffered) and their key tiles through a ring
//               of 128-byte-swizzled K-major stages
//   warps 1, 3  MMA issuers (one thread each, kind::f16 or kind::f8f6f4);
//               warp 1 owns the TMEM allocation
//   warp 4      staging: the item's head weights (FP8: times the query-row
//               scale) and, in filter mode, its thresholds, one item ahead
//   warps 5-20  epilogue, eight per pipeline (two per TMEM sub-partition,
//               each taking half of the 256 columns): TMEM -> registers
//               (32 columns per load), ReLU, weighted head sum on packed
//               fp32x2 FMAs, causal mask, fp32 store
// Every wait is bounded (see tc.cuh).
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
constexpr int TC_GRP = 2;                  // independent pipelines, one per key-tile parity
constexpr int TC_GROUP = INDEXER_GROUP;    // key tiles per work item
#ifndef SA_TC_ITEM_COST
#define SA_TC_ITEM_COST 8
#endif
constexpr int TC_ITEM_COST = SA_TC_ITEM_COST;   // scheduling cost of an item beyond its tiles (in tiles)
constexpr int TC_EPI_PER_GRP = 8;          // epilogue warps of a pipeline (two per TMEM sub-partition)
constexpr int TC_EPI_WARPS = TC_GRP * TC_EPI_PER_GRP;
// warps 0 / 2: TMA producers of pipelines 0 / 1; warps 1 / 3: their MMA
// issuers; warp 4: staging; warps 5 ..: epilogue (pipeline 0 first)
constexpr int TC_STAGE_WARP = 4;
constexpr int TC_EPI_WARP0 = 5;
constexpr int TC_THREADS = 32 * (TC_EPI_WARP0 + TC_EPI_WARPS);
constexpr int TC_EPI_THREADS = 32 * TC_EPI_WARPS;
constexpr int TC_EPI_COLS = TC_BN * 4 / TC_EPI_PER_GRP;   // accumulator columns per epilogue warp
static_assert(TC_EPI_PER_GRP % 4 == 0 && TC_EPI_COLS % 32 == 0, "epilogue warps cover TMEM evenly");
static_assert(TC_GRP * TC_BN <= 512, "one TMEM accumulator per pipeline");

template <int ES, int DI, int HI, bool FILTER = false>
struct TcCfg {
    static constexpr int TQ = TC_BN / HI;                  // queries per tile
    static constexpr int ROWB = DI * ES;                   // bytes per operand row
    static constexpr int KB = ROWB < 128 ? ROWB : 128;     // K-block bytes = swizzle span
    static constexpr int NKB = ROWB / KB;
    static constexpr int KSTEPS = KB / 32;                 // MMAs per K-block (K = 32 bytes)
    static constexpr int A_BYTES = TC_BM * ROWB;
    static constexpr int B_BYTES = TC_BN * ROWB;
    // key-tile stages per pipeline (filter mode keeps room for its lists)
    static constexpr int STG = FILTER ? 2 : (A_BYTES <= 8192 ? 4 : (A_BYTES <= 16384 ? 3 : 2));
    static constexpr int B_BUFS = (TC_GRP * STG * A_BYTES + 2 * B_BYTES <= 176 * 1024) ? 2 : 1;
    static constexpr int OFF_B = TC_GRP * STG * A_BYTES;
    static constexpr int OFF_W = OFF_B + B_BUFS * B_BYTES;     // [2][TC_BN] staged head weights
    static constexpr int OFF_THR = OFF_W + 2 * TC_BN * 4;      // filter: [2][TQ] staged thresholds
    static constexpr int NSUB = 4 * TC_GRP;                    // sub-lists per query (sub-partition x pipeline)
    static constexpr int OFF_CNT = OFF_THR + 2 * TQ * 4;       // filter: [TQ][NSUB] sub-list counts
    // filter mode: the local candidate lists
    static constexpr int OFF_C = (OFF_CNT + TQ * NSUB * 4 + 1023) / 1024 * 1024;
    static constexpr int BAR_BYTES = 8 * (2 * TC_GRP * STG + 4 + 2 * TC_GRP + 4) + 16;
    static constexpr int SMEM_MAX = 227 * 1024 - 1024;         // opt-in maximum less the alignment slack
    // candidates per query and work item kept in shared memory (filter mode)
    static constexpr int LCAP_FIT = (SMEM_MAX - OFF_C - BAR_BYTES) / (TQ * 8);
    // a query's list is NSUB sub-lists, each filled by the one warp that owns
    // those 32 keys of the tiles of one pipeline
    static constexpr int LCAP = (LCAP_FIT > 1024 ? 1024 : (LCAP_FIT < NSUB ? NSUB : LCAP_FIT)) / NSUB * NSUB;
    static constexpr int SUBCAP = LCAP / NSUB;
    // filter mode keeps one count register per query of a warp's slice
    static constexpr bool FILTER_OK = LCAP_FIT >= 64 && HI >= 4;
    static constexpr int L_BYTES = FILTER && FILTER_OK ? TQ * LCAP * 8 : 0;
    static constexpr int OFF_BAR = OFF_C + L_BYTES;
    // never less than 116 KB, so that two CTAs cannot share an SM (each holds
    // all 512 TMEM columns)
    static constexpr int SMEM_NEED = OFF_BAR + BAR_BYTES + 1024;
    static constexpr int SMEM = SMEM_NEED > 116 * 1024 ? SMEM_NEED : 116 * 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(SUBCAP * NSUB == LCAP, "whole sub-lists per query");
    static_assert(HI <= 32 && TC_EPI_COLS % HI == 0, "a warp's columns hold whole queries");
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

// The fp32 value v with score_key(v) == key, as a comparison bound:
// score_key(s) >= key  <=>  s >= key_threshold(key) for every non-NaN s.
// Keys at or below the key of -inf admit every score (-inf); keys above the
// key of +inf admit none (NaN compares false).
SA_DEVINL float key_threshold(uint32_t key)
{
    if (key <= 0x007FFFFFu) return __uint_as_float(0xFF800000u);
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The registers of a finished TMEM load, passed through an empty asm after
// the wait, so that no use of them is scheduled before the wait.
SA_DEVINL void reg_fence32(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Weighted ReLU head sum of one (key, query) score from its HI accumulator
// columns; w holds the query's HI head weights (16-byte aligned). With four or
// more heads the sum runs on packed fp32x2 lanes (two heads per instruction).
template <int HI>
SA_DEVINL float head_sum(const uint32_t* r, const float* w)
{
    if constexpr (HI >= 4) {
        float2 acc2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int h4 = 0; h4 < HI; h4 += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(w + h4);
            acc2 = __ffma2_rn(make_float2(fmaxf(__uint_as_float(r[h4]), 0.0f), fmaxf(__uint_as_float(r[h4 + 1]), 0.0f)),
                              make_float2(w4.x, w4.y), acc2);
            acc2 = __ffma2_rn(make_float2(fmaxf(__uint_as_float(r[h4 + 2]), 0.0f), fmaxf(__uint_as_float(r[h4 + 3]), 0.0f)),
                              make_float2(w4.z, w4.w), acc2);
        }
        return acc2.x + acc2.y;
    } else {
        float s = 0.0f;
#pragma unroll
        for (int h = 0; h < HI; ++h) s = fmaf(w[h], fmaxf(__uint_as_float(r[h]), 0.0f), s);
        return s;
    }
}

// Epilogue of one accumulator tile for one warp: its key (TMEM lane) x its
// TC_EPI_COLS columns (TC_EPI_COLS / HI queries), read in chunks of 32
// columns. The accumulator is released (one arrival per warp) as soon as the
// last chunk has arrived in registers, so that the next MMA into this buffer
// overlaps the last chunk's arithmetic. FULL tiles lie inside every query's
// causal window; the others test each (query, key) pair: kept iff t < T and
// j < n_t.
//
// Store mode writes the score (a warp writes 32 consecutive keys of one
// query). Filter mode keeps a pair iff its score reaches the query's
// threshold: the warp ballots its 32 keys per query and appends the kept ones
// to its own sub-list of the query (no other warp writes there, so the count
// is a register of this warp); counts keep growing past subcap (the overflow
// is detected when the item is written out). A kept pair is stored as
// (score bits << 32 | ~j); the selection turns the bits into the
// order-preserving key when it gathers the pairs. Sub-lists of one query lie
// nsub * subcap entries apart.
template <int HI, bool FULL, bool FP8, bool FILTER, int NSUB>
SA_DEVINL void epi_tile(uint32_t taddr, const float* w, const float* thr, float ks, float* p, int64_t ld_s,
                        int64_t j, int t_first, const IndexerArgs& a, unsigned (&cnt)[TC_EPI_COLS / HI],
                        unsigned long long* lsub, int subcap, uint64_t* empty_bar)
{
    constexpr int NCH = TC_EPI_COLS / 32;
    constexpr int QPC = 32 / HI;                       // queries per 32-column chunk
    const int lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    uint32_t r[32];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        tmem_ld32(taddr + c * 32, r);
        tmem_ld_wait();
        reg_fence32(r);
        if (c + 1 == NCH) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar);
        }
#pragma unroll
        for (int qq = 0; qq < QPC; ++qq) {
            const int q = c * QPC + qq;
            float s = head_sum<HI>(r + qq * HI, w + q * HI);
            if (FP8) s *= ks;
            bool in = true;
            if (!FULL) {
                const int t = t_first + q;
                in = t < a.T && j < indexer_row_n(a, t);
            }
            if constexpr (!FILTER) {
                if (in) p[(int64_t)q * ld_s] = s;
            } else {
                const bool pass = in && s >= thr[q];
                const unsigned m = __ballot_sync(0xFFFFFFFFu, pass);
                if (m) {                               // warp-uniform
                    const unsigned slot = cnt[q] + (unsigned)__popc(m & below);
                    if (pass && slot < (unsigned)subcap)
                        lsub[(size_t)q * NSUB * subcap + slot] =
                            ((unsigned long long)__float_as_uint(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)j);
                    cnt[q] += (unsigned)__popc(m);
                }
            }
        }
    }
}


// Two independent pipelines share the CTA: pipeline g takes the key tiles of
// parity g (counted over the CTA's whole item range), with its own TMA
// producer, stage ring, MMA issuer, TMEM accumulator (256 columns each) and
// eight epilogue warps; the query tile of an item and its staged weights are
// shared. One pipeline's waits (each mbarrier round trip and each MMA issue
// costs the single issuing thread hundreds of cycles) then overlap the
// other's, and its epilogue overlaps the other's MMAs.
template <int ES, int DI, int HI, bool FILTER>
__global__ void __launch_bounds__(TC_THREADS, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  IndexerArgs a, const __grid_constant__ TcSchedule sched)
{
    using C = TcCfg<ES, DI, HI, FILTER>;
    constexpr int TQ = C::TQ;
    constexpr int STG = C::STG;
    constexpr int NQ = TC_EPI_COLS / HI;               // queries of one epilogue warp's slice
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment (the swizzled TMA tiles) by pointer arithmetic on
    // the shared-memory pointer itself, so that the compiler keeps every
    // access below in the shared address space (32-bit shared loads and
    // stores rather than generic ones)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = smem;                                                 // [TC_GRP][STG] key tiles
    uint8_t* sB = smem + C::OFF_B;
    float* sW = reinterpret_cast<float*>(smem + C::OFF_W);             // [2][TC_BN]
    float* sThr = reinterpret_cast<float*>(smem + C::OFF_THR);         // [2][TQ]
    unsigned* sCnt = reinterpret_cast<unsigned*>(smem + C::OFF_CNT);   // [TQ][NSUB]
    unsigned long long* sL = reinterpret_cast<unsigned long long*>(smem + C::OFF_C);   // [TQ][LCAP], filter mode
    constexpr bool filter = FILTER && C::FILTER_OK;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* a_full = bars;                           // [TC_GRP][STG]
    uint64_t* a_empty = bars + TC_GRP * STG;           // [TC_GRP][STG]
    uint64_t* b_full = bars + 2 * TC_GRP * STG;        // [2]
    uint64_t* b_empty = b_full + 2;                    // [2] (one commit per pipeline)
    uint64_t* acc_full = b_empty + 2;                  // [TC_GRP]
    uint64_t* acc_empty = acc_full + TC_GRP;           // [TC_GRP]
    uint64_t* st_full = acc_empty + TC_GRP;            // [2] staged weights / thresholds ready
    uint64_t* st_empty = st_full + 2;                  // [2] staged buffer free again
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(st_empty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < TC_GRP * STG; ++i) { mbar_init(&a_full[i], 1); mbar_init(&a_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&b_full[i], 1); mbar_init(&b_empty[i], TC_GRP); }
        for (int i = 0; i < TC_GRP; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], TC_EPI_PER_GRP); }
        for (int i = 0; i < 2; ++i) { mbar_init(&st_full[i], 32); mbar_init(&st_empty[i], TC_EPI_WARPS); }
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

    if (warp < 4 && (warp & 1) == 0) {
        // ------------------------------------------------------------ producer of pipeline g
        const int g = warp >> 1;
        if (lane == 0) {
            int s = 0, bb = 0, gt = 0;
            uint32_t aph = 0, bph = 0;
            uint64_t* af = a_full + g * STG;
            uint64_t* ae = a_empty + g * STG;
            uint8_t* sAg = sA + (size_t)g * STG * C::A_BYTES;
            for (; it.valid(); item_next<TQ>(a, it)) {
                const int t0 = a.t_begin + it.qi * TQ;
                const int ntiles = item_tiles_total<TQ>(a, it.qi);
                const int k_begin = it.g * TC_GROUP, k_end = min(ntiles, k_begin + TC_GROUP);
                if (g == 0) {                            // the query tile, for both pipelines
                    if (!mbar_wait(&b_empty[bb], bph ^ 1, &g_tc_error)) break;
                    mbar_arrive_expect_tx(&b_full[bb], C::B_BYTES);
                    uint8_t* bdst = sB + (C::B_BUFS == 2 ? bb : 0) * C::B_BYTES;
                    for (int kb = 0; kb < C::NKB; ++kb)
                        tma_load_2d(bdst + kb * TC_BN * C::KB, &tm_q, kb * (C::KB / ES), t0 * HI, &b_full[bb]);
                    if (C::B_BUFS == 2) { bb ^= 1; if (bb == 0) bph ^= 1; } else { bph ^= 1; }
                }
                bool ok = true;
                for (int kt = k_begin; kt < k_end; ++kt) {
                    if ((gt++ & 1) != g) continue;
                    if (!mbar_wait(&ae[s], aph ^ 1, &g_tc_error)) { ok = false; break; }
                    mbar_arrive_expect_tx(&af[s], C::A_BYTES);
                    uint8_t* adst = sAg + s * C::A_BYTES;
                    for (int kb = 0; kb < C::NKB; ++kb)
                        tma_load_2d(adst + kb * TC_BM * C::KB, &tm_k, kb * (C::KB / ES), kt * TC_BM, &af[s]);
                    if (++s == STG) { s = 0; aph ^= 1; }
                }
                if (!ok) break;
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ MMA issuer of pipeline g
        const int g = warp >> 1;
        if (lane == 0) {
            int s = 0, bb = 0, gt = 0;
            uint32_t aph = 0, bph = 0, acph = 0;
            uint64_t* af = a_full + g * STG;
            uint64_t* ae = a_empty + g * STG;
            const uint32_t sAg = smem_u32(sA + (size_t)g * STG * C::A_BYTES);
            const uint32_t d = tmem + (uint32_t)(g * TC_BN);
            for (; it.valid(); item_next<TQ>(a, it)) {
                const int ntiles = item_tiles_total<TQ>(a, it.qi);
                const int k_begin = it.g * TC_GROUP, k_end = min(ntiles, k_begin + TC_GROUP);
                if (!mbar_wait(&b_full[bb], bph, &g_tc_error)) break;
                tc_fence_after();
                const uint32_t b_base = smem_u32(sB + (C::B_BUFS == 2 ? bb : 0) * C::B_BYTES);
                bool ok = true;
                for (int kt = k_begin; kt < k_end; ++kt) {
                    if ((gt++ & 1) != g) continue;
                    if (!mbar_wait(&af[s], aph, &g_tc_error) || !mbar_wait(&acc_empty[g], acph ^ 1, &g_tc_error)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = sAg + s * C::A_BYTES;
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
                    tc_commit(&ae[s]);               // smem stage free once these MMAs finish
                    tc_commit(&acc_full[g]);         // accumulator ready for the epilogue
                    if (++s == STG) { s = 0; aph ^= 1; }
                    acph ^= 1;
                }
                if (!ok) break;
                tc_commit(&b_empty[bb]);             // this pipeline is done with the query tile
                if (C::B_BUFS == 2) { bb ^= 1; if (bb == 0) bph ^= 1; } else { bph ^= 1; }
            }
        }
    } else if (warp == TC_STAGE_WARP) {
        // ------------------------------------------------------------ staging
        // Head weights of the item's query tile (FP8: times the query-row
        // scale) and, in filter mode, its thresholds as fp32 bounds, staged
        // one item ahead into a double buffer.
        int sb = 0;
        uint32_t sph = 0;
        for (; it.valid(); item_next<TQ>(a, it)) {
            if (!mbar_wait(&st_empty[sb], sph ^ 1, &g_tc_error)) break;
            const int t0 = a.t_begin + it.qi * TQ;
            float* wd = sW + sb * TC_BN;
            for (int i = lane; i < TC_BN; i += 32) {
                const int t = t0 + i / HI;
                float wv = 0.0f;
                if (t < a.T) {
                    wv = a.w[(int64_t)t * HI + (i % HI)];
                    if (ES == 1) wv *= a.q_scale[(int64_t)t * HI + (i % HI)];
                }
                wd[i] = wv;
            }
            if (filter) {
                for (int q = lane; q < TQ; q += 32) {
                    const int t = t0 + q;
                    sThr[sb * TQ + q] = t < a.T ? key_threshold(a.thr[t - a.t_begin]) : __uint_as_float(0x7FFFFFFFu);
                }
            }
            mbar_arrive(&st_full[sb]);               // one arrival per lane, after its own writes
            if (++sb == 2) { sb = 0; sph ^= 1; }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = threadIdx.x - 32 * TC_EPI_WARP0;  // 0 .. TC_EPI_THREADS - 1
        const int g = (warp - TC_EPI_WARP0) / TC_EPI_PER_GRP;   // pipeline of this warp
        const int sub = warp & 3;                       // TMEM sub-partition of this warp
        const int part = ((warp - TC_EPI_WARP0) % TC_EPI_PER_GRP) >> 2;   // which TC_EPI_COLS columns
        const int row = sub * 32 + lane;                // TMEM lane = key within the tile
        const int col0 = part * TC_EPI_COLS;
        const int tq_first = col0 / HI;
        const bool fp8 = (ES == 1);
        int sb = 0, gt = 0;
        uint32_t acph = 0, sph = 0;
        bool ok = true;
        // After a timed-out wait the loop keeps its shape (same named-barrier
        // count in every epilogue warp) but touches neither TMEM nor memory.
        for (; it.valid(); item_next<TQ>(a, it)) {
            const int t0 = a.t_begin + it.qi * TQ;
            const int ntiles = item_tiles_total<TQ>(a, it.qi);
            const int k_begin = it.g * TC_GROUP, k_end = min(ntiles, k_begin + TC_GROUP);
            if (ok) ok = mbar_wait(&st_full[sb], sph, &g_tc_error);
            ok = __all_sync(0xffffffffu, ok);
            const float* w_s = sW + sb * TC_BN + col0;
            const float* thr_s = sThr + sb * TQ + tq_first;
            unsigned cnt[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) cnt[q] = 0u;
            unsigned long long* lc = sL + ((size_t)tq_first * C::NSUB + g * 4 + sub) * C::SUBCAP;

            // tiles whose every key is visible to every query of the tile
            // skip the per-query causal mask
            const int64_t n_first = indexer_row_n(a, t0);
            const bool rows_full = t0 + TQ <= a.T;
            // FP8 key scales are loaded one tile (of this pipeline) ahead
            auto key_scale = [&](int kt) -> float {
                const int64_t jj = (int64_t)kt * TC_BM + row;
                return (fp8 && kt < k_end && jj < a.N) ? __ldg(a.k_scale + jj) : 1.0f;
            };
            const int k_mine = k_begin + ((gt & 1) != g ? 1 : 0);
            float ks_next = key_scale(k_mine);
            for (int kt = k_mine; kt < k_end; kt += 2) {
                const int64_t j = (int64_t)kt * TC_BM + row;
                const float ks = ks_next;
                if (fp8) ks_next = key_scale(kt + 2);
                const bool full = rows_full && (int64_t)kt * TC_BM + TC_BM <= n_first;
                if (ok) ok = mbar_wait(&acc_full[g], acph, &g_tc_error);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
                    const uint32_t taddr = tmem + ((uint32_t)(sub * 32) << 16) + (uint32_t)(g * TC_BN + col0);
                    float* p = filter ? nullptr : a.scores + (int64_t)(t0 + tq_first - a.t_begin) * a.ld_s + j;
                    if (full)
                        epi_tile<HI, true, ES == 1, filter, C::NSUB>(taddr, w_s, thr_s, ks, p, a.ld_s, j, t0 + tq_first,
                                                                     a, cnt, lc, C::SUBCAP, &acc_empty[g]);
                    else
                        epi_tile<HI, false, ES == 1, filter, C::NSUB>(taddr, w_s, thr_s, ks, p, a.ld_s, j, t0 + tq_first,
                                                                      a, cnt, lc, C::SUBCAP, &acc_empty[g]);
                }
                acph ^= 1;
            }
            gt += k_end - k_begin;
            // the staged weights and thresholds of this item are no longer read
            __syncwarp();
            if (lane == 0) mbar_arrive(&st_empty[sb]);
            if (++sb == 2) { sb = 0; sph ^= 1; }
            if constexpr (filter) {
                // the item's segment: query t0 + q of this item goes to
                // segment it.g of its row; the count is the true one
                if (lane == 0) {
#pragma unroll
                    for (int q = 0; q < NQ; ++q) sCnt[(tq_first + q) * C::NSUB + g * 4 + sub] = cnt[q];
                }
                asm volatile("bar.sync 1, %0;" :: "r"(TC_EPI_THREADS) : "memory");
                constexpr int TPQ = TC_EPI_THREADS / TQ;              // threads per query
                static_assert(TPQ >= 1, "one thread per query at least");
                const int q = e / TPQ, k0 = e % TPQ;
                const int t = t0 + q;
                if (ok && t < a.T) {
                    unsigned cs[C::NSUB];
                    unsigned cnt_q = 0;
                    bool lost = false;
#pragma unroll
                    for (int sbk = 0; sbk < C::NSUB; ++sbk) {
                        cs[sbk] = sCnt[q * C::NSUB + sbk];
                        cnt_q += cs[sbk];
                        lost = lost || cs[sbk] > (unsigned)C::SUBCAP;
                    }
                    const int64_t seg = (int64_t)(t - a.t_begin) * a.nseg + it.g;
                    unsigned long long* dst = a.seg_cand + seg * a.cap_seg;
                    if (!lost && cnt_q <= (unsigned)a.cap_seg) {
                        unsigned off = 0;
#pragma unroll
                        for (int sbk = 0; sbk < C::NSUB; ++sbk) {
                            const unsigned long long* src = sL + ((size_t)q * C::NSUB + sbk) * C::SUBCAP;
                            for (unsigned k = k0; k < cs[sbk]; k += TPQ) dst[off + k] = src[k];
                            off += cs[sbk];
                        }
                    }
                    // a sub-list that lost pairs makes the segment count as overflowed
                    if (k0 == 0) a.seg_cnt[seg] = lost ? (unsigned)a.cap_seg + 1u : cnt_q;
                }
                // the lists and counts are refilled by the next item
                asm volatile("bar.sync 1, %0;" :: "r"(TC_EPI_THREADS) : "memory");
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
    // items in (qi, g) order, cut into contiguous ranges of about equal cost:
    // a key tile costs one unit and an item TC_ITEM_COST more (its query tile
    // is loaded and its weights staged once per item, which matters in the
    // short items at the start of the causal triangle)
    const int nq = (a.T - a.t_begin + C::TQ - 1) / C::TQ;
    int64_t tiles = 0, items = 0;
    for (int qi = 0; qi < nq; ++qi) {
        const int nt = item_tiles_total<C::TQ>(a, qi);
        const int ng = (nt + TC_GROUP - 1) / TC_GROUP;
        tiles += nt + (int64_t)ng * TC_ITEM_COST;
        items += ng;
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
            done += min(TC_GROUP, nt - g * TC_GROUP) + TC_ITEM_COST;
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
