// Exact attention over the kept rows of prefill queries on the 5th-generation
// tensor core ("Hybrid Attention Architectures...", section 3.1: exact
// attention over the candidate set; the sigmoid output gate of the section 3.3
// pseudocode in the epilogue; section 5, item 1: the gather of non-contiguous
// rows is the operator to get right). dqk = dv = 128, bf16, one key/value head
// shared by every group of 16 query heads.
//
// Work item = (query row, group of 16 heads). Persistent CTAs, one per SM,
// take the items round robin; an item's kept rows are taken in tiles of 128:
//   - warps 0..7 gather each tile's key and value rows (16 rows each, one
//     warp instruction of 16-byte cp.async per row: half the lanes copy the
//     key, half the value) into a 3-stage ring of 64 KB stages, in the
//     128-byte-swizzled layout the MMAs read: the key tile is the K-major A
//     operand of S^T = K Q^T (M = 128 keys) and the value tile, byte for
//     byte, the MN-major A operand of O^T += V^T P^T (M = 128 value columns).
//     The copies arrive on the stage's barrier by themselves when they land
//     (cp.async.mbarrier.arrive.noinc), so a producer only ever waits for a
//     free stage; the MMA thread orders the landed rows before its
//     async-proxy reads with a proxy fence. Measured at the 8K prefill
//     rows: 4 gathering warps 2.68 ms, 8 warps 1.31 ms (the copies' issue
//     rate per warp bounds it), 16 warps spill registers. TMA gather4 fills
//     the same layout from one thread, but delivered about 7 bytes per clock
//     per SM (2.4 ms).
//   - warp 8 (one thread) issues the MMAs (M = 128, N = 16 heads): S^T of a
//     tile into one of two TMEM buffers, and O^T of an item into one of two
//     TMEM buffers, accumulated over the item's tiles; S^T of tile j + 1 is
//     computed while the softmax of tile j runs. The query tile comes by TMA.
//   - warps 9..12 run the softmax, one TMEM lane quarter each: a thread owns
//     one key of the tile and its 16 head scores. The 16 running maxima are
//     common to all 128 threads (one barrier-with-OR per tile decides whether
//     any score exceeds its maximum by more than 2^8 in the exp2 domain; only
//     then are the maxima raised and O^T and the partial sums rescaled, which
//     does not change the result). P^T is written to shared memory in bf16 as
//     the K-major B operand of the PV product; the sums add the same rounded
//     values. At the end of the item a thread owns one value column of the
//     16 heads' outputs, divides by the sums and applies the gate.
// At 16 query heads per key/value head the work is the gather, not the
// arithmetic; a 64 KB tile is usable only once the last of its 4096 copies
// has landed, which makes this kernel slower than the per-warp rings of the
// mma.sync kernel (22.8 against 16.3 ms at the 128K prefill rows), so it runs
// only when chosen (SA_ATTN_TCGEN05).
#include "attn_common.cuh"
#include "tc.cuh"
#include "../../include/sparse_attn.h"

namespace sa {

__device__ unsigned g_attn_tc_error = 0;

namespace {

constexpr int AT_D = 128;                      // dqk = dv
constexpr int AT_KEYS = 128;                   // keys per tile (the MMA M of S^T)
constexpr int AT_HEADS = 16;                   // heads per item (the MMA N)
constexpr int AT_STAGES = 3;
constexpr int AT_CB = AT_KEYS * 128;           // one 64-column block of a tile: 128 rows x 128 B
constexpr int AT_KV_BYTES = 2 * AT_CB;         // key (or value) tile: two column blocks
constexpr int AT_STAGE = 2 * AT_KV_BYTES;      // key tile + value tile
constexpr int AT_HB = AT_HEADS * 128;          // 16 rows x 128 B: a column block of Q or P^T
constexpr int AT_QP = 2 * AT_HB;               // Q tile or P^T tile (two column blocks)
constexpr int AT_OFF_Q = AT_STAGES * AT_STAGE;            // [2] query tiles
constexpr int AT_OFF_P = AT_OFF_Q + 2 * AT_QP;            // [2] P^T tiles
constexpr int AT_OFF_RED = AT_OFF_P + 2 * AT_QP;          // [4][16] per-warp maxima
constexpr int AT_OFF_SUM = AT_OFF_RED + 4 * 16 * 4;       // [4][16] per-warp sums
constexpr int AT_OFF_BAR = AT_OFF_SUM + 4 * 16 * 4;
constexpr int AT_NBAR = 2 * AT_STAGES + 5 * 2 * 2 + 1;    // kv, q, s, p, o: full + empty; drain
constexpr int AT_SMEM = AT_OFF_BAR + AT_NBAR * 8 + 16 + 1024;   // + tmem slot, + alignment slack
constexpr int AT_PRODUCERS = 8;                // gathering warps
constexpr int AT_RPW = AT_KEYS / AT_PRODUCERS; // rows of a tile per gathering warp
static_assert(AT_RPW <= 32 && AT_KEYS % AT_PRODUCERS == 0, "a lane holds the position of one of its warp's rows");
constexpr int AT_MMA_WARP = AT_PRODUCERS;
constexpr int AT_THREADS = (AT_PRODUCERS + 1 + 4) * 32;

constexpr int AT_EPI_THREADS = 128;
constexpr uint32_t AT_TMEM_COLS = 64;          // S^T [2] x 16 columns, O^T [2] x 16 columns
constexpr float AT_RESCALE = 8.0f;             // lazy-rescale margin (exp2 domain)
static_assert(AT_SMEM <= 227 * 1024, "one CTA per SM");
static_assert(AT_OFF_Q % 1024 == 0 && AT_OFF_P % 1024 == 0, "swizzled tiles sit on 1024-byte boundaries");

constexpr uint32_t AT_IDESC_QK = mma_idesc(1u, AT_KEYS, AT_HEADS);                // A = keys (K-major)
constexpr uint32_t AT_IDESC_PV = mma_idesc(1u, AT_D, AT_HEADS, /*a_mn=*/true);    // A = values (MN-major)

// Arrive on `bar` once all of this thread's earlier cp.async copies have
// landed (the barrier's expected count includes this arrival).
SA_DEVINL void cp_async_arrive_noinc(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}
SA_DEVINL void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

SA_DEVINL bool bar_red_or(bool v)              // the four softmax warps
{
    uint32_t r;
    asm volatile("{ .reg .pred p, q; setp.ne.u32 q, %1, 0; bar.red.or.pred p, 1, %2, q; selp.u32 %0, 1, 0, p; }"
                 : "=r"(r) : "r"((uint32_t)v), "r"(AT_EPI_THREADS) : "memory");
    return r != 0;
}
SA_DEVINL void bar_epi() { asm volatile("bar.sync 2, %0;" :: "r"(AT_EPI_THREADS) : "memory"); }

struct AtItem {
    int r, hg, n_sel, ntiles;
    int64_t n;
};

SA_DEVINL AtItem at_item(const AttnArgs& a, int i, int groups)
{
    AtItem it;
    it.r = i / groups;
    it.hg = i % groups;
    it.n = attn_hist_len(a, it.r);
    it.n_sel = attn_kept(a, it.r, it.n);
    it.ntiles = (it.n_sel + AT_KEYS - 1) / AT_KEYS;
    return it;
}

// The CTA's tiles in order (items round robin, tiles of an item in order),
// for the gathers and the prefetch of their kept positions.
struct TileWalk {
    int i, j;
    AtItem it;
};

SA_DEVINL void walk_skip_empty(TileWalk& w, const AttnArgs& a, int groups, int items)
{
    for (; w.i < items; w.i += gridDim.x) {
        w.it = at_item(a, w.i, groups);
        if (w.it.ntiles > 0) return;
    }
}

SA_DEVINL void walk_next(TileWalk& w, const AttnArgs& a, int groups, int items)
{
    if (++w.j < w.it.ntiles) return;
    w.j = 0;
    w.i += gridDim.x;
    walk_skip_empty(w, a, groups, items);
}

// Key row of slot `row` of the walker's tile (slots past the kept entries,
// and positions outside the history, read row 0 of the sequence: masked
// or never expected).
SA_DEVINL int64_t walk_row(const TileWalk& w, const AttnArgs& a, int row)
{
    const int slot = w.j * AT_KEYS + row;
    int p = slot < w.it.n_sel ? a.idx[(int64_t)w.it.r * a.K + slot] : 0;
    if (p < 0 || p >= w.it.n) p = 0;
    return attn_base(a, w.it.r) + p;
}

constexpr int AT_PQ = 3;                       // tiles whose positions are loaded ahead of their copies

__global__ void __launch_bounds__(AT_THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, AttnArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment (the swizzled tiles) by arithmetic on the shared
    // pointer itself, so that every access stays in the shared address space
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + AT_OFF_BAR);   // [STAGES] tile landed
    uint64_t* kv_empty = kv_full + AT_STAGES;                            // [STAGES] tile consumed
    uint64_t* q_full = kv_empty + AT_STAGES;                             // [2] query tile landed
    uint64_t* q_empty = q_full + 2;                                      // [2] item's last S^T issued
    uint64_t* s_full = q_empty + 2;                                      // [2] S^T in TMEM
    uint64_t* s_empty = s_full + 2;                                      // [2] S^T read by the softmax
    uint64_t* p_full = s_empty + 2;                                      // [2] P^T in smem
    uint64_t* p_empty = p_full + 2;                                      // [2] PV product of that P^T done
    uint64_t* o_full = p_empty + 2;                                      // [2] item's O^T complete
    uint64_t* o_empty = o_full + 2;                                      // [2] O^T read out
    uint64_t* drain = o_empty + 2;                                       // MMAs settled after an abort
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    uint32_t* abort_flag = tmem_slot + 1;
    float* red = reinterpret_cast<float*>(smem + AT_OFF_RED);
    float* sums = reinterpret_cast<float*>(smem + AT_OFF_SUM);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < AT_STAGES; ++i) { mbar_init(&kv_full[i], AT_PRODUCERS * 32); mbar_init(&kv_empty[i], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1);
            mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], 4);
            mbar_init(&p_full[i], 4); mbar_init(&p_empty[i], 1);
            mbar_init(&o_full[i], 1); mbar_init(&o_empty[i], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
    }
    if (warp == AT_MMA_WARP) tmem_alloc(tmem_slot, AT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_wait();                          // the kept positions
    griddep_launch();

    const int groups = a.Hq / AT_HEADS;
    const int items = a.rows * groups;
    unsigned* err = &g_attn_tc_error;
    int issued_items = 0;                    // query tiles requested (warp 0): drained after an abort

    if (warp < AT_PRODUCERS) {
        // ---------------------------------------------------------------- gathers
        // this lane's 16-byte piece of a row: pieces 0..15 of the key, 16..31 of
        // the value; its place in a swizzled row depends on the row (below)
        const bool is_v = lane >= 16;
        const int piece = lane & 15;
        const bf16* src_base = (is_v ? static_cast<const bf16*>(a.v) : static_cast<const bf16*>(a.k)) + piece * 8;
        const int64_t src_ld = is_v ? a.ld_v : a.ld_k;
        const int dst_base = (is_v ? AT_KV_BYTES : 0) + (piece >> 3) * AT_CB;
        const int row0 = warp * AT_RPW;          // this warp's rows of each tile
        const int my_row = row0 + lane % AT_RPW; // the row whose position this lane holds
        // Each thread's copies into a stage arrive on the stage's barrier when
        // they land (cp.async.mbarrier.arrive.noinc): the producers never wait
        // for their own copies, only for a free stage.
        TileWalk wi, wp;                     // the tile being issued; the one whose positions load next
        wi.i = blockIdx.x;
        wi.j = 0;
        walk_skip_empty(wi, a, groups, items);
        wp = wi;
        int64_t pq[AT_PQ];                   // row of this lane's slot in the next AT_PQ tiles
#pragma unroll
        for (int u = 0; u < AT_PQ; ++u) {
            pq[u] = wp.i < items ? walk_row(wp, a, my_row) : 0;
            if (wp.i < items) walk_next(wp, a, groups, items);
        }
        int g = 0, ia = -1;
        bool ok = true;
        for (; wi.i < items; walk_next(wi, a, groups, items), ++g) {
            const int st = g % AT_STAGES;
            if (wi.j == 0) {                 // a new item: its query tile
                ++ia;
                if (warp == 0) {
                    const int qb = ia & 1;
                    if (lane == 0) {
                        ok = mbar_wait(&q_empty[qb], ((ia >> 1) & 1) ^ 1, err);
                        if (ok) {
                            mbar_arrive_expect_tx(&q_full[qb], AT_QP);
                            uint8_t* qd = smem + AT_OFF_Q + qb * AT_QP;
                            const int y = wi.it.r * a.Hq + wi.it.hg * AT_HEADS;
                            tma_load_2d(qd, &tm_q, 0, y, &q_full[qb]);
                            tma_load_2d(qd + AT_HB, &tm_q, 64, y, &q_full[qb]);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
                    if (!ok) break;
                    ++issued_items;
                }
            }
            const int64_t grow = pq[0];
#pragma unroll
            for (int u = 0; u + 1 < AT_PQ; ++u) pq[u] = pq[u + 1];
            pq[AT_PQ - 1] = wp.i < items ? walk_row(wp, a, my_row) : 0;
            if (wp.i < items) walk_next(wp, a, groups, items);
            if (lane == 0) ok = mbar_wait(&kv_empty[st], ((g / AT_STAGES) & 1) ^ 1, err);
            ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
            if (!ok) break;
            uint8_t* stage = smem + st * AT_STAGE + dst_base;
#pragma unroll 8
            for (int rr = 0; rr < AT_RPW; ++rr) {
                const int r = row0 + rr;
                const int64_t gr = __shfl_sync(0xffffffffu, grow, rr);
                cp_async16(stage + r * 128 + (((piece & 7) ^ (r & 7)) << 4), src_base + gr * src_ld, true);
            }
            cp_async_arrive_noinc(&kv_full[st]);
        }
        cp_async_wait_all();                 // nothing in flight when the CTA ends
        if (!ok && lane == 0) *abort_flag = 1u;
    } else if (warp == AT_MMA_WARP) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            int g = 0, ia = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
                const AtItem it = at_item(a, i, groups);
                if (it.ntiles == 0) continue;
                const int qb = ia & 1, ob = ia & 1;
                if (!mbar_wait(&q_full[qb], (ia >> 1) & 1, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t qa = smem_u32(smem + AT_OFF_Q + qb * AT_QP);
                const uint32_t o_t = tmem + 32u + (uint32_t)(ob * 16);
                for (int j = 0; j <= it.ntiles; ++j) {
                    if (j < it.ntiles) {                 // S^T of tile j
                        const int gg = g + j, st = gg % AT_STAGES, sb = gg & 1;
                        ok = mbar_wait(&kv_full[st], (gg / AT_STAGES) & 1, err) &&
                             mbar_wait(&s_empty[sb], ((gg >> 1) & 1) ^ 1, err);
                        if (!ok) break;
                        // the gathered rows were written by cp.async (generic
                        // proxy): order them before the MMAs' (async proxy) reads
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint32_t ka = smem_u32(smem + st * AT_STAGE);
#pragma unroll
                        for (int ks = 0; ks < AT_D / 16; ++ks) {
                            const uint64_t ad = smem_desc_kmajor(ka + (ks >> 2) * AT_CB + (ks & 3) * 32, 128);
                            const uint64_t bd = smem_desc_kmajor(qa + (ks >> 2) * AT_HB + (ks & 3) * 32, 128);
                            tc_mma_f16(tmem + (uint32_t)(sb * 16), ad, bd, AT_IDESC_QK, ks > 0);
                        }
                        tc_commit(&s_full[sb]);
                        if (j == it.ntiles - 1) tc_commit(&q_empty[qb]);
                    }
                    if (j > 0) {                         // O^T += V^T P^T of tile j - 1
                        const int gp = g + j - 1, st = gp % AT_STAGES, pb = gp & 1;
                        if (j == 1) ok = mbar_wait(&o_empty[ob], ((ia >> 1) & 1) ^ 1, err);
                        if (ok) ok = mbar_wait(&p_full[pb], (gp >> 1) & 1, err);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t va = smem_u32(smem + st * AT_STAGE + AT_KV_BYTES);
                        const uint32_t pa = smem_u32(smem + AT_OFF_P + pb * AT_QP);
#pragma unroll
                        for (int ks = 0; ks < AT_KEYS / 16; ++ks) {
                            const uint64_t ad = smem_desc_mnmajor128(va + ks * 2048, AT_CB, 1024);
                            const uint64_t bd = smem_desc_kmajor(pa + (ks >> 2) * AT_HB + (ks & 3) * 32, 128);
                            tc_mma_f16(o_t, ad, bd, AT_IDESC_PV, (j > 1 || ks > 0) ? 1u : 0u);
                        }
                        tc_commit(&kv_empty[st]);
                        tc_commit(&p_empty[pb]);
                        if (j == it.ntiles) tc_commit(&o_full[ob]);
                    }
                }
                g += it.ntiles;
                ++ia;
            }
            if (!ok) *abort_flag = 1u;
        }
    } else {
        // ---------------------------------------------------------------- softmax and output
        const int q4 = warp & 3;                                   // TMEM lane quarter of this warp
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int kt = q4 * 32 + lane;                             // key of the tile / value column
        const float sl2 = a.softmax_scale * LOG2E;
        const uint32_t kin = (uint32_t)(kt & 63);
        // this thread's bf16 of P^T, row h: K-major, 128-byte swizzle (16-byte
        // chunk index XOR the row's index within its 8-row group)
        const int p_off = (kt >> 6) * AT_HB + (int)((kin & 7u) << 1);
        int g = 0, ia = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < items; i += gridDim.x) {
            const AtItem it = at_item(a, i, groups);
            bf16* out = static_cast<bf16*>(a.out) + ((int64_t)it.r * a.Hq + it.hg * AT_HEADS) * AT_D + kt;
            if (it.ntiles == 0) {                                  // nothing kept: zero output
#pragma unroll
                for (int h = 0; h < AT_HEADS; ++h) out[h * AT_D] = __float2bfloat16_rn(0.0f);
                continue;
            }
            const uint32_t o_t = tmem + lane_off + 32u + (uint32_t)((ia & 1) * 16);
            float m[AT_HEADS], l[AT_HEADS];
#pragma unroll
            for (int h = 0; h < AT_HEADS; ++h) { m[h] = -INFINITY; l[h] = 0.0f; }
            for (int j = 0; j < it.ntiles; ++j) {
                const int gg = g + j, sb = gg & 1;
                if (ok) ok = mbar_wait(&s_full[sb], (gg >> 1) & 1, err);
                tc_fence_after();
                uint32_t sr[AT_HEADS];
                tmem_ld16(tmem + lane_off + (uint32_t)(sb * 16), sr);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                const bool valid = j * AT_KEYS + kt < it.n_sel;
                float s[AT_HEADS];
                bool need = j == 0;
#pragma unroll
                for (int h = 0; h < AT_HEADS; ++h) {
                    s[h] = valid ? __uint_as_float(sr[h]) * sl2 : -INFINITY;
                    need |= s[h] > m[h] + AT_RESCALE;
                }
                if (bar_red_or(need)) {
                    // raise the maxima to the tile's (common to the 128 threads)
                    float t[AT_HEADS];
#pragma unroll
                    for (int h = 0; h < AT_HEADS; ++h) t[h] = s[h];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                        for (int h = 0; h < AT_HEADS; ++h) t[h] = fmaxf(t[h], __shfl_xor_sync(0xffffffffu, t[h], off));
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int h = 0; h < AT_HEADS; ++h) red[q4 * AT_HEADS + h] = t[h];
                    }
                    bar_epi();
                    float f[AT_HEADS];
#pragma unroll
                    for (int h = 0; h < AT_HEADS; ++h) {
                        const float mx = fmaxf(fmaxf(fmaxf(red[h], red[16 + h]), fmaxf(red[32 + h], red[48 + h])), m[h]);
                        f[h] = m[h] == -INFINITY ? 0.0f : exp2f(m[h] - mx);
                        m[h] = mx;
                        l[h] *= f[h];
                    }
                    if (j > 0) {
                        // O^T holds tiles 0..j-1 once the PV product of tile j - 1 is done
                        const int gp = gg - 1;
                        if (ok) ok = mbar_wait(&p_empty[gp & 1], (gp >> 1) & 1, err);
                        tc_fence_after();
                        uint32_t o[AT_HEADS];
                        tmem_ld16(o_t, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int h = 0; h < AT_HEADS; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * f[h]);
                        tmem_st16(o_t, o);
                        tmem_st_wait();
                        tc_fence_before();
                    }
                }
                // P^T of the tile, once the PV product two tiles back has read the buffer
                if (ok) ok = mbar_wait(&p_empty[sb], ((gg >> 1) & 1) ^ 1, err);
                uint8_t* pt = smem + AT_OFF_P + sb * AT_QP + p_off;
#pragma unroll
                for (int h = 0; h < AT_HEADS; ++h) {
                    const bf16 pb = __float2bfloat16_rn(exp2f(s[h] - m[h]));
                    l[h] += __bfloat162float(pb);
                    *reinterpret_cast<bf16*>(pt + h * 128 + (int)((((kin >> 3) ^ (uint32_t)(h & 7))) << 4)) = pb;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sb]);
            }
            g += it.ntiles;
            // the item's output: sums over the 128 keys' threads, O^T column of this thread
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int h = 0; h < AT_HEADS; ++h) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
            }
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < AT_HEADS; ++h) sums[q4 * AT_HEADS + h] = l[h];
            }
            if (ok) ok = mbar_wait(&o_full[ia & 1], (ia >> 1) & 1, err);
            tc_fence_after();
            uint32_t o[AT_HEADS];
            tmem_ld16(o_t, o);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[ia & 1]);
            bar_epi();
#pragma unroll
            for (int h = 0; h < AT_HEADS; ++h) {
                const float L = (sums[h] + sums[16 + h]) + (sums[32 + h] + sums[48 + h]);
                const float gs = L > 0.0f ? gate_of(a, it.r, it.hg * AT_HEADS + h) / L : 0.0f;
                out[h * AT_D] = __float2bfloat16_rn(__uint_as_float(o[h]) * gs);
            }
            ++ia;
        }
        if (!ok && lane == 0) *abort_flag = 1u;
    }

    // After a wait gave up (never expected): let the copies and MMAs still in
    // flight land, with bounded waits, before the shared memory and TMEM go.
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {                    // the query tiles (the gathers landed above)
            for (int t = max(0, issued_items - 2); t < issued_items; ++t)
                (void)mbar_wait(&q_full[t & 1], (t >> 1) & 1, err);
        }
        if (warp == AT_MMA_WARP && lane == 0) {          // this thread's MMAs
            tc_commit(drain);
            (void)mbar_wait(drain, 0, err);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == AT_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, AT_TMEM_COLS);
    }
}

}  // namespace

cudaError_t attention_tc_device_errors(unsigned* bits, bool reset)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, g_attn_tc_error, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_attn_tc_error, &zero, sizeof(unsigned));
    }
    return e;
}

bool attention_tc_supported(const AttnArgs& a)
{
    if (a.dtype != SA_BF16 || a.v_aliases_k) return false;
    if (a.dqk != AT_D || a.dv != AT_D || a.Hq <= 0 || a.Hq % AT_HEADS != 0) return false;
    if (a.splits != 1 || a.row_base || a.ctx_len) return false;   // prefill rows: keys of one sequence
    if (a.n_cap <= 0 || a.n_cap > INT32_MAX || (int64_t)a.rows * a.Hq > INT32_MAX) return false;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v) |
                           reinterpret_cast<uintptr_t>(a.q);
    if (addr & 15) return false;
    return a.ld_k % 8 == 0 && a.ld_v % 8 == 0 && a.ld_k >= AT_D && a.ld_v >= AT_D;
}

cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
    CUtensorMap tq;                          // the query tiles: 16 heads x one 64-column block per box
    if (!make_tensor_map_2d(&tq, a.q, 2, (int64_t)a.rows * a.Hq, AT_D, AT_D, 64, AT_HEADS))
        return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
    }
    const int64_t items = (int64_t)a.rows * (a.Hq / AT_HEADS);
    const int grid = (int)min64(items, (int64_t)device_sm_count());
    // (no programmatic dependent launch: the persistent CTAs, placed early,
    // would hold the SMs' shared memory while the previous kernel still
    // needs them; measured 4.4 ms against 0.93 ms at 8K prefill rows)
    return launch_kernel(attn_tc_kernel, dim3(grid), dim3(AT_THREADS), (size_t)AT_SMEM, s, false, tq, a);
}

}  // namespace sa
