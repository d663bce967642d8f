// Dense causal attention with the sigmoid output gate on the 5th-generation
// tensor core: the full-attention control branch ("From Full Attention to
// Sparsity": sparse attention pays off once the indexer's cost is below the
// attention it saves) and, in the sparse prefill, the rows whose kept set is
// all or most of their history, masked to the kept positions ("Hybrid
// Attention Architectures...", section 3.1: exact attention over the
// candidate set). dqk = dv = 128, bf16, 16 query heads sharing one key/value
// head.
//
// One CTA per 16 consecutive queries, as two Q tiles of 8 queries: a tile's
// 8 x 16 (query, head) rows are the M = 128 side of its MMAs, so a softmax
// thread owns one whole row of S and of O (TMEM lane = row), and the row's
// running maximum and sum stay in its registers. CTAs are issued from the
// last queries down (longest rows first).
//   - warp 0: TMA loads of the two Q tiles (once) and of 64-key K and V
//     tiles (128-byte swizzle) through a 3-stage ring; both Q tiles use each
//     K/V tile;
//   - warp 1 (one thread): per key tile, S = Q K^T (M = 128, N = 64 keys) of
//     each Q tile into one of its two TMEM buffers, then O += P V (M = 128,
//     N = 128 value columns, the value tile read MN-major) of the previous
//     key tile into each Q tile's TMEM accumulator (the two tiles use all
//     512 TMEM columns);
//   - warps 2..5 and 6..9: the softmax of Q tile 0 and of Q tile 1, one TMEM
//     lane quarter per warp, the two warpgroups running side by side (one
//     warp per sub-partition was too few to hide the softmax's latencies:
//     631 -> 674 TFLOP/s at 16K): scale to the exp2 domain, causal mask
//     (and, for rows t >= mask_from, the kept-position bitmap), row maximum,
//     P = exp2(s - m) (the ex2.approx unit) in bf16 to shared memory as the
//     K-major A operand of the PV product, row sum of the same rounded
//     values. A row's maximum is raised only when a score exceeds it by more
//     than 2^8 (then the thread's O row in TMEM and its sum are rescaled,
//     which does not change the result); at the end the gate and the bf16
//     store of the thread's row.
#include "attn_common.cuh"
#include "tc.cuh"
#include "../../include/sparse_attn.h"

namespace sa {

__device__ unsigned g_dense_tc_error = 0;

namespace {

constexpr int DT_D = 128;
constexpr int DT_Q = 8;                        // queries per Q tile
constexpr int DT_H = 16;                       // heads per query (one key/value head)
constexpr int DT_M = DT_Q * DT_H;              // 128 MMA rows per Q tile
constexpr int DT_G = 2;                        // Q tiles per CTA, each with its own softmax warpgroup
constexpr int DT_CQ = DT_G * DT_Q;             // queries per CTA
constexpr int DT_N = 64;                       // keys per tile
constexpr int DT_STAGES = 3;
constexpr int DT_QCB = DT_M * 128;             // a 64-column block of a Q tile: 128 rows x 128 B
constexpr int DT_QBYTES = 2 * DT_QCB;          // 32 KB per Q tile
constexpr int DT_KCB = DT_N * 128;             // a 64-column block of a key / value tile: 64 rows x 128 B
constexpr int DT_KV = 2 * DT_KCB;              // 16 KB
constexpr int DT_STAGE = 2 * DT_KV;            // key tile + value tile
constexpr int DT_PBYTES = DT_M * 128;          // P tile: 128 rows x 64 keys bf16
constexpr int DT_OFF_Q = 0;                                      // [G]
constexpr int DT_OFF_KV = DT_OFF_Q + DT_G * DT_QBYTES;           // [STAGES]
constexpr int DT_OFF_P = DT_OFF_KV + DT_STAGES * DT_STAGE;       // [G] (one P tile per group)
constexpr int DT_OFF_BAR = DT_OFF_P + DT_G * DT_PBYTES;
constexpr int DT_GBAR = 2 * 2 + 3;                               // per group: s full + empty [2], p full, p empty, o full
constexpr int DT_NBAR = 2 * DT_STAGES + 1 + DT_G * DT_GBAR + 1;  // kv, q, groups, drain
constexpr int DT_OFF_BM = DT_OFF_BAR + DT_NBAR * 8 + 16;         // [CQ][words] kept-position bitmaps
constexpr int DT_SOFT = 4 * 32;                                  // softmax threads per group
constexpr int DT_THREADS = (2 + 4 * DT_G) * 32;
constexpr uint32_t DT_TMEM_COLS = 512;        // per group: S [2] x 64 columns, O 128 columns
constexpr float DT_RESCALE = 8.0f;
static_assert(DT_OFF_KV % 1024 == 0 && DT_OFF_P % 1024 == 0 && DT_STAGE % 1024 == 0, "1024-byte tiles");
static_assert(DT_G * 256 <= (int)DT_TMEM_COLS, "TMEM per group");

constexpr uint32_t DT_IDESC_QK = mma_idesc(1u, DT_M, DT_N);                          // A = Q, B = K (K-major)
constexpr uint32_t DT_IDESC_PV = mma_idesc(1u, DT_M, DT_D, false, /*b_mn=*/true);    // A = P, B = V (MN-major)

// 2^x by the special-function unit (PTX ex2.approx, flush-to-zero; 2^-inf = 0)
SA_DEVINL float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

SA_DEVINL float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

SA_DEVINL void bar_soft() { asm volatile("bar.sync 1, %0;" :: "r"(DT_G * DT_SOFT) : "memory"); }

__host__ __device__ inline int64_t dt_words(const DenseArgs& a) { return a.idx ? (a.L + 31) / 32 : 0; }

size_t dt_smem(const DenseArgs& a) { return (size_t)DT_OFF_BM + (size_t)DT_CQ * dt_words(a) * 4 + 1024; }

__global__ void __launch_bounds__(DT_THREADS, 1)
attn_dense_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, DenseArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + DT_OFF_BAR);   // [STAGES] tile landed
    uint64_t* kv_empty = kv_full + DT_STAGES;                            // [STAGES] both PV products done
    uint64_t* q_full = kv_empty + DT_STAGES;
    uint64_t* gbar = q_full + 1;                                         // [G][GBAR]
    uint64_t* drain = gbar + DT_G * DT_GBAR;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    uint32_t* abort_flag = tmem_slot + 1;
    uint32_t* bm = reinterpret_cast<uint32_t*>(smem + DT_OFF_BM);       // [CQ][words]
    // per group g: s_full [2], s_empty [2], p_full, p_empty (the PV product of the
    // P tile done: one phase per key tile), o_full
    auto s_full = [&](int g, int b) { return gbar + g * DT_GBAR + b; };
    auto s_empty = [&](int g, int b) { return gbar + g * DT_GBAR + 2 + b; };
    auto p_full = [&](int g) { return gbar + g * DT_GBAR + 4; };
    auto p_empty = [&](int g) { return gbar + g * DT_GBAR + 5; };
    auto o_full = [&](int g) { return gbar + g * DT_GBAR + 6; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)(gridDim.x - 1 - blockIdx.x) * DT_CQ;
    const int64_t t_last = min64(t0 + DT_CQ, a.L) - 1;
    const int ntiles = (int)((t_last + DT_N) / DT_N);                   // keys 0 .. t_last
    unsigned* err = &g_dense_tc_error;

    if (threadIdx.x == 0) {
        for (int i = 0; i < DT_STAGES; ++i) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 1); }
        mbar_init(q_full, 1);
        for (int g = 0; g < DT_G; ++g) {
            for (int b = 0; b < 2; ++b) { mbar_init(s_full(g, b), 1); mbar_init(s_empty(g, b), 4); }
            mbar_init(p_full(g), 4);
            mbar_init(p_empty(g), 1);
            mbar_init(o_full(g), 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) tmem_alloc(tmem_slot, DT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;                          // tiles requested (producer): drained after an abort

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA loads
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(q_full, DT_G * DT_QBYTES);
            for (int g = 0; g < DT_G; ++g) {
                const int y = (int)((t0 + g * DT_Q) * DT_H);
                tma_load_2d(smem + DT_OFF_Q + g * DT_QBYTES, &tm_q, 0, y, q_full);
                tma_load_2d(smem + DT_OFF_Q + g * DT_QBYTES + DT_QCB, &tm_q, 64, y, q_full);
            }
            for (int kt = 0; kt < ntiles && ok; ++kt) {
                const int st = kt % DT_STAGES;
                ok = mbar_wait(&kv_empty[st], ((kt / DT_STAGES) & 1) ^ 1, err);
                if (!ok) break;
                mbar_arrive_expect_tx(&kv_full[st], DT_STAGE);
                uint8_t* kd = smem + DT_OFF_KV + st * DT_STAGE;
                const int y = kt * DT_N;
                tma_load_2d(kd, &tm_k, 0, y, &kv_full[st]);
                tma_load_2d(kd + DT_KCB, &tm_k, 64, y, &kv_full[st]);
                tma_load_2d(kd + DT_KV, &tm_v, 0, y, &kv_full[st]);
                tma_load_2d(kd + DT_KV + DT_KCB, &tm_v, 64, y, &kv_full[st]);
                ++issued;
            }
            if (!ok) *abort_flag = 1u;
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            bool ok = mbar_wait(q_full, 0, err);
            tc_fence_after();
            for (int j = 0; ok && j <= ntiles; ++j) {
                if (j < ntiles) {                    // S = Q K^T of tile j, both Q tiles
                    const int st = j % DT_STAGES, sb = j & 1;
                    ok = mbar_wait(&kv_full[st], (j / DT_STAGES) & 1, err);
                    const uint32_t ka = smem_u32(smem + DT_OFF_KV + st * DT_STAGE);
                    for (int g = 0; ok && g < DT_G; ++g) {
                        ok = mbar_wait(s_empty(g, sb), ((j >> 1) & 1) ^ 1, err);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t qa = smem_u32(smem + DT_OFF_Q + g * DT_QBYTES);
#pragma unroll
                        for (int ks = 0; ks < DT_D / 16; ++ks) {
                            const uint64_t ad = smem_desc_kmajor(qa + (ks >> 2) * DT_QCB + (ks & 3) * 32, 128);
                            const uint64_t bd = smem_desc_kmajor(ka + (ks >> 2) * DT_KCB + (ks & 3) * 32, 128);
                            tc_mma_f16(tmem + (uint32_t)(g * 256 + sb * DT_N), ad, bd, DT_IDESC_QK, ks > 0);
                        }
                        tc_commit(s_full(g, sb));
                    }
                    if (!ok) break;
                }
                if (j > 0) {                         // O += P V of tile j - 1, both Q tiles
                    const int jp = j - 1, st = jp % DT_STAGES;
                    const uint32_t va = smem_u32(smem + DT_OFF_KV + st * DT_STAGE + DT_KV);
                    for (int g = 0; ok && g < DT_G; ++g) {
                        ok = mbar_wait(p_full(g), jp & 1, err);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t pa = smem_u32(smem + DT_OFF_P + g * DT_PBYTES);
#pragma unroll
                        for (int ks = 0; ks < DT_N / 16; ++ks) {
                            const uint64_t ad = smem_desc_kmajor(pa + ks * 32, 128);
                            const uint64_t bd = smem_desc_mnmajor128(va + ks * 2048, DT_KCB, 1024);
                            tc_mma_f16(tmem + (uint32_t)(g * 256 + 128), ad, bd, DT_IDESC_PV,
                                       (jp > 0 || ks > 0) ? 1u : 0u);
                        }
                        tc_commit(p_empty(g));
                        if (j == ntiles) tc_commit(o_full(g));
                    }
                    if (!ok) break;
                    tc_commit(&kv_empty[st]);
                }
            }
            if (!ok) *abort_flag = 1u;
        }
    } else {
        // ---------------------------------------------------------------- softmax and output
        const int g = (warp - 2) >> 2;                             // Q tile of this warpgroup
        const int q4 = warp & 3;                                   // TMEM lane quarter of this warp
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_t = tmem + lane_off + (uint32_t)(g * 256);
        const uint32_t o_t = s_t + 128u;
        const int r = q4 * 32 + lane;                              // row: query r / 16 of the tile, head r % 16
        const int qi = g * DT_Q + r / DT_H, h = r % DT_H;
        const int64_t t = t0 + qi;
        const float sl2 = a.softmax_scale * LOG2E;
        const int64_t words = dt_words(a);
        // kept-position bitmaps of the CTA's masked queries (rows t >= mask_from)
        const bool masked = a.idx != nullptr && t >= a.mask_from && t < a.L;
        if (a.idx) {
            const int et = threadIdx.x - 64;                       // 0 .. G * 128 - 1
            for (int64_t i = et; i < DT_CQ * words; i += DT_G * DT_SOFT) bm[i] = 0u;
            bar_soft();
            for (int qq = 0; qq < DT_CQ; ++qq) {
                const int64_t tq = t0 + qq;
                if (tq >= a.L || tq < a.mask_from) continue;
                const int32_t* sel = a.idx + tq * a.K;
                for (int i = et; i < a.K; i += DT_G * DT_SOFT) {
                    const int32_t p = sel[i];
                    if (p >= 0 && p <= tq) atomicOr(&bm[qq * words + (p >> 5)], 1u << (p & 31));
                }
            }
            bar_soft();
        }
        const uint32_t* mybm = bm + qi * words;
        uint8_t* prow = smem + DT_OFF_P + g * DT_PBYTES + r * 128;
        float m = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int sb = j & 1;
            if (ok) ok = mbar_wait(s_full(g, sb), (j >> 1) & 1, err);
            tc_fence_after();
            uint32_t sr[DT_N];
            tmem_ld32(s_t + (uint32_t)(sb * DT_N), *reinterpret_cast<uint32_t(*)[32]>(sr));
            tmem_ld32(s_t + (uint32_t)(sb * DT_N + 32), *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty(g, sb));
            // keys j0 .. j0 + 63: causal (<= t) and, for masked rows, kept
            const int64_t j0 = (int64_t)j * DT_N;
            uint64_t keep = ~0ull;
            if (masked) keep = (uint64_t)mybm[j0 >> 5] | ((uint64_t)mybm[(j0 >> 5) + 1 < words ? (j0 >> 5) + 1 : (j0 >> 5)] << 32);
            if (masked && (j0 >> 5) + 1 >= words) keep &= 0xFFFFFFFFull;
            const int64_t lim = t - j0;                            // keys c <= lim are visible
            if (lim < 63) keep &= lim < 0 ? 0ull : ((2ull << lim) - 1ull);
            if (t >= a.L) keep = 0ull;
            // the row maximum on the raw scores (the scale is positive); masked
            // keys become -inf, which the exponential below maps to 0
            if (!__all_sync(0xffffffffu, keep == ~0ull)) {
#pragma unroll
                for (int c = 0; c < DT_N; ++c)
                    if (!((keep >> c) & 1ull)) sr[c] = __float_as_uint(-INFINITY);
            }
            // four independent chains of three-input maxima (not one 64-deep chain)
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < DT_N; c += 8) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    mx[u] = fmax3(mx[u], __uint_as_float(sr[c + 2 * u]), __uint_as_float(sr[c + 2 * u + 1]));
            }
            float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
            const bool need = tmax > m + DT_RESCALE;
            if (__any_sync(0xffffffffu, need)) {
                // raise this warp's maxima that need it and rescale their O rows
                // (O holds tiles 0 .. j-1 once the PV product of tile j - 1 is done)
                float f = 1.0f;
                if (need) {
                    f = m == -INFINITY ? 0.0f : exp2f(m - tmax);
                    m = tmax;
                    l *= f;
                }
                if (j > 0) {
                    if (ok) ok = mbar_wait(p_empty(g), (j - 1) & 1, err);
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < DT_D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(o_t + (uint32_t)c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
                        tmem_st32(o_t + (uint32_t)c0, o);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
            }
            // P of the tile, once the PV product of the previous tile has read the buffer
            if (ok) ok = mbar_wait(p_empty(g), (j & 1) ^ 1, err);
            const float nref = m == -INFINITY ? 0.0f : -m;
            float2 l2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                            make_float2(0.0f, 0.0f)};
#pragma unroll
            for (int c8 = 0; c8 < DT_N / 8; ++c8) {
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t pk = pack_bf16x2(ex2_approx(fmaf(__uint_as_float(sr[c8 * 8 + 2 * e]), sl2, nref)),
                                                    ex2_approx(fmaf(__uint_as_float(sr[c8 * 8 + 2 * e + 1]), sl2, nref)));
                    l2[e] = __fadd2_rn(l2[e], bf16x2_to_f32x2(pk));
                    w4[e] = pk;
                }
                *reinterpret_cast<uint4*>(prow + ((c8 ^ (r & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            l += ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y)) + ((l2[2].x + l2[2].y) + (l2[3].x + l2[3].y));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(g));
        }
        // the row's output
        if (ok) ok = mbar_wait(o_full(g), 0, err);
        tc_fence_after();
        const float gs = (t < a.L && l > 0.0f) ? (1.0f / (1.0f + expf(-a.gate[t * a.Hq + h]))) / l : 0.0f;
        bf16* out = static_cast<bf16*>(a.out) + (t * a.Hq + h) * DT_D;
#pragma unroll
        for (int c0 = 0; c0 < DT_D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(o_t + (uint32_t)c0, o);
            tmem_ld_wait();
            if (t < a.L) {
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(o[c]) * gs, __uint_as_float(o[c + 1]) * gs);
                    v.y = pack_bf16x2(__uint_as_float(o[c + 2]) * gs, __uint_as_float(o[c + 3]) * gs);
                    v.z = pack_bf16x2(__uint_as_float(o[c + 4]) * gs, __uint_as_float(o[c + 5]) * gs);
                    v.w = pack_bf16x2(__uint_as_float(o[c + 6]) * gs, __uint_as_float(o[c + 7]) * gs);
                    *reinterpret_cast<uint4*>(out + c0 + c) = v;
                }
            }
        }
        tc_fence_before();
        if (!ok && lane == 0) *abort_flag = 1u;
    }

    // After a wait gave up (never expected): let the copies and MMAs still in
    // flight land, with bounded waits, before the shared memory and TMEM go.
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            (void)mbar_wait(q_full, 0, err);
            for (int kt = max(0, issued - DT_STAGES); kt < issued; ++kt)
                (void)mbar_wait(&kv_full[kt % DT_STAGES], (kt / DT_STAGES) & 1, err);
        }
        if (warp == 1 && lane == 0) {
            tc_commit(drain);
            (void)mbar_wait(drain, 0, err);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, DT_TMEM_COLS);
    }
}

}  // namespace

cudaError_t attention_dense_tc_device_errors(unsigned* bits, bool reset)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, g_dense_tc_error, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_dense_tc_error, &zero, sizeof(unsigned));
    }
    return e;
}

bool attention_dense_tc_supported(const DenseArgs& a)
{
    if (a.D != DT_D || a.Hq != DT_H || a.L <= 0 || a.L * DT_H > INT32_MAX) return false;
    if (!(a.softmax_scale > 0.0f)) return false;            // the row maximum is taken on raw scores
    const uintptr_t addr = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
                           reinterpret_cast<uintptr_t>(a.v);
    if (addr & 15) return false;
    if (a.ld_k % 8 != 0 || a.ld_v % 8 != 0 || a.ld_k < DT_D || a.ld_v < DT_D) return false;
    if (a.idx && a.K < 1) return false;
    return dt_smem(a) <= 227 * 1024;
}

cudaError_t launch_attention_dense_tc(const DenseArgs& a, cudaStream_t s)
{
    if (a.L <= 0) return cudaSuccess;
    CUtensorMap tq, tk, tv;
    if (!make_tensor_map_2d(&tq, a.q, 2, a.L * DT_H, DT_D, DT_D, 64, DT_M) ||
        !make_tensor_map_2d(&tk, a.k, 2, a.L, DT_D, a.ld_k, 64, DT_N) ||
        !make_tensor_map_2d(&tv, a.v, 2, a.L, DT_D, a.ld_v, 64, DT_N))
        return cudaErrorNotSupported;
    const size_t smem = dt_smem(a);
    cudaError_t e = cudaFuncSetAttribute(attn_dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
    }
    const unsigned grid = (unsigned)((a.L + DT_CQ - 1) / DT_CQ);
    return launch_kernel(attn_dense_tc_kernel, dim3(grid), dim3(DT_THREADS), smem, s, false, tq, tk, tv, a);
}

}  // namespace sa
