// Exact attention over the kept rows, for MQA heads of width 64 or 128
// ("Hybrid Attention Architectures...", section 3.1, exact computation stage
// over the candidate set; the sigmoid output gate of the section 3.3
// pseudocode is applied in the epilogue). The pages name the gather of
// non-contiguous rows as the operator to get right (same page, section 5,
// item 1).
//
// One CTA per (query row, split of its kept rows, group of 16 heads). The 16
// heads of a token share every gathered K/V row (one KV head), so a row is
// fetched once for all of them. The four warps work independently: warp w
// takes the 16-row steps w, w + 4, w + 8, ... of the CTA's kept rows, copies
// each step's K and V rows with 16-byte cp.async into its own three-stage
// ring of padded shared-memory rows (one warp instruction per row: half the
// lanes copy the key, half the value), and keeps its own online softmax
// (running max, sum, 16 x dv fp32 accumulator) over the rows it sees. Every
// warp thus keeps its own loads in flight, and no barrier is needed until
// the end. S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 -> fp32),
// P passing from the S accumulators straight into the A fragments. The
// running max is raised only when a new score exceeds it by more than 2^8 in
// the exp2 domain (the result does not depend on when it is raised; this only
// skips rescales).
// At the end the four warps' (max, sum, accumulator) triples are merged in
// shared memory; with one split the gate is applied and bf16 rows written.
// With up to eight splits the row's splits run as one thread-block cluster
// and merge through distributed shared memory (each CTA finishes the heads
// hh with hh % splits == its rank); with more, the partials go to the
// workspace and the last CTA of the row (atomic ticket) merges them.
#include "attn_common.cuh"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int GA_W = 4;                        // warps per CTA
constexpr int GA_THREADS = 32 * GA_W;
constexpr int GA_ROWS = 16;                    // kept rows per warp step (the MMA key tile)
constexpr float GA_RESCALE = 8.0f;             // lazy-rescale margin (exp2 domain)
constexpr int GA_PQ = 4;                       // steps whose positions are in flight ahead of their copies
constexpr int GA_MAX_CLUSTER = 8;              // portable thread-block cluster size

template <int DQK, int DV, int GA_STAGES>
struct GaCfg {
    static constexpr int K_LD = DQK + 8, V_LD = DV + 8;       // padded rows (bf16 elements)
    static constexpr int KBYTES = GA_ROWS * K_LD * 2;         // K part of one warp stage
    static constexpr int WSTAGE = KBYTES + GA_ROWS * V_LD * 2;
    static constexpr int WRING = GA_STAGES * WSTAGE;          // one warp's ring
    static constexpr int Q_LD = DQK + 8;
    static constexpr int OFF_Q = GA_W * WRING;
    static constexpr int SMEM = OFF_Q + 16 * Q_LD * 2;
    static constexpr int PK = DQK / 8;                        // 16-byte pieces of a key row
    static constexpr int PR = DQK / 8 + DV / 8;               // pieces of a key row + value row
    static constexpr int RPI = 32 / PR;                       // rows per copy instruction
    static_assert(PR == 32 || PR == 16, "one or two rows per warp instruction");
    static_assert(4 * 16 * DV * 4 + 2 * 4 * 16 * 4 + 16 * (DV + 2) * 4 <= OFF_Q, "merge scratch fits the rings");
};

// GA_STAGES = per-warp ring depth: 3 (two CTAs per SM) or 2 (three CTAs per SM)
template <int DQK, int DV, int GA_STAGES, bool CLUSTER>
__global__ void __launch_bounds__(GA_THREADS, GA_STAGES == 2 ? 3 : 2)
attn_gather_kernel(AttnArgs a)
{
    using C = GaCfg<DQK, DV, GA_STAGES>;
    extern __shared__ __align__(16) uint8_t smem[];
    bf16* Qs = reinterpret_cast<bf16*>(smem + C::OFF_Q);
    __shared__ int sh_flag;

    griddep_wait();                          // the kept positions
    griddep_launch();
    const int r = blockIdx.x, split = blockIdx.y, hg = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3, mat = lane >> 3, rr = lane & 7;
    const int64_t n = attn_hist_len(a, r);
    const int n_sel = attn_kept(a, r, n);
    const int per = (a.K + a.splits - 1) / a.splits;
    const int begin = min(split * per, n_sel), end = min(begin + per, n_sel);
    const int cnt = end - begin;
    const int nsteps = (cnt + GA_ROWS - 1) / GA_ROWS;
    const int my_steps = nsteps > warp ? (nsteps - warp + GA_W - 1) / GA_W : 0;
    const int64_t base = attn_base(a, r);
    const int32_t* sel = a.idx + (int64_t)r * a.K;
    const int fallback = cnt > 0 ? sel[begin] : 0;      // a kept position: always a valid row

    // Q tile: 16 heads of this group
    {
        const bf16* q = static_cast<const bf16*>(a.q);
        for (int i = threadIdx.x; i < 16 * (DQK / 8); i += GA_THREADS) {
            const int row = i / (DQK / 8), pc = i % (DQK / 8), h = hg * 16 + row;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < a.Hq) v = *reinterpret_cast<const uint4*>(q + ((int64_t)r * a.Hq + h) * DQK + pc * 8);
            *reinterpret_cast<uint4*>(Qs + row * C::Q_LD + pc * 8) = v;
        }
    }

    // this warp's ring; step k of the warp is CTA step warp + 4k
    uint8_t* ring = smem + warp * C::WRING;
    const int piece = lane % C::PR, sub = lane / C::PR;
    const bool is_k = piece < C::PK;
    const bf16* src_base = is_k ? static_cast<const bf16*>(a.k) + piece * 8
                                : static_cast<const bf16*>(a.v) + (piece - C::PK) * 8;
    const int64_t src_ld = is_k ? a.ld_k : a.ld_v;
    const int dst_ld = is_k ? C::K_LD : C::V_LD;
    const int dst_off = is_k ? piece * 8 : C::KBYTES / 2 + (piece - C::PK) * 8;
    // lanes 0..15 hold the positions of one step's 16 rows
    auto load_pos = [&](int k) -> int {
        int pos = fallback;
        if (k < my_steps && lane < GA_ROWS) {
            const int slot = begin + (warp + k * GA_W) * GA_ROWS + lane;
            pos = slot < end ? sel[slot] : fallback;
            if (pos < 0 || pos >= n) pos = fallback;
        }
        return pos;
    };
    auto issue = [&](int k, int pos) {
        if (k < my_steps) {
            const int64_t grow = base + pos;
            bf16* dst = reinterpret_cast<bf16*>(ring + (k % GA_STAGES) * C::WSTAGE) + dst_off;
#pragma unroll
            for (int r0 = 0; r0 < GA_ROWS; r0 += C::RPI) {
                const int rrow = r0 + sub;
                const int64_t gr = __shfl_sync(0xffffffffu, grow, rrow);
                cp_async16(dst + rrow * dst_ld, src_base + gr * src_ld, true);
            }
        }
        cp_async_commit();                   // one group per step, empty past the end
    };

    // positions are fetched GA_PQ steps before their gathers are issued, so
    // that an index load from L2 never sits between a step and its copies
    int pq[GA_PQ];
#pragma unroll
    for (int i = 0; i < GA_PQ; ++i) pq[i] = load_pos(i);
#pragma unroll
    for (int k = 0; k < GA_STAGES - 1; ++k) {
        issue(k, pq[0]);
#pragma unroll
        for (int i = 0; i + 1 < GA_PQ; ++i) pq[i] = pq[i + 1];
        pq[GA_PQ - 1] = load_pos(k + GA_PQ);
    }
    __syncthreads();                         // the Q tile

    float o[DV / 8][4];
#pragma unroll
    for (int i = 0; i < DV / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const float sl2 = a.softmax_scale * LOG2E;
    const uint32_t qbase = smem_u32(Qs);

    for (int k = 0; k < my_steps; ++k) {
        issue(k + GA_STAGES - 1, pq[0]);
#pragma unroll
        for (int i = 0; i + 1 < GA_PQ; ++i) pq[i] = pq[i + 1];
        pq[GA_PQ - 1] = load_pos(k + GA_STAGES - 1 + GA_PQ);
        cp_async_wait<GA_STAGES - 1>();      // this lane's copies of step k have landed
        __syncwarp();                        // ... and every lane's
        const uint32_t st = smem_u32(ring + (k % GA_STAGES) * C::WSTAGE);
        const uint32_t vst = st + C::KBYTES;
        const int slot0 = begin + (warp + k * GA_W) * GA_ROWS;

        // S = Q K^T for the step's 16 rows (keys)
        float sc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
        for (int ks = 0; ks < DQK / 16; ++ks) {
            uint32_t af[4], bfm[4];
            ldsm_x4(af, qbase + (uint32_t)((((mat & 1) * 8 + rr) * C::Q_LD + ks * 16 + (mat >> 1) * 8) * 2));
            const int krow = (mat >> 1) * 8 + rr;
            const int dim = ks * 16 + (mat & 1) * 8;
            ldsm_x4(bfm, st + (uint32_t)((krow * C::K_LD + dim) * 2));
            mma_16816(sc[0], af, bfm[0], bfm[1]);
            mma_16816(sc[1], af, bfm[2], bfm[3]);
        }
        // mask slots past the end, scale to the exp2 domain
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool valid = slot0 + nt * 8 + 2 * t4 + e < end;
                sc[nt][e] = valid ? sc[nt][e] * sl2 : -INFINITY;
                sc[nt][2 + e] = valid ? sc[nt][2 + e] * sl2 : -INFINITY;
                mx0 = fmaxf(mx0, sc[nt][e]);
                mx1 = fmaxf(mx1, sc[nt][2 + e]);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const bool up0 = mx0 > m0 + GA_RESCALE, up1 = mx1 > m1 + GA_RESCALE;
        if (__any_sync(0xffffffffu, up0 || up1)) {
            float a0 = 1.0f, a1 = 1.0f;
            if (up0) { a0 = (m0 == -INFINITY) ? 0.0f : exp2f(m0 - mx0); m0 = mx0; }
            if (up1) { a1 = (m1 == -INFINITY) ? 0.0f : exp2f(m1 - mx1); m1 = mx1; }
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int i = 0; i < DV / 8; ++i) {
                o[i][0] *= a0; o[i][1] *= a0; o[i][2] *= a1; o[i][3] *= a1;
            }
        }
        const float ref0 = (m0 == -INFINITY) ? 0.0f : m0, ref1 = (m1 == -INFINITY) ? 0.0f : m1;
        uint32_t pa[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t p01 = pack_bf16x2(exp2f(sc[nt][0] - ref0), exp2f(sc[nt][1] - ref0));
            const uint32_t p23 = pack_bf16x2(exp2f(sc[nt][2] - ref1), exp2f(sc[nt][3] - ref1));
            const float2 f01 = bf16x2_to_f32x2(p01), f23 = bf16x2_to_f32x2(p23);
            l0 += f01.x + f01.y;
            l1 += f23.x + f23.y;
            pa[2 * nt] = p01;
            pa[2 * nt + 1] = p23;
        }
        // O += P V over the step's 16 rows
#pragma unroll
        for (int np = 0; np < DV / 16; ++np) {
            uint32_t bfm[4];
            const int vrow = (mat & 1) * 8 + rr;
            const int col = np * 16 + (mat >> 1) * 8;
            ldsm_x4_trans(bfm, vst + (uint32_t)((vrow * C::V_LD + col) * 2));
            mma_16816(o[2 * np], pa, bfm[0], bfm[1]);
            mma_16816(o[2 * np + 1], pa, bfm[2], bfm[3]);
        }
        __syncwarp();                        // the slot is refilled by the next issue
    }
    cp_async_wait<0>();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // merge the four warps' partial triples (the rings are free now)
    __syncthreads();
    float* Ow = reinterpret_cast<float*>(smem);                   // [4][16][DV]
    float* mw = Ow + 4 * 16 * DV;                                 // [4][16]
    float* lw = mw + 4 * 16;                                      // [4][16]
    float* cpart = lw + 4 * 16;                                   // [16][DV + 2] cluster mode: this CTA's partial
#pragma unroll
    for (int i = 0; i < DV / 8; ++i) {
        const int col = i * 8 + 2 * t4;
        *reinterpret_cast<float2*>(&Ow[(warp * 16 + g) * DV + col]) = make_float2(o[i][0], o[i][1]);
        *reinterpret_cast<float2*>(&Ow[(warp * 16 + g + 8) * DV + col]) = make_float2(o[i][2], o[i][3]);
    }
    if (t4 == 0) {
        mw[warp * 16 + g] = m0; mw[warp * 16 + g + 8] = m1;
        lw[warp * 16 + g] = l0; lw[warp * 16 + g + 8] = l1;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 16 * (DV / 2); e += GA_THREADS) {
        const int hh = e / (DV / 2), col = 2 * (e % (DV / 2)), h = hg * 16 + hh;
        if (h >= a.Hq) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < GA_W; ++w) M = fmaxf(M, mw[w * 16 + hh]);
        float L = 0.0f, O0 = 0.0f, O1 = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < GA_W; ++w) {
                const float mwv = mw[w * 16 + hh];
                const float f = mwv == -INFINITY ? 0.0f : exp2f(mwv - M);
                L = fmaf(lw[w * 16 + hh], f, L);
                const float2 ov = *reinterpret_cast<const float2*>(&Ow[(w * 16 + hh) * DV + col]);
                O0 = fmaf(ov.x, f, O0);
                O1 = fmaf(ov.y, f, O1);
            }
        }
        if (CLUSTER) {
            float* p = cpart + hh * (DV + 2);
            *reinterpret_cast<float2*>(p + col) = make_float2(O0, O1);
            if (col == 0) { p[DV] = M; p[DV + 1] = L; }
        } else if (a.splits == 1) {
            const float gs = L > 0.0f ? gate_of(a, r, h) / L : 0.0f;
            *reinterpret_cast<uint32_t*>(static_cast<bf16*>(a.out) + ((int64_t)r * a.Hq + h) * DV + col) =
                pack_bf16x2(O0 * gs, O1 * gs);
        } else {
            float* p = a.part + (((int64_t)r * a.splits + split) * a.Hq + h) * (DV + 2);
            *reinterpret_cast<float2*>(p + col) = make_float2(O0, O1);
            if (col == 0) { p[DV] = M; p[DV + 1] = L; }
        }
    }

    if constexpr (CLUSTER) {
        // the row's splits form one thread-block cluster: after the barrier
        // every CTA reads the partial (max, sum, accumulator) of each head it
        // finishes straight from the peers' shared memory (heads hh with
        // hh % splits == its rank), merges them by log-sum-exp and writes
        // the gated output; a second barrier keeps every CTA's partial alive
        // until the peers are done reading it
        cluster_sync_all();
        const unsigned rank = cluster_rank();
        const int S = a.splits;
        for (int e = threadIdx.x; e < 16 * (DV / 2); e += GA_THREADS) {
            const int hh = e / (DV / 2), col = 2 * (e % (DV / 2)), h = hg * 16 + hh;
            if (h >= a.Hq || hh % S != (int)rank) continue;
            const float* lp = cpart + hh * (DV + 2);
            float M = -INFINITY;
            for (int q = 0; q < S; ++q) M = fmaxf(M, ld_cluster_f32(lp + DV, (unsigned)q));
            float L = 0.0f, O0 = 0.0f, O1 = 0.0f;
            if (M != -INFINITY) {
                for (int q = 0; q < S; ++q) {
                    const float mq = ld_cluster_f32(lp + DV, (unsigned)q);
                    if (mq == -INFINITY) continue;
                    const float f = exp2f(mq - M);
                    L = fmaf(ld_cluster_f32(lp + DV + 1, (unsigned)q), f, L);
                    const float2 ov = ld_cluster_f32x2(lp + col, (unsigned)q);
                    O0 = fmaf(ov.x, f, O0);
                    O1 = fmaf(ov.y, f, O1);
                }
            }
            const float gs = L > 0.0f ? gate_of(a, r, h) / L : 0.0f;
            *reinterpret_cast<uint32_t*>(static_cast<bf16*>(a.out) + ((int64_t)r * a.Hq + h) * DV + col) =
                pack_bf16x2(O0 * gs, O1 * gs);
        }
        cluster_sync_all();
    } else if (a.splits > 1) {
        const int groups = (a.Hq + 15) / 16;
        if (take_ticket(a.tickets + (int64_t)r * groups + hg, a.splits, &sh_flag)) {
            combine_splits<bf16>(a, r, hg * 16, min(a.Hq, hg * 16 + 16));
            if (threadIdx.x == 0) a.tickets[(int64_t)r * groups + hg] = 0u;
        }
    }
}

template <int DQK, int DV, int ST>
cudaError_t launch_ga_st(const AttnArgs& a, cudaStream_t s)
{
    using C = GaCfg<DQK, DV, ST>;
    dim3 grid(a.rows, a.splits, (a.Hq + 15) / 16);
    // split rows merge in a cluster of their splits when it is a portable
    // cluster size; else through the workspace and an atomic ticket
    const bool cluster = a.splits > 1 && a.splits <= GA_MAX_CLUSTER;
    auto kern = cluster ? attn_gather_kernel<DQK, DV, ST, true> : attn_gather_kernel<DQK, DV, ST, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
    }
    // (clusters are launched without programmatic dependent launch: clusters
    // placed early and parked at the dependency wait slowed the kernels they
    // were meant to overlap; measured 145.5 against 137.1 us per 128K step)
    if (cluster)
        return launch_kernel_cluster(kern, grid, dim3(GA_THREADS), (size_t)C::SMEM, s, false, dim3(1, a.splits, 1), a);
    return launch_kernel(kern, grid, dim3(GA_THREADS), (size_t)C::SMEM, s, a.pdl, a);
}

// Many CTAs (a CTA per query row, prefill): occupancy hides the gather
// latency best, so three CTAs per SM with two-stage rings. Few CTAs (split
// decode rows): deeper three-stage rings, two CTAs per SM. Both measured.
template <int DQK, int DV>
cudaError_t launch_ga(const AttnArgs& a, cudaStream_t s)
{
    const int64_t ctas = (int64_t)a.rows * a.splits * ((a.Hq + 15) / 16);
    if (ctas >= 4 * 148) return launch_ga_st<DQK, DV, 2>(a, s);
    return launch_ga_st<DQK, DV, 3>(a, s);
}

}  // namespace

bool attention_gather_supported(const AttnArgs& a)
{
    if (a.dtype != SA_BF16 || a.v_aliases_k) return false;
    if (!((a.dqk == 128 && a.dv == 128) || (a.dqk == 64 && a.dv == 64))) return false;
    if ((reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v)) & 15) return false;
    if (a.ld_k % 8 != 0 || a.ld_v % 8 != 0) return false;
    return a.splits <= MAX_SPLITS;
}

cudaError_t launch_attention_gather(const AttnArgs& a, cudaStream_t s)
{
    if (a.dqk == 128) return launch_ga<128, 128>(a, s);
    return launch_ga<64, 64>(a, s);
}

}  // namespace sa
