// Gradients of the gated attention over a fixed index set on the tensor
// cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation) for bf16
// inputs with heads of width 64 or 128 (the training path: "Hybrid Attention
// Architectures...", section 3.1, the selected set is fixed once chosen;
// section 3.3, the gate scales the output).
//
// One CTA per query row t, its 16 heads as the M side; four warps, warp w
// taking the 16-row steps w, w + 4, ... of the kept rows through its own
// cp.async ring of K and V rows (as the forward does). Two passes:
//   pass 1  S = Q K^T and dP' = dout V^T per step; an online max m, sum l
//           and sum of exp(s - m) dP' per head give, after merging the four
//           warps, lse and D = g * (dout . o) without forming o;
//   pass 2  p = exp(s - lse), ds = p (g dP' - D); dq += ds K; the step's
//           dk = ds^T q and dv = (g p)^T dout are staged in shared memory and
//           added to the key / value rows with 16-byte fp32 atomics.
// S and dP' multiply exact bf16 inputs. The fp32 operands ds and g p are
// split into a bf16 head and a bf16 remainder (two MMAs), which keeps about
// 16 significant bits: the gradients stay within fp32-accumulation error of
// the exact ones.
#include "attn_common.cuh"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int TB_W = 4;
constexpr int TB_THREADS = 32 * TB_W;
constexpr int TB_ROWS = 16;
constexpr int TB_STAGES = 2;

template <int D>
struct TbCfg {
    static constexpr int LDP = D + 8;                        // padded bf16 row
    static constexpr int KB = TB_ROWS * LDP * 2;             // K rows of one step
    static constexpr int WSTAGE = 2 * KB;                    // K and V
    static constexpr int WRING = TB_STAGES * WSTAGE;
    static constexpr int TLD = 24;                           // transpose tile row (bf16)
    static constexpr int TBYTES = 2 * 16 * TLD * 2;          // hi and lo tiles
    static constexpr int SLD = D / 2 + 4;                    // staging row (fp32), half the columns
    static constexpr int SBYTES = 16 * SLD * 4;
    static constexpr int WPRIV = WRING + TBYTES + SBYTES;    // one warp's private space
    static constexpr int OFF_Q = TB_W * WPRIV;
    static constexpr int OFF_DO = OFF_Q + 16 * LDP * 2;
    static constexpr int SMEM = OFF_DO + 16 * LDP * 2;
    static constexpr int PK = D / 8;                         // 16-byte pieces of a row
    static constexpr int RPI = 32 / (2 * PK);                // rows per copy instruction (K and V)
    static_assert(2 * PK == 32 || 2 * PK == 16, "one or two rows per warp instruction");
    static_assert(TB_W * 16 * D * 4 <= OFF_Q, "dq merge scratch fits the private spaces");
};

SA_DEVINL uint32_t bf16_hi_lo(float x, float& rem)
{
    const bf16 h = __float2bfloat16_rn(x);
    rem = x - __bfloat162float(h);
    return (uint32_t)__bfloat16_as_ushort(h);
}

template <int D>
__global__ void __launch_bounds__(TB_THREADS, 2)
attn_bwd_tc_kernel(BwdArgs a)
{
    using C = TbCfg<D>;
    extern __shared__ __align__(128) uint8_t tb_smem[];
    __shared__ float st_m[TB_W][16], st_l[TB_W][16], st_d[TB_W][16];
    __shared__ float lse2_s[16], D_s[16], g_s[16];
    __shared__ int jrow[TB_W][TB_ROWS];

    const int r = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3, mat = lane >> 3, rr = lane & 7;
    const int Hq = a.Hq;
    const int32_t* sel = a.idx + (int64_t)r * a.K;
    int n_sel = 0;                                           // kept entries sit at the front
    for (int i = 0; i < a.K; ++i) {
        if (sel[i] < 0) break;
        ++n_sel;
    }
    const int nsteps = (n_sel + TB_ROWS - 1) / TB_ROWS;
    const int my_steps = nsteps > warp ? (nsteps - warp + TB_W - 1) / TB_W : 0;
    const int fallback = n_sel > 0 ? sel[0] : 0;

    bf16* Qs = reinterpret_cast<bf16*>(tb_smem + C::OFF_Q);
    bf16* Os = reinterpret_cast<bf16*>(tb_smem + C::OFF_DO);     // dout tile
    {
        const bf16* q = static_cast<const bf16*>(a.q);
        const bf16* dout = static_cast<const bf16*>(a.dout);
        for (int i = threadIdx.x; i < 16 * (D / 8); i += TB_THREADS) {
            const int row = i / (D / 8), pc = i % (D / 8);
            uint4 vq = make_uint4(0, 0, 0, 0), vo = vq;
            if (row < Hq) {
                vq = *reinterpret_cast<const uint4*>(q + ((int64_t)r * Hq + row) * D + pc * 8);
                vo = *reinterpret_cast<const uint4*>(dout + ((int64_t)r * Hq + row) * D + pc * 8);
            }
            *reinterpret_cast<uint4*>(Qs + row * C::LDP + pc * 8) = vq;
            *reinterpret_cast<uint4*>(Os + row * C::LDP + pc * 8) = vo;
        }
        if (threadIdx.x < 16) {
            const int h = threadIdx.x;
            g_s[h] = h < Hq ? 1.0f / (1.0f + __expf(-a.gate[(int64_t)r * Hq + h])) : 0.0f;
        }
    }

    uint8_t* priv = tb_smem + warp * C::WPRIV;
    uint8_t* ring = priv;
    bf16* tt = reinterpret_cast<bf16*>(priv + C::WRING);              // [2][16][TLD]: hi, lo
    float* stg = reinterpret_cast<float*>(priv + C::WRING + C::TBYTES); // [16][SLD]
    const int piece = lane % (2 * C::PK), sub = lane / (2 * C::PK);
    const bool is_k = piece < C::PK;
    const bf16* src_base = is_k ? static_cast<const bf16*>(a.k) + piece * 8
                                : static_cast<const bf16*>(a.v) + (piece - C::PK) * 8;
    const int64_t src_ld = is_k ? a.ld_k : a.ld_v;
    const int dst_off = is_k ? piece * 8 : C::KB / 2 + (piece - C::PK) * 8;
    auto load_pos = [&](int k) -> int {
        int pos = fallback;
        if (k < my_steps && lane < TB_ROWS) {
            const int slot = (warp + k * TB_W) * TB_ROWS + lane;
            pos = slot < n_sel ? sel[slot] : fallback;
            if (pos < 0 || pos >= a.L) pos = fallback;
        }
        return pos;
    };
    auto issue = [&](int k, int pos) {
        if (k < my_steps) {
            bf16* dst = reinterpret_cast<bf16*>(ring + (k % TB_STAGES) * C::WSTAGE) + dst_off;
#pragma unroll
            for (int r0 = 0; r0 < TB_ROWS; r0 += C::RPI) {
                const int rrow = r0 + sub;
                const int64_t gr = __shfl_sync(0xffffffffu, (int64_t)pos, rrow);
                cp_async16(dst + rrow * C::LDP, src_base + gr * src_ld, true);
            }
        }
        cp_async_commit();
    };
    const uint32_t qbase = smem_u32(Qs), obase = smem_u32(Os);
    const float sl2 = a.softmax_scale * LOG2E;

    // S = Q K^T and dP' = dout V^T for the 16 rows of the step in stage st
    auto scores = [&](uint32_t st, float (&sc)[2][4], float (&dp)[2][4]) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) { sc[nt][e] = 0.0f; dp[nt][e] = 0.0f; }
        const uint32_t vst = st + C::KB;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t af[4], ao[4], bk[4], bv[4];
            const uint32_t aoff = (uint32_t)((((mat & 1) * 8 + rr) * C::LDP + ks * 16 + (mat >> 1) * 8) * 2);
            ldsm_x4(af, qbase + aoff);
            ldsm_x4(ao, obase + aoff);
            const uint32_t boff = (uint32_t)((((mat >> 1) * 8 + rr) * C::LDP + ks * 16 + (mat & 1) * 8) * 2);
            ldsm_x4(bk, st + boff);
            ldsm_x4(bv, vst + boff);
            mma_16816(sc[0], af, bk[0], bk[1]);
            mma_16816(sc[1], af, bk[2], bk[3]);
            mma_16816(dp[0], ao, bv[0], bv[1]);
            mma_16816(dp[1], ao, bv[2], bv[3]);
        }
    };

    // ---------------- pass 1: softmax statistics and D ----------------
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f, d0 = 0.0f, d1 = 0.0f;
    {
        int pos_next = load_pos(0);
        for (int k = 0; k < TB_STAGES - 1; ++k) {
            const int pos = pos_next;
            pos_next = load_pos(k + 1);
            issue(k, pos);
        }
        __syncthreads();                                      // Q and dout tiles
        for (int k = 0; k < my_steps; ++k) {
            {
                const int pos = pos_next;
                pos_next = load_pos(k + TB_STAGES);
                issue(k + TB_STAGES - 1, pos);
            }
            cp_async_wait<TB_STAGES - 1>();
            __syncwarp();
            const uint32_t st = smem_u32(ring + (k % TB_STAGES) * C::WSTAGE);
            const int slot0 = (warp + k * TB_W) * TB_ROWS;
            float sc[2][4], dp[2][4];
            scores(st, sc, dp);
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool valid = slot0 + nt * 8 + 2 * t4 + e < n_sel;
                    sc[nt][e] = valid ? sc[nt][e] * sl2 : -INFINITY;
                    sc[nt][2 + e] = valid ? sc[nt][2 + e] * sl2 : -INFINITY;
                    mx0 = fmaxf(mx0, sc[nt][e]);
                    mx1 = fmaxf(mx1, sc[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float a0 = (m0 == -INFINITY) ? 0.0f : exp2f(m0 - n0);
            const float a1 = (m1 == -INFINITY) ? 0.0f : exp2f(m1 - n1);
            m0 = n0; m1 = n1;
            l0 *= a0; l1 *= a1; d0 *= a0; d1 *= a1;
            const float ref0 = (m0 == -INFINITY) ? 0.0f : m0, ref1 = (m1 == -INFINITY) ? 0.0f : m1;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float p0 = exp2f(sc[nt][e] - ref0), p1 = exp2f(sc[nt][2 + e] - ref1);
                    l0 += p0; l1 += p1;
                    d0 = fmaf(p0, dp[nt][e], d0);
                    d1 = fmaf(p1, dp[nt][2 + e], d1);
                }
            __syncwarp();
        }
        cp_async_wait<0>();
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
        d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
        d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
        d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
        if (t4 == 0) {
            st_m[warp][g] = m0; st_m[warp][g + 8] = m1;
            st_l[warp][g] = l0; st_l[warp][g + 8] = l1;
            st_d[warp][g] = d0; st_d[warp][g + 8] = d1;
        }
        __syncthreads();
        if (threadIdx.x < 16) {
            const int h = threadIdx.x;
            float M = -INFINITY;
            for (int w = 0; w < TB_W; ++w) M = fmaxf(M, st_m[w][h]);
            float L = 0.0f, S = 0.0f;
            if (M != -INFINITY) {
                for (int w = 0; w < TB_W; ++w) {
                    const float f = st_m[w][h] == -INFINITY ? 0.0f : exp2f(st_m[w][h] - M);
                    L = fmaf(st_l[w][h], f, L);
                    S = fmaf(st_d[w][h], f, S);
                }
            }
            const float gh = g_s[h];
            const float dsum = L > 0.0f ? S / L : 0.0f;                 // dout . o
            lse2_s[h] = L > 0.0f ? M + __log2f(L) : 0.0f;
            D_s[h] = gh * dsum;
            if (h < Hq) a.dgate[(int64_t)r * Hq + h] = gh * (1.0f - gh) * dsum;
        }
        __syncthreads();
    }

    // ---------------- pass 2: gradients ----------------
    float dq[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.0f;
    const float lse0 = lse2_s[g], lse1 = lse2_s[g + 8], D0 = D_s[g], D1 = D_s[g + 8];
    const float gg0 = g_s[g], gg1 = g_s[g + 8];
    bf16* thi = tt;
    bf16* tlo = tt + 16 * C::TLD;
    {
        int pos_next = load_pos(0);
        for (int k = 0; k < TB_STAGES - 1; ++k) {
            const int pos = pos_next;
            pos_next = load_pos(k + 1);
            issue(k, pos);
        }
        for (int k = 0; k < my_steps; ++k) {
            int pos_cur;
            {
                const int pos = pos_next;
                pos_next = load_pos(k + TB_STAGES);
                issue(k + TB_STAGES - 1, pos);
            }
            pos_cur = load_pos(k);
            cp_async_wait<TB_STAGES - 1>();
            __syncwarp();
            const uint32_t st = smem_u32(ring + (k % TB_STAGES) * C::WSTAGE);
            const uint32_t vst = st + C::KB;
            const int slot0 = (warp + k * TB_W) * TB_ROWS;
            if (lane < TB_ROWS) jrow[warp][lane] = slot0 + lane < n_sel ? pos_cur : -1;
            float sc[2][4], dp[2][4];
            scores(st, sc, dp);
            // p, ds (rows: heads g and g + 8; columns: the step's keys)
            float ds[2][4], pg[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool valid = slot0 + nt * 8 + 2 * t4 + e < n_sel;
                    const float p0 = valid ? exp2f(sc[nt][e] * sl2 - lse0) : 0.0f;
                    const float p1 = valid ? exp2f(sc[nt][2 + e] * sl2 - lse1) : 0.0f;
                    ds[nt][e] = p0 * (gg0 * dp[nt][e] - D0);
                    ds[nt][2 + e] = p1 * (gg1 * dp[nt][2 + e] - D1);
                    pg[nt][e] = p0 * gg0;
                    pg[nt][2 + e] = p1 * gg1;
                }
            // A fragments of ds (head and remainder) for dq += ds K
            uint32_t ah[4], al[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float r0, r1, r2, r3;
                const uint32_t h0 = bf16_hi_lo(ds[nt][0], r0), h1 = bf16_hi_lo(ds[nt][1], r1);
                const uint32_t h2 = bf16_hi_lo(ds[nt][2], r2), h3 = bf16_hi_lo(ds[nt][3], r3);
                ah[2 * nt] = h0 | (h1 << 16);
                ah[2 * nt + 1] = h2 | (h3 << 16);
                al[2 * nt] = pack_bf16x2(r0, r1);
                al[2 * nt + 1] = pack_bf16x2(r2, r3);
            }
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t bfm[4];
                const int krow = (mat & 1) * 8 + rr;
                const int col = np * 16 + (mat >> 1) * 8;
                ldsm_x4_trans(bfm, st + (uint32_t)((krow * C::LDP + col) * 2));
                mma_16816(dq[2 * np], ah, bfm[0], bfm[1]);
                mma_16816(dq[2 * np + 1], ah, bfm[2], bfm[3]);
                mma_16816(dq[2 * np], al, bfm[0], bfm[1]);
                mma_16816(dq[2 * np + 1], al, bfm[2], bfm[3]);
            }
            // dk = ds^T q and dv = (g p)^T dout: the transposed A operands go
            // through the warp's tile (head rows, key columns)
            for (int which = 0; which < 2; ++which) {
                const float (&x)[2][4] = which == 0 ? ds : pg;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float r0, r1, r2, r3;
                    const uint32_t h0 = bf16_hi_lo(x[nt][0], r0), h1 = bf16_hi_lo(x[nt][1], r1);
                    const uint32_t h2 = bf16_hi_lo(x[nt][2], r2), h3 = bf16_hi_lo(x[nt][3], r3);
                    const int col = nt * 8 + 2 * t4;
                    *reinterpret_cast<uint32_t*>(thi + g * C::TLD + col) = h0 | (h1 << 16);
                    *reinterpret_cast<uint32_t*>(thi + (g + 8) * C::TLD + col) = h2 | (h3 << 16);
                    *reinterpret_cast<uint32_t*>(tlo + g * C::TLD + col) = pack_bf16x2(r0, r1);
                    *reinterpret_cast<uint32_t*>(tlo + (g + 8) * C::TLD + col) = pack_bf16x2(r2, r3);
                }
                __syncwarp();
                // A = tile^T: matrix mi of the x4 load covers keys (mi & 1) * 8, heads (mi >> 1) * 8
                uint32_t th[4], tl[4];
                {
                    const int trow = (mat >> 1) * 8 + rr, tcol = (mat & 1) * 8;
                    ldsm_x4_trans(th, smem_u32(thi + trow * C::TLD + tcol));
                    ldsm_x4_trans(tl, smem_u32(tlo + trow * C::TLD + tcol));
                }
                const uint32_t bbase = which == 0 ? qbase : obase;
                float* dst = which == 0 ? a.dk : a.dv;
                const float fs = which == 0 ? a.softmax_scale : 1.0f;
                for (int half = 0; half < 2; ++half) {
                    float c[D / 16][4];
#pragma unroll
                    for (int i = 0; i < D / 16; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.0f;
#pragma unroll
                    for (int np = 0; np < D / 32; ++np) {
                        uint32_t bfm[4];
                        const int hrow = (mat & 1) * 8 + rr;
                        const int col = half * (D / 2) + np * 16 + (mat >> 1) * 8;
                        ldsm_x4_trans(bfm, bbase + (uint32_t)((hrow * C::LDP + col) * 2));
                        mma_16816(c[2 * np], th, bfm[0], bfm[1]);
                        mma_16816(c[2 * np + 1], th, bfm[2], bfm[3]);
                        mma_16816(c[2 * np], tl, bfm[0], bfm[1]);
                        mma_16816(c[2 * np + 1], tl, bfm[2], bfm[3]);
                    }
#pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        const int col = i * 8 + 2 * t4;
                        *reinterpret_cast<float2*>(stg + g * C::SLD + col) = make_float2(c[i][0] * fs, c[i][1] * fs);
                        *reinterpret_cast<float2*>(stg + (g + 8) * C::SLD + col) = make_float2(c[i][2] * fs, c[i][3] * fs);
                    }
                    __syncwarp();
                    // one staged row per (4-column piece, lane) group: 16-byte atomics along rows
                    for (int x4 = lane; x4 < 16 * (D / 8); x4 += 32) {
                        const int row = x4 / (D / 8), c4 = (x4 % (D / 8)) * 4;
                        const int j = jrow[warp][row];
                        if (j >= 0)
                            atomicAdd(reinterpret_cast<float4*>(dst + (int64_t)j * D + half * (D / 2) + c4),
                                      *reinterpret_cast<const float4*>(stg + row * C::SLD + c4));
                    }
                    __syncwarp();
                }
            }
            __syncwarp();                                         // the stage is refilled next
        }
        cp_async_wait<0>();
    }

    // merge the four warps' dq (the private spaces are free now)
    __syncthreads();
    float* dqw = reinterpret_cast<float*>(tb_smem);                  // [4][16][D]
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + 2 * t4;
        *reinterpret_cast<float2*>(&dqw[(warp * 16 + g) * D + col]) = make_float2(dq[i][0], dq[i][1]);
        *reinterpret_cast<float2*>(&dqw[(warp * 16 + g + 8) * D + col]) = make_float2(dq[i][2], dq[i][3]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < Hq * D; e += TB_THREADS) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < TB_W; ++w) s += dqw[w * 16 * D + e];
        a.dq[(int64_t)r * Hq * D + e] = s * a.softmax_scale;
    }
}

}  // namespace

bool attention_backward_tc_supported(const BwdArgs& a)
{
    return a.dtype == SA_BF16 && (a.D == 64 || a.D == 128) && a.Hq >= 1 && a.Hq <= 16 && a.ld_k % 8 == 0 &&
           a.ld_v % 8 == 0;
}

cudaError_t launch_attention_backward_tc(const BwdArgs& a, cudaStream_t s)
{
    const int smem = a.D == 64 ? TbCfg<64>::SMEM : TbCfg<128>::SMEM;
    cudaError_t e = a.D == 64
        ? cudaFuncSetAttribute(attn_bwd_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
        : cudaFuncSetAttribute(attn_bwd_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (a.D == 64) attn_bwd_tc_kernel<64><<<a.L, TB_THREADS, smem, s>>>(a);
    else attn_bwd_tc_kernel<128><<<a.L, TB_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sa
