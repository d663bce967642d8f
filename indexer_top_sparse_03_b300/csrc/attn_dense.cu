// Dense causal attention with the sigmoid output gate: the full-attention
// control branch the sparse layer is measured against ("From Full Attention
// to Sparsity": sparse attention pays off once the indexer's cost is below
// the attention it saves; the break-even is a measurement of full attention
// minus sparse attention minus the indexer across lengths).
//
// One CTA per 8 consecutive query rows and group of 16 heads; warp w owns
// query t0 + w with its 16 heads as the M side of mma.sync m16n8k16 (the
// heads share the one KV head). The CTA streams the key/value rows 0 .. t0+7
// in 64-row tiles through a two-stage cp.async ring shared by its 8 warps;
// each warp runs the 16-row steps of a tile below its own causal limit: S =
// Q K^T, an fp32 online softmax in the exp2 domain, O += P V, and at the end
// the gate and a bf16 store of its own row. CTAs are issued from the last
// query rows down, so that the longest rows start first.
//
// With a kept-position list (rows t >= mask_from), each such warp first sets
// one bit per kept position of its query in a shared-memory bitmap; the
// logits of the other positions are -inf and 16-row steps without a kept
// position are skipped. That is exact attention over the kept set, and it is
// cheaper than gathering the rows one query at a time while the kept set is
// a large share of the history.
#include "attn_common.cuh"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int DN_W = 8;                    // warps = query rows per CTA
constexpr int DN_THREADS = 32 * DN_W;
constexpr int DN_TILE = 64;                // key rows per tile
constexpr int DN_STAGES = 2;

template <int D>
struct DnCfg {
    static constexpr int LDP = D + 8;                           // padded row (bf16 elements)
    static constexpr int TBYTES = DN_TILE * LDP * 2;            // one K (or V) tile
    static constexpr int STAGE = 2 * TBYTES;                    // K and V
    static constexpr int QBYTES = 16 * LDP * 2;                 // one warp's Q tile
    static constexpr int SMEM = DN_STAGES * STAGE + DN_W * QBYTES;    // + DN_W bitmaps when masked
};

__host__ __device__ __forceinline__ int64_t dense_mask_words(const DenseArgs& a) { return a.idx ? (a.L + 31) / 32 : 0; }

template <int D>
__global__ void __launch_bounds__(DN_THREADS, 2)
attn_dense_kernel(DenseArgs a)
{
    using C = DnCfg<D>;
    extern __shared__ __align__(128) uint8_t dn_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3, mat = lane >> 3, rr = lane & 7;
    const int64_t t0 = (int64_t)(gridDim.x - 1 - blockIdx.x) * DN_W;
    const int hg = blockIdx.z;
    const int64_t t = t0 + warp;                                  // this warp's query
    const int64_t t_last = min64(t0 + DN_W, a.L) - 1;
    const int ntiles = (int)((t_last + DN_TILE) / DN_TILE);
    const bf16* kp = static_cast<const bf16*>(a.k);
    const bf16* vp = static_cast<const bf16*>(a.v);

    // Q tiles (16 heads of each warp's query; rows past L or Hq are zero)
    bf16* Qs = reinterpret_cast<bf16*>(dn_smem + DN_STAGES * C::STAGE);
    {
        const bf16* q = static_cast<const bf16*>(a.q);
        for (int i = threadIdx.x; i < DN_W * 16 * (D / 8); i += DN_THREADS) {
            const int w = i / (16 * (D / 8)), rem = i % (16 * (D / 8));
            const int row = rem / (D / 8), pc = rem % (D / 8), h = hg * 16 + row;
            const int64_t tq = t0 + w;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < a.Hq && tq < a.L) v = *reinterpret_cast<const uint4*>(q + (tq * a.Hq + h) * D + pc * 8);
            *reinterpret_cast<uint4*>(Qs + (w * 16 + row) * C::LDP + pc * 8) = v;
        }
    }
    // one tile of K and V rows through cp.async (rows past t_last are not read)
    auto issue = [&](int kt) {
        if (kt < ntiles) {
            uint8_t* st = dn_smem + (kt % DN_STAGES) * C::STAGE;
            for (int i = threadIdx.x; i < DN_TILE * (D / 8) * 2; i += DN_THREADS) {
                const int isv = i >= DN_TILE * (D / 8);
                const int ii = isv ? i - DN_TILE * (D / 8) : i;
                const int row = ii / (D / 8), pc = ii % (D / 8);
                const int64_t j = (int64_t)kt * DN_TILE + row;
                const bool ok = j <= t_last;
                const bf16* src = isv ? vp + (ok ? j : 0) * a.ld_v + pc * 8 : kp + (ok ? j : 0) * a.ld_k + pc * 8;
                bf16* dst = reinterpret_cast<bf16*>(st + isv * C::TBYTES) + row * C::LDP + pc * 8;
                cp_async16(dst, src, ok);
            }
        }
        cp_async_commit();
    };

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const float sl2 = a.softmax_scale * LOG2E;
    const uint32_t qbase = smem_u32(Qs + warp * 16 * C::LDP);

    // kept-position bitmap of this warp's query (rows t >= mask_from)
    const bool masked = a.idx != nullptr && t >= a.mask_from && t < a.L;
    uint32_t* bm = reinterpret_cast<uint32_t*>(dn_smem + C::SMEM) + warp * dense_mask_words(a);
    if (masked) {
        const int words = (int)(t >> 5) + 1;
        for (int i = lane; i < words; i += 32) bm[i] = 0u;
        __syncwarp();
        const int32_t* sel = a.idx + t * a.K;
        for (int i = lane; i < a.K; i += 32) {
            const int32_t p = sel[i];
            if (p >= 0 && p <= t) atomicOr(&bm[p >> 5], 1u << (p & 31));
        }
        __syncwarp();
    }

    issue(0);
    for (int kt = 0; kt < ntiles; ++kt) {
        issue(kt + 1);
        cp_async_wait<1>();
        __syncthreads();                                          // tile kt (and the Q tiles) visible
        const uint32_t kst = smem_u32(dn_smem + (kt % DN_STAGES) * C::STAGE);
        const uint32_t vst = kst + C::TBYTES;
        for (int s16 = 0; s16 < DN_TILE / 16; ++s16) {
            const int64_t j0 = (int64_t)kt * DN_TILE + s16 * 16;
            if (j0 > t) break;                                    // warp-uniform: past this query
            uint32_t keep = 0xFFFFu;                              // kept rows of this step (bit i: j0 + i)
            if (masked) {
                keep = (bm[j0 >> 5] >> (j0 & 31)) & 0xFFFFu;
                if (keep == 0u) continue;                         // warp-uniform: nothing kept here
            }
            float sc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t af[4], bfm[4];
                ldsm_x4(af, qbase + (uint32_t)((((mat & 1) * 8 + rr) * C::LDP + ks * 16 + (mat >> 1) * 8) * 2));
                const int krow = s16 * 16 + (mat >> 1) * 8 + rr;
                const int dim = ks * 16 + (mat & 1) * 8;
                ldsm_x4(bfm, kst + (uint32_t)((krow * C::LDP + dim) * 2));
                mma_16816(sc[0], af, bfm[0], bfm[1]);
                mma_16816(sc[1], af, bfm[2], bfm[3]);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = nt * 8 + 2 * t4 + e;
                    const bool valid = j0 + c <= t && ((keep >> c) & 1u);
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
            if (mx0 > m0 || mx1 > m1) {
                const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
                const float a0 = (m0 == -INFINITY) ? 0.0f : exp2f(m0 - n0);
                const float a1 = (m1 == -INFINITY) ? 0.0f : exp2f(m1 - n1);
                m0 = n0; m1 = n1;
                l0 *= a0; l1 *= a1;
#pragma unroll
                for (int i = 0; i < D / 8; ++i) { o[i][0] *= a0; o[i][1] *= a0; o[i][2] *= a1; o[i][3] *= a1; }
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
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t bfm[4];
                const int vrow = s16 * 16 + (mat & 1) * 8 + rr;
                const int col = np * 16 + (mat >> 1) * 8;
                ldsm_x4_trans(bfm, vst + (uint32_t)((vrow * C::LDP + col) * 2));
                mma_16816(o[2 * np], pa, bfm[0], bfm[1]);
                mma_16816(o[2 * np + 1], pa, bfm[2], bfm[3]);
            }
        }
        __syncthreads();                                          // the stage is refilled next
    }
    cp_async_wait<0>();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (t >= a.L) return;
    bf16* out = static_cast<bf16*>(a.out);
    const int h0 = hg * 16 + g, h1 = h0 + 8;
    const float gs0 = (h0 < a.Hq && l0 > 0.0f) ? 1.0f / (1.0f + expf(-a.gate[t * a.Hq + h0])) / l0 : 0.0f;
    const float gs1 = (h1 < a.Hq && l1 > 0.0f) ? 1.0f / (1.0f + expf(-a.gate[t * a.Hq + h1])) / l1 : 0.0f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + 2 * t4;
        if (h0 < a.Hq)
            *reinterpret_cast<uint32_t*>(out + (t * a.Hq + h0) * D + col) = pack_bf16x2(o[i][0] * gs0, o[i][1] * gs0);
        if (h1 < a.Hq)
            *reinterpret_cast<uint32_t*>(out + (t * a.Hq + h1) * D + col) = pack_bf16x2(o[i][2] * gs1, o[i][3] * gs1);
    }
}

template <int D>
cudaError_t launch_dense_d(const DenseArgs& a, cudaStream_t s)
{
    const size_t smem = DnCfg<D>::SMEM + (size_t)DN_W * dense_mask_words(a) * 4;
    cudaError_t e = cudaFuncSetAttribute(attn_dense_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.L + DN_W - 1) / DN_W), 1, (unsigned)((a.Hq + 15) / 16));
    attn_dense_kernel<D><<<grid, DN_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool attention_dense_supported(const DenseArgs& a)
{
    const int64_t mask_bytes = (int64_t)DN_W * dense_mask_words(a) * 4;
    const int64_t base = a.D == 64 ? DnCfg<64>::SMEM : DnCfg<128>::SMEM;
    return (a.D == 64 || a.D == 128) && a.Hq >= 1 && a.Hq <= 64 && a.ld_k % 8 == 0 && a.ld_v % 8 == 0 &&
           (!a.idx || (a.K >= 1 && base + mask_bytes <= 200 * 1024));
}

cudaError_t launch_attention_dense(const DenseArgs& a, cudaStream_t s)
{
    if (a.L <= 0) return cudaSuccess;
    if (attention_dense_tc_supported(a)) {
        const cudaError_t e = launch_attention_dense_tc(a, s);
        if (e != cudaErrorNotSupported) return e;
    }
    return a.D == 64 ? launch_dense_d<64>(a, s) : launch_dense_d<128>(a, s);
}

}  // namespace sa
