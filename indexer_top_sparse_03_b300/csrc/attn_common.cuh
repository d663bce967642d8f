// Pieces shared by the attention kernels: row lengths and bases, the sigmoid
// gate, the atomic ticket that elects the last CTA of a split row, and the
// log-sum-exp merge of split partials.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace sa {

constexpr float LOG2E = 1.4426950408889634f;

SA_DEVINL int64_t attn_hist_len(const AttnArgs& a, int r)
{
    int64_t n = a.ctx_len ? (int64_t)a.ctx_len[r] : a.causal_first + r + 1;
    return n < 0 ? 0 : (n > a.n_cap ? a.n_cap : n);
}

SA_DEVINL int64_t attn_base(const AttnArgs& a, int r) { return a.row_base ? a.row_base[r] : 0; }

// entries of idx row r that hold kept positions (all at the front)
SA_DEVINL int attn_kept(const AttnArgs& a, int r, int64_t n)
{
    const int64_t k = a.kept_len ? (int64_t)a.kept_len[r] : n;
    return (int)min64(a.K, k < 0 ? 0 : (k > n ? n : k));
}

SA_DEVINL float gate_of(const AttnArgs& a, int r, int h)
{
    const float x = a.gate[(int64_t)r * a.Hq + h];
    return 1.0f / (1.0f + expf(-x));
}

template <typename T> SA_DEVINL void store_out(T* p, float v);
template <> SA_DEVINL void store_out<float>(float* p, float v) { *p = v; }
template <> SA_DEVINL void store_out<bf16>(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// Merge the split partials of heads [h0, h1) of row r (whole CTA). Each
// thread takes four consecutive columns of one head and loads, for up to 8
// splits at a time and all at once, the splits' (max, sum) pairs and their
// accumulators; the weights 2^(m_s - M) / L follow locally, so the merge costs
// one round of independent loads.
constexpr int MAX_SPLITS = 64;

template <typename T>
__device__ void combine_splits(const AttnArgs& a, int r, int h0, int h1)
{
    const int dv = a.dv, S = a.splits;
    const int64_t stride = (int64_t)a.Hq * (dv + 2);
    const float* base = a.part + (int64_t)r * S * stride;
    for (int e = threadIdx.x * 4; e < (h1 - h0) * dv; e += blockDim.x * 4) {
        const int hh = e / dv, col = e % dv, h = h0 + hh;
        const float* p = base + (int64_t)h * (dv + 2);
        float M = -INFINITY, L = 0.0f;
        float O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int s0 = 0; s0 < S; s0 += 8) {
            float2 ml[8], x[8][2];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (s0 + u < S) {
                    const float* ps = p + (s0 + u) * stride;
                    ml[u] = __ldcg(reinterpret_cast<const float2*>(ps + dv));
                    x[u][0] = __ldcg(reinterpret_cast<const float2*>(ps + col));
                    x[u][1] = __ldcg(reinterpret_cast<const float2*>(ps + col + 2));
                }
            }
            float Mb = M;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (s0 + u < S) Mb = fmaxf(Mb, ml[u].x);
            if (Mb == -INFINITY) continue;                          // nothing kept yet
            const float f_old = (M == -INFINITY) ? 0.0f : exp2f(M - Mb);
            L *= f_old;
            O[0] *= f_old; O[1] *= f_old; O[2] *= f_old; O[3] *= f_old;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (s0 + u < S && ml[u].x != -INFINITY) {
                    const float f = exp2f(ml[u].x - Mb);
                    L = fmaf(ml[u].y, f, L);
                    O[0] = fmaf(f, x[u][0].x, O[0]); O[1] = fmaf(f, x[u][0].y, O[1]);
                    O[2] = fmaf(f, x[u][1].x, O[2]); O[3] = fmaf(f, x[u][1].y, O[3]);
                }
            }
            M = Mb;
        }
        const float gs = L > 0.0f ? gate_of(a, r, h) / L : 0.0f;
        T* o = static_cast<T*>(a.out) + ((int64_t)r * a.Hq + h) * dv + col;
#pragma unroll
        for (int i = 0; i < 4; ++i) store_out<T>(o + i, gs * O[i]);
    }
}

// Ticket: returns true in every thread of the CTA that finished row r's group last.
// Thread-block cluster helpers: rank in the cluster, a full cluster barrier
// (release / acquire: shared-memory writes before it are visible to every
// peer after it), and loads of a peer CTA's shared memory at the address the
// same variable has in this CTA.
SA_DEVINL unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
SA_DEVINL void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
SA_DEVINL uint32_t cluster_map(const void* p, unsigned rank)
{
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_u32(p)), "r"(rank));
    return d;
}
SA_DEVINL float ld_cluster_f32(const float* p, unsigned rank)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_map(p, rank)) : "memory");
    return v;
}
SA_DEVINL float2 ld_cluster_f32x2(const float* p, unsigned rank)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(cluster_map(p, rank)) : "memory");
    return v;
}

SA_DEVINL bool take_ticket(unsigned* ticket, int splits, int* sh_flag)
{
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(ticket, 1u);
        *sh_flag = (prev == (unsigned)splits - 1u);
    }
    __syncthreads();
    const bool last = *sh_flag != 0;
    if (last) __threadfence();
    return last;
}

}  // namespace sa
