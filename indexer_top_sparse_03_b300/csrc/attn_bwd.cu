// Gradients of the gated attention over a fixed index set: the training path
// of the layer ("Hybrid Attention Architectures...", section 3.1: once the
// indexer has chosen the set, attention over it is ordinary softmax
// attention; section 3.3: the gate scales its output).
//
// One CTA per query row t (MQA: its Hq heads share every selected key and
// value row), 256 threads, the kept rows in chunks of 32:
//   pass 1  the forward again (online softmax) -> o_h, the log-sum-exp per
//           head, D_h = do_h . o_h with do_h = g_h dout_h, and dgate_h =
//           (1 - g_h) D_h;
//   pass 2  per chunk: p = exp(l - lse), dp = do . v, ds = p (dp - D);
//           dq += scale ds k (registers), and the chunk's dk = scale ds^T q
//           and dv = p^T do go to the key / value rows with fp32 vector
//           atomics (a row is shared by every query that selected it).
// fp32 arithmetic throughout on CUDA cores; inputs are converted once per
// chunk into shared memory, and every product loop is register-blocked over
// 16-byte shared-memory loads.
#include "common.cuh"
#include "kernels.h"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int BW_THREADS = 256;
constexpr int BW_CH = 32;                  // kept rows per chunk (one per lane in the softmax)
constexpr int BW_MAX_HQ = 16;

template <int D>
struct BwCfg {
    static constexpr int LD = D + 4;                       // padded row of the chunk tiles (16-byte aligned)
    static constexpr int TPH = D / 8;                      // dq: threads per head, 8 columns each
    static size_t smem(int Hq)
    {
        return sizeof(float) * ((size_t)3 * Hq * D + 2 * (size_t)BW_CH * LD + 2 * (size_t)Hq * (BW_CH + 1) + 6 * Hq);
    }
};

template <typename T>
SA_DEVINL float ld_elem(const T* p) { return to_f32(*p); }

// 8 consecutive elements as floats (16-byte aligned source for bf16, 32 for fp32)
SA_DEVINL void load8(const bf16* p, float* o)
{
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    float2 f;
    f = bf16x2_to_f32x2(u.x); o[0] = f.x; o[1] = f.y;
    f = bf16x2_to_f32x2(u.y); o[2] = f.x; o[3] = f.y;
    f = bf16x2_to_f32x2(u.z); o[4] = f.x; o[5] = f.y;
    f = bf16x2_to_f32x2(u.w); o[6] = f.x; o[7] = f.y;
}
SA_DEVINL void load8(const float* p, float* o)
{
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

SA_DEVINL float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
SA_DEVINL float dot4(float4 a, float4 b, float s)
{
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, s))));
}

template <int D, typename T>
__global__ void __launch_bounds__(BW_THREADS, 3)
attn_bwd_kernel(BwdArgs a)
{
    using C = BwCfg<D>;
    extern __shared__ __align__(16) float bw_smem[];
    const int Hq = a.Hq;
    float* qs = bw_smem;                        // [Hq][D]
    float* dos = qs + Hq * D;                   // [Hq][D]  do = g * dout
    float* dos_raw = dos + Hq * D;              // [Hq][D]  dout (for dgate)
    float* ks = dos_raw + Hq * D;               // [BW_CH][LD]
    float* vs = ks + BW_CH * C::LD;             // [BW_CH][LD]
    float* ps = vs + BW_CH * C::LD;             // [Hq][BW_CH + 1]
    float* dss = ps + Hq * (BW_CH + 1);         // [Hq][BW_CH + 1]
    float* st = dss + Hq * (BW_CH + 1);         // per head: m, l, alpha, lse, Dsum, dout.o
    float* m_s = st, *l_s = st + Hq, *al_s = st + 2 * Hq, *lse_s = st + 3 * Hq, *D_s = st + 4 * Hq,
         *dto_s = st + 5 * Hq;
    __shared__ int jrow[BW_CH];

    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T* q = static_cast<const T*>(a.q);
    const T* kk = static_cast<const T*>(a.k);
    const T* vv = static_cast<const T*>(a.v);
    const T* dout = static_cast<const T*>(a.dout);
    const int32_t* sel = a.idx + (int64_t)t * a.K;

    for (int i = tid; i < Hq * D; i += BW_THREADS) {
        const int h = i / D;
        const float g = 1.0f / (1.0f + __expf(-a.gate[(int64_t)t * Hq + h]));
        qs[i] = ld_elem(q + (int64_t)t * Hq * D + i);
        const float dt = ld_elem(dout + (int64_t)t * Hq * D + i);
        dos_raw[i] = dt;
        dos[i] = g * dt;
    }
    for (int h = tid; h < Hq; h += BW_THREADS) {
        m_s[h] = -INFINITY; l_s[h] = 0.0f; D_s[h] = 0.0f; dto_s[h] = 0.0f;
    }

    // pass 1 output of this thread: head oh, columns od0 .. od0 + 7
    const int oh = tid / C::TPH, od0 = (tid % C::TPH) * 8;
    float oa[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) oa[u] = 0.0f;

    // chunk loader: rows of k and v for kept entries c0 .. c0 + BW_CH - 1
    auto load_chunk = [&](int c0) {
        if (tid < BW_CH) {
            const int i = c0 + tid;
            const int j = i < a.K ? sel[i] : -1;
            jrow[tid] = (j >= 0 && j < a.L) ? j : -1;
        }
        __syncthreads();
        for (int x = tid; x < BW_CH * (D / 8); x += BW_THREADS) {
            const int c = x / (D / 8), d0 = (x % (D / 8)) * 8;
            const int j = jrow[c];
            float kv[8], vw[8];
            if (j >= 0) {
                load8(kk + (int64_t)j * a.ld_k + d0, kv);
                load8(vv + (int64_t)j * a.ld_v + d0, vw);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) { kv[u] = 0.0f; vw[u] = 0.0f; }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) { ks[c * C::LD + d0 + u] = kv[u]; vs[c * C::LD + d0 + u] = vw[u]; }
        }
        __syncthreads();
    };

    // ---------------- pass 1: the forward, online softmax ----------------
    for (int c0 = 0; c0 < a.K; c0 += BW_CH) {
        load_chunk(c0);
        for (int p = tid; p < Hq * (BW_CH / 2); p += BW_THREADS) {   // rows c and c + 16 of head h
            const int h = p / (BW_CH / 2), c = p % (BW_CH / 2);
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll 4
            for (int d = 0; d < D; d += 4) {
                const float4 qv = lds4(qs + h * D + d);
                s0 = dot4(qv, lds4(ks + c * C::LD + d), s0);
                s1 = dot4(qv, lds4(ks + (c + 16) * C::LD + d), s1);
            }
            ps[h * (BW_CH + 1) + c] = jrow[c] >= 0 ? s0 * a.softmax_scale : -INFINITY;
            ps[h * (BW_CH + 1) + c + 16] = jrow[c + 16] >= 0 ? s1 * a.softmax_scale : -INFINITY;
        }
        __syncthreads();
        for (int h = warp; h < Hq; h += BW_THREADS / 32) {        // one warp per head, lane = row
            const float s = ps[h * (BW_CH + 1) + lane];
            float mc = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, o));
            const float m_old = m_s[h];
            const float m_new = fmaxf(m_old, mc);
            const float e = m_new == -INFINITY ? 0.0f : __expf(s - m_new);
            float se = e;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xFFFFFFFFu, se, o);
            ps[h * (BW_CH + 1) + lane] = e;
            __syncwarp();
            if (lane == 0) {
                const float alpha = m_old == -INFINITY ? 0.0f : __expf(m_old - m_new);
                l_s[h] = l_s[h] * alpha + se;
                m_s[h] = m_new;
                al_s[h] = alpha;
            }
        }
        __syncthreads();
        // o = o * alpha + p v: this thread's head and 8 consecutive columns
        if (oh < Hq) {
            const float al = al_s[oh];
#pragma unroll
            for (int u = 0; u < 8; ++u) oa[u] *= al;
#pragma unroll 4
            for (int c = 0; c < BW_CH; ++c) {
                const float w = ps[oh * (BW_CH + 1) + c];
                const float4 v0 = lds4(vs + c * C::LD + od0), v1 = lds4(vs + c * C::LD + od0 + 4);
                oa[0] = fmaf(w, v0.x, oa[0]); oa[1] = fmaf(w, v0.y, oa[1]);
                oa[2] = fmaf(w, v0.z, oa[2]); oa[3] = fmaf(w, v0.w, oa[3]);
                oa[4] = fmaf(w, v1.x, oa[4]); oa[5] = fmaf(w, v1.y, oa[5]);
                oa[6] = fmaf(w, v1.z, oa[6]); oa[7] = fmaf(w, v1.w, oa[7]);
            }
        }
        __syncthreads();
    }
    // o = oa / l; D_h = do . o; dout . o for the gate
    if (oh < Hq) {
        const float il = l_s[oh] > 0.0f ? 1.0f / l_s[oh] : 0.0f;
        float dsum = 0.0f, tsum = 0.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float o = oa[u] * il;
            dsum = fmaf(dos[oh * D + od0 + u], o, dsum);
            tsum = fmaf(dos_raw[oh * D + od0 + u], o, tsum);
        }
        atomicAdd(&D_s[oh], dsum);
        atomicAdd(&dto_s[oh], tsum);
    }
    float dqa[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) dqa[u] = 0.0f;
    __syncthreads();
    for (int h = tid; h < Hq; h += BW_THREADS) {
        lse_s[h] = m_s[h] == -INFINITY ? 0.0f : m_s[h] + __logf(l_s[h]);
        const float g = 1.0f / (1.0f + __expf(-a.gate[(int64_t)t * Hq + h]));
        a.dgate[(int64_t)t * Hq + h] = g * (1.0f - g) * dto_s[h];
    }
    __syncthreads();

    // ---------------- pass 2: gradients ----------------
    for (int c0 = 0; c0 < a.K; c0 += BW_CH) {
        load_chunk(c0);
        for (int p = tid; p < Hq * (BW_CH / 2); p += BW_THREADS) {   // rows c and c + 16 of head h
            const int h = p / (BW_CH / 2), c = p % (BW_CH / 2);
            float s0 = 0.0f, s1 = 0.0f, dp0 = 0.0f, dp1 = 0.0f;
#pragma unroll 4
            for (int d = 0; d < D; d += 4) {
                const float4 qv = lds4(qs + h * D + d), dv4 = lds4(dos + h * D + d);
                s0 = dot4(qv, lds4(ks + c * C::LD + d), s0);
                s1 = dot4(qv, lds4(ks + (c + 16) * C::LD + d), s1);
                dp0 = dot4(dv4, lds4(vs + c * C::LD + d), dp0);
                dp1 = dot4(dv4, lds4(vs + (c + 16) * C::LD + d), dp1);
            }
            const float p0 = jrow[c] >= 0 ? __expf(s0 * a.softmax_scale - lse_s[h]) : 0.0f;
            const float p1 = jrow[c + 16] >= 0 ? __expf(s1 * a.softmax_scale - lse_s[h]) : 0.0f;
            ps[h * (BW_CH + 1) + c] = p0;
            ps[h * (BW_CH + 1) + c + 16] = p1;
            dss[h * (BW_CH + 1) + c] = p0 * (dp0 - D_s[h]);
            dss[h * (BW_CH + 1) + c + 16] = p1 * (dp1 - D_s[h]);
        }
        __syncthreads();
        // dq += scale * ds k: this thread's head and 8 consecutive columns
        {
            const int h = tid / C::TPH, d0 = (tid % C::TPH) * 8;
            if (h < Hq) {
#pragma unroll 4
                for (int c = 0; c < BW_CH; ++c) {
                    const float w = dss[h * (BW_CH + 1) + c];
                    const float4 k0 = lds4(ks + c * C::LD + d0), k1 = lds4(ks + c * C::LD + d0 + 4);
                    dqa[0] = fmaf(w, k0.x, dqa[0]); dqa[1] = fmaf(w, k0.y, dqa[1]);
                    dqa[2] = fmaf(w, k0.z, dqa[2]); dqa[3] = fmaf(w, k0.w, dqa[3]);
                    dqa[4] = fmaf(w, k1.x, dqa[4]); dqa[5] = fmaf(w, k1.y, dqa[5]);
                    dqa[6] = fmaf(w, k1.z, dqa[6]); dqa[7] = fmaf(w, k1.w, dqa[7]);
                }
            }
        }
        // this chunk's dk = scale ds^T q and dv = p^T do: a warp covers whole
        // rows (four columns per lane, one coalesced 16-byte atomic per lane
        // and row); a thread takes RPT rows
        {
            constexpr int LPR = D / 4;                 // lanes per row
            constexpr int RPW = 32 / LPR;              // rows per warp and step
            constexpr int RPT = BW_CH / (RPW * (BW_THREADS / 32));
            const int d0 = (lane % LPR) * 4;
            const int cbase = warp * RPW + lane / LPR;
            float4 gk[RPT], gv[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) { gk[r] = make_float4(0.f, 0.f, 0.f, 0.f); gv[r] = gk[r]; }
            for (int h = 0; h < Hq; ++h) {
                const float4 qv = lds4(qs + h * D + d0), dv4 = lds4(dos + h * D + d0);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int c = cbase + r * RPW * (BW_THREADS / 32);
                    const float dsv = dss[h * (BW_CH + 1) + c], pv = ps[h * (BW_CH + 1) + c];
                    gk[r].x = fmaf(dsv, qv.x, gk[r].x); gk[r].y = fmaf(dsv, qv.y, gk[r].y);
                    gk[r].z = fmaf(dsv, qv.z, gk[r].z); gk[r].w = fmaf(dsv, qv.w, gk[r].w);
                    gv[r].x = fmaf(pv, dv4.x, gv[r].x); gv[r].y = fmaf(pv, dv4.y, gv[r].y);
                    gv[r].z = fmaf(pv, dv4.z, gv[r].z); gv[r].w = fmaf(pv, dv4.w, gv[r].w);
                }
            }
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int c = cbase + r * RPW * (BW_THREADS / 32);
                const int j = jrow[c];
                if (j < 0) continue;
                const float sc = a.softmax_scale;
                atomicAdd(reinterpret_cast<float4*>(a.dk + (int64_t)j * D + d0),
                          make_float4(gk[r].x * sc, gk[r].y * sc, gk[r].z * sc, gk[r].w * sc));
                atomicAdd(reinterpret_cast<float4*>(a.dv + (int64_t)j * D + d0), gv[r]);
            }
        }
        __syncthreads();
    }
    {
        const int h = tid / C::TPH, d0 = (tid % C::TPH) * 8;
        if (h < Hq) {
#pragma unroll
            for (int u = 0; u < 8; ++u) a.dq[((int64_t)t * Hq + h) * D + d0 + u] = dqa[u] * a.softmax_scale;
        }
    }
}

template <int D, typename T>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t s)
{
    const size_t smem = BwCfg<D>::smem(a.Hq);
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attn_bwd_kernel<D, T><<<a.L, BW_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool attention_backward_supported(const BwdArgs& a)
{
    return (a.D == 64 || a.D == 128) && a.Hq >= 1 && a.Hq <= BW_MAX_HQ && (a.dtype == SA_BF16 || a.dtype == SA_F32);
}

cudaError_t launch_attention_backward(const BwdArgs& a, cudaStream_t s)
{
    if (a.L <= 0) return cudaSuccess;
    cudaError_t e = launch_zero(a.dk, sizeof(float) * (size_t)a.L * a.D, s);
    if (e == cudaSuccess) e = launch_zero(a.dv, sizeof(float) * (size_t)a.L * a.D, s);
    if (e != cudaSuccess) return e;
    if (attention_backward_tc_supported(a)) return launch_attention_backward_tc(a, s);
    if (a.dtype == SA_BF16) return a.D == 64 ? launch_bwd_t<64, bf16>(a, s) : launch_bwd_t<128, bf16>(a, s);
    return a.D == 64 ? launch_bwd_t<64, float>(a, s) : launch_bwd_t<128, float>(a, s);
}

}  // namespace sa
