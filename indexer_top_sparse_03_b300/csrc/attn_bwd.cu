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
// chunk into shared memory (rows padded by one word: conflict-free columns).
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
    static constexpr int LD = D + 1;                       // padded row of the chunk tiles
    static constexpr int PER = BW_MAX_HQ * D / BW_THREADS; // (head, column) outputs per thread
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

template <int D, typename T>
__global__ void __launch_bounds__(BW_THREADS)
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

    // (head, column) outputs of this thread: index tid + BW_THREADS * k
    float acc[C::PER];
#pragma unroll
    for (int k = 0; k < C::PER; ++k) acc[k] = 0.0f;

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
        for (int p = tid; p < Hq * BW_CH; p += BW_THREADS) {
            const int h = p / BW_CH, c = p % BW_CH;
            float s = 0.0f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) s = fmaf(qs[h * D + d], ks[c * C::LD + d], s);
            ps[h * (BW_CH + 1) + c] = jrow[c] >= 0 ? s * a.softmax_scale : -INFINITY;
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
#pragma unroll
        for (int k = 0; k < C::PER; ++k) {
            const int i = tid + BW_THREADS * k;
            const int h = i / D, e = i % D;
            if (h < Hq) {
                float o = acc[k] * al_s[h];
#pragma unroll 8
                for (int c = 0; c < BW_CH; ++c) o = fmaf(ps[h * (BW_CH + 1) + c], vs[c * C::LD + e], o);
                acc[k] = o;
            }
        }
        __syncthreads();
    }
    // o = acc / l; D_h = do . o; dout . o for the gate
#pragma unroll
    for (int k = 0; k < C::PER; ++k) {
        const int i = tid + BW_THREADS * k;
        const int h = i / D;
        float dsum = 0.0f, tsum = 0.0f;
        if (h < Hq) {
            const float o = l_s[h] > 0.0f ? acc[k] / l_s[h] : 0.0f;
            dsum = dos[i] * o;
            tsum = dos_raw[i] * o;
        }
        // a warp's 32 outputs share one head (D is a multiple of 32)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            dsum += __shfl_xor_sync(0xFFFFFFFFu, dsum, o);
            tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, o);
        }
        if (lane == 0 && h < Hq) { atomicAdd(&D_s[h], dsum); atomicAdd(&dto_s[h], tsum); }
        acc[k] = 0.0f;                          // reused for dq
    }
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
        for (int p = tid; p < Hq * BW_CH; p += BW_THREADS) {
            const int h = p / BW_CH, c = p % BW_CH;
            float s = 0.0f, dp = 0.0f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) {
                s = fmaf(qs[h * D + d], ks[c * C::LD + d], s);
                dp = fmaf(dos[h * D + d], vs[c * C::LD + d], dp);
            }
            const float pr = jrow[c] >= 0 ? __expf(s * a.softmax_scale - lse_s[h]) : 0.0f;
            ps[h * (BW_CH + 1) + c] = pr;
            dss[h * (BW_CH + 1) + c] = pr * (dp - D_s[h]);
        }
        __syncthreads();
        // dq += scale * ds k
#pragma unroll
        for (int k = 0; k < C::PER; ++k) {
            const int i = tid + BW_THREADS * k;
            const int h = i / D, d = i % D;
            if (h < Hq) {
                float g = acc[k];
#pragma unroll 8
                for (int c = 0; c < BW_CH; ++c) g = fmaf(dss[h * (BW_CH + 1) + c], ks[c * C::LD + d], g);
                acc[k] = g;
            }
        }
        // this chunk's dk = scale ds^T q and dv = p^T do, four columns per atomic
        for (int x = tid; x < BW_CH * (D / 4); x += BW_THREADS) {
            const int c = x / (D / 4), d0 = (x % (D / 4)) * 4;
            const int j = jrow[c];
            if (j < 0) continue;
            float4 gk = make_float4(0.f, 0.f, 0.f, 0.f), gv = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int h = 0; h < Hq; ++h) {
                const float dsv = dss[h * (BW_CH + 1) + c], pv = ps[h * (BW_CH + 1) + c];
                const float* qh = qs + h * D + d0;
                const float* dh = dos + h * D + d0;
                gk.x = fmaf(dsv, qh[0], gk.x); gk.y = fmaf(dsv, qh[1], gk.y);
                gk.z = fmaf(dsv, qh[2], gk.z); gk.w = fmaf(dsv, qh[3], gk.w);
                gv.x = fmaf(pv, dh[0], gv.x); gv.y = fmaf(pv, dh[1], gv.y);
                gv.z = fmaf(pv, dh[2], gv.z); gv.w = fmaf(pv, dh[3], gv.w);
            }
            gk.x *= a.softmax_scale; gk.y *= a.softmax_scale; gk.z *= a.softmax_scale; gk.w *= a.softmax_scale;
            atomicAdd(reinterpret_cast<float4*>(a.dk + (int64_t)j * D + d0), gk);
            atomicAdd(reinterpret_cast<float4*>(a.dv + (int64_t)j * D + d0), gv);
        }
        __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < C::PER; ++k) {
        const int i = tid + BW_THREADS * k;
        if (i < Hq * D) a.dq[(int64_t)t * Hq * D + i] = acc[k] * a.softmax_scale;
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
    if (a.dtype == SA_BF16) return a.D == 64 ? launch_bwd_t<64, bf16>(a, s) : launch_bwd_t<128, bf16>(a, s);
    return a.D == 64 ? launch_bwd_t<64, float>(a, s) : launch_bwd_t<128, float>(a, s);
}

}  // namespace sa
