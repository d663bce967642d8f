// Exact softmax attention over the kept rows only, then the sigmoid output
// gate ("Hybrid Attention Architectures...", section 3.1, exact computation
// stage, and the pseudocode of section 3.3: attn_out over kv_history[idx],
// returned as gate * attn_out).
//
//   o[t,h] = sum_{j in S_t} softmax_j(scale * q[t,h] . k[j]) v[j]
//   out[t,h] = sigmoid(gate[t,h]) * o[t,h]
//
// Queries of all heads share one key/value head (MQA, "Sparse Attention and
// Hybrid Attention Architecture Design", section 2), so one gathered row
// serves every head of the token: a CTA takes one query row and 16 heads
// (the M side of the m16n8k16 MMA), gathers the kept K/V rows 64 at a time
// into shared memory with cp.async (double-buffered), and runs an online
// softmax in fp32. With splits > 1 (decode) the kept rows are divided among
// CTAs and the last CTA of a row, found through an atomic ticket, merges the
// partial (max, sum, acc) triples with a log-sum-exp combine. Nothing waits
// on another CTA.
#include <atomic>

#include "attn_common.cuh"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int AT_THREADS = 128;     // 4 warps
constexpr int CHUNK = 64;           // kept rows per pipeline stage
constexpr int PAD = 8;              // bf16 elements of row padding (16 B)
constexpr int MMA_POS_CAP = 2048;   // kept positions a CTA stages in shared memory

// ---------------------------------------------------------------------------
// bf16 tensor-core path (mma.sync m16n8k16); dv = 32 * NT, NT even
// ---------------------------------------------------------------------------
template <int NT, int CH>
__global__ void __launch_bounds__(AT_THREADS)
attn_mma_kernel(AttnArgs a)
{
    constexpr int KPW = CH / 4;            // keys of a chunk per warp (S = Q K^T)
    constexpr int NTW = KPW / 8;           // their 8-key n-tiles
    static_assert(NTW == 1 || NTW == 2, "16 or 8 keys per warp");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ float red_max[4][16], red_sum[4][16];
    __shared__ int sh_flag;
    __shared__ int spos[MMA_POS_CAP];        // the CTA's kept positions (-1: none), when they fit

    griddep_wait();                          // the kept positions
    griddep_launch();
    const int r = blockIdx.x, split = blockIdx.y, hg = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int dqk = a.dqk, dv = a.dv;
    const int qs_ld = dqk + PAD, ks_ld = dqk + PAD, vs_ld = dv + PAD, ps_ld = CH + PAD;

    const int stages = a.stages;
    bf16* Qs = reinterpret_cast<bf16*>(smem_raw);
    bf16* Ks = Qs + 16 * qs_ld;
    bf16* Vs = Ks + stages * CH * ks_ld;
    bf16* Ps = Vs + (a.v_aliases_k ? 0 : stages * CH * vs_ld);
    const int vld = a.v_aliases_k ? ks_ld : vs_ld;

    const int64_t n = attn_hist_len(a, r);
    const int n_sel = attn_kept(a, r, n);
    const int per = (a.K + a.splits - 1) / a.splits;
    const int begin = min(split * per, n_sel), end = min(begin + per, n_sel);
    const int cnt = end - begin;
    const int64_t base = attn_base(a, r);
    const int32_t* sel = a.idx + (int64_t)r * a.K;
    const bf16* kp = static_cast<const bf16*>(a.k);
    const bf16* vp = static_cast<const bf16*>(a.v);

    // Q tile: 16 heads of this group
    {
        const bf16* q = static_cast<const bf16*>(a.q);
        const int pieces = dqk / 8;
        for (int i = tid; i < 16 * pieces; i += AT_THREADS) {
            const int row = i / pieces, pc = i % pieces, h = hg * 16 + row;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < a.Hq) v = *reinterpret_cast<const uint4*>(q + ((int64_t)r * a.Hq + h) * dqk + pc * 8);
            *reinterpret_cast<uint4*>(Qs + row * qs_ld + pc * 8) = v;
        }
    }

    // the positions of the CTA's kept rows are staged once, so that no copy
    // below waits on an index load
    const bool staged = cnt <= MMA_POS_CAP;
    if (staged) {
        for (int i = tid; i < cnt; i += AT_THREADS) {
            const int pos = sel[begin + i];
            spos[i] = (pos >= 0 && pos < n) ? pos : -1;
        }
        __syncthreads();
    }
    auto pos_of = [&](int slot) -> int {
        if (slot >= end) return -1;
        if (staged) return spos[slot - begin];
        const int pos = sel[slot];
        return (pos >= 0 && pos < n) ? pos : -1;
    };
    // a warp copies whole rows (its lanes stride over the row's 16-byte
    // pieces), so that no per-piece index arithmetic is needed
    auto issue = [&](int c, int buf) {
        const int kpieces = dqk / 8, vpieces = dv / 8;
        bf16* kdst = Ks + buf * CH * ks_ld;
        bf16* vdst = Vs + buf * CH * vs_ld;
        for (int row = warp; row < CH; row += AT_THREADS / 32) {
            const int pos = pos_of(begin + c * CH + row);
            const bool ok = pos >= 0;
            const bf16* ksrc = kp + (ok ? (base + pos) * a.ld_k : 0);
            bf16* kd = kdst + row * ks_ld;
            for (int pc = lane; pc < kpieces; pc += 32) cp_async16(kd + pc * 8, ksrc + pc * 8, ok);
            if (!a.v_aliases_k) {
                const bf16* vsrc = vp + (ok ? (base + pos) * a.ld_v : 0);
                bf16* vd = vdst + row * vs_ld;
                for (int pc = lane; pc < vpieces; pc += 32) cp_async16(vd + pc * 8, vsrc + pc * 8, ok);
            }
        }
        cp_async_commit();
    };

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const float sl2 = a.softmax_scale * LOG2E;
    const int nchunks = (cnt + CH - 1) / CH;
    const int mat = lane >> 3, rr = lane & 7;
    const int colbase = warp * (dv / 4);

    // cp.async pipeline: chunk c lives in buffer c % stages; up to stages - 1
    // chunks are in flight while one is being consumed
    for (int c = 0; c < min(nchunks, max(stages - 1, 1)); ++c) issue(c, c);
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c % stages;
        const int pending = min(nchunks - 1, c + stages - 2) - c;     // groups allowed in flight
        if (pending >= 2) cp_async_wait<2>();
        else if (pending == 1) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();
        if (stages >= 2 && c + stages - 1 < nchunks) issue(c + stages - 1, (c + stages - 1) % stages);

        const bf16* Kb = Ks + buf * CH * ks_ld;
        const bf16* Vb = a.v_aliases_k ? Kb : Vs + buf * CH * vs_ld;

        // S = Q K^T for this warp's KPW keys
        float s[NTW][4];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
        if constexpr (NTW == 2) {
            for (int ks = 0; ks < dqk / 16; ++ks) {
                uint32_t af[4], bfm[4];
                ldsm_x4(af, smem_u32(Qs + ((mat & 1) * 8 + rr) * qs_ld + ks * 16 + (mat >> 1) * 8));
                ldsm_x4(bfm, smem_u32(Kb + (warp * 16 + (mat >> 1) * 8 + rr) * ks_ld + ks * 16 + (mat & 1) * 8));
                mma_16816(s[0], af, bfm[0], bfm[1]);
                mma_16816(s[NTW - 1], af, bfm[2], bfm[3]);
            }
        } else {
            // 8 keys per warp: one B load covers two k-steps (dqk % 32 == 0)
            for (int ks = 0; ks < dqk / 16; ks += 2) {
                uint32_t af0[4], af1[4], bfm[4];
                ldsm_x4(af0, smem_u32(Qs + ((mat & 1) * 8 + rr) * qs_ld + ks * 16 + (mat >> 1) * 8));
                ldsm_x4(af1, smem_u32(Qs + ((mat & 1) * 8 + rr) * qs_ld + (ks + 1) * 16 + (mat >> 1) * 8));
                ldsm_x4(bfm, smem_u32(Kb + (warp * 8 + rr) * ks_ld + ks * 16 + (mat & 1) * 8 + (mat >> 1) * 16));
                mma_16816(s[0], af0, bfm[0], bfm[1]);
                mma_16816(s[0], af1, bfm[2], bfm[3]);
            }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kc = warp * KPW + nt * 8 + 2 * t4 + e;
                const bool ok = begin + c * CH + kc < end;
                s[nt][e] = ok ? s[nt][e] * sl2 : -INFINITY;
                s[nt][2 + e] = ok ? s[nt][2 + e] * sl2 : -INFINITY;
                mx0 = fmaxf(mx0, s[nt][e]);
                mx1 = fmaxf(mx1, s[nt][2 + e]);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        if (t4 == 0) { red_max[warp][g] = mx0; red_max[warp][g + 8] = mx1; }
        __syncthreads();
        float cm0 = fmaxf(fmaxf(red_max[0][g], red_max[1][g]), fmaxf(red_max[2][g], red_max[3][g]));
        float cm1 = fmaxf(fmaxf(red_max[0][g + 8], red_max[1][g + 8]), fmaxf(red_max[2][g + 8], red_max[3][g + 8]));
        const float mn0 = fmaxf(m0, cm0), mn1 = fmaxf(m1, cm1);
        const float al0 = (m0 == -INFINITY) ? 0.0f : exp2f(m0 - mn0);
        const float al1 = (m1 == -INFINITY) ? 0.0f : exp2f(m1 - mn1);
        const float ref0 = (mn0 == -INFINITY) ? 0.0f : mn0;
        const float ref1 = (mn1 == -INFINITY) ? 0.0f : mn1;
        m0 = mn0; m1 = mn1;
        float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            const uint32_t p01 = pack_bf16x2(exp2f(s[nt][0] - ref0), exp2f(s[nt][1] - ref0));
            const uint32_t p23 = pack_bf16x2(exp2f(s[nt][2] - ref1), exp2f(s[nt][3] - ref1));
            const float2 f01 = bf16x2_to_f32x2(p01), f23 = bf16x2_to_f32x2(p23);
            ps0 += f01.x + f01.y;
            ps1 += f23.x + f23.y;
            const int col = warp * KPW + nt * 8 + 2 * t4;
            *reinterpret_cast<uint32_t*>(Ps + g * ps_ld + col) = p01;
            *reinterpret_cast<uint32_t*>(Ps + (g + 8) * ps_ld + col) = p23;
        }
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
        if (t4 == 0) { red_sum[warp][g] = ps0; red_sum[warp][g + 8] = ps1; }
        __syncthreads();
        l0 = l0 * al0 + (red_sum[0][g] + red_sum[1][g] + red_sum[2][g] + red_sum[3][g]);
        l1 = l1 * al1 + (red_sum[0][g + 8] + red_sum[1][g + 8] + red_sum[2][g + 8] + red_sum[3][g + 8]);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            o[i][0] *= al0; o[i][1] *= al0; o[i][2] *= al1; o[i][3] *= al1;
        }
        // O += P V for this warp's value columns
#pragma unroll
        for (int ks = 0; ks < CH / 16; ++ks) {
            uint32_t af[4];
            ldsm_x4(af, smem_u32(Ps + ((mat & 1) * 8 + rr) * ps_ld + ks * 16 + (mat >> 1) * 8));
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t bfm[4];
                ldsm_x4_trans(bfm, smem_u32(Vb + (ks * 16 + (mat & 1) * 8 + rr) * vld + colbase + np * 16 + (mat >> 1) * 8));
                mma_16816(o[2 * np], af, bfm[0], bfm[1]);
                mma_16816(o[2 * np + 1], af, bfm[2], bfm[3]);
            }
        }
        if (stages == 1 && c + 1 < nchunks) {     // single buffer: refill once everyone is done
            __syncthreads();
            issue(c + 1, 0);
        }
    }

    const int h0 = hg * 16 + g, h1 = hg * 16 + g + 8;
    if (a.splits == 1) {
        const float gs0 = h0 < a.Hq ? gate_of(a, r, h0) / (l0 > 0.0f ? l0 : 1.0f) : 0.0f;
        const float gs1 = h1 < a.Hq ? gate_of(a, r, h1) / (l1 > 0.0f ? l1 : 1.0f) : 0.0f;
        bf16* out = static_cast<bf16*>(a.out);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int col = colbase + i * 8 + 2 * t4;
            if (h0 < a.Hq)
                *reinterpret_cast<uint32_t*>(out + ((int64_t)r * a.Hq + h0) * dv + col) = pack_bf16x2(o[i][0] * gs0, o[i][1] * gs0);
            if (h1 < a.Hq)
                *reinterpret_cast<uint32_t*>(out + ((int64_t)r * a.Hq + h1) * dv + col) = pack_bf16x2(o[i][2] * gs1, o[i][3] * gs1);
        }
        return;
    }

    // split partial: unnormalised acc, running max (log2 units), running sum
    float* p0 = a.part + (((int64_t)r * a.splits + split) * a.Hq + h0) * (dv + 2);
    float* p1 = a.part + (((int64_t)r * a.splits + split) * a.Hq + h1) * (dv + 2);
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        const int col = colbase + i * 8 + 2 * t4;
        if (h0 < a.Hq) *reinterpret_cast<float2*>(p0 + col) = make_float2(o[i][0], o[i][1]);
        if (h1 < a.Hq) *reinterpret_cast<float2*>(p1 + col) = make_float2(o[i][2], o[i][3]);
    }
    if (warp == 0 && t4 == 0) {
        if (h0 < a.Hq) { p0[dv] = m0; p0[dv + 1] = l0; }
        if (h1 < a.Hq) { p1[dv] = m1; p1[dv + 1] = l1; }
    }
    const int groups = (a.Hq + 15) / 16;
    if (take_ticket(a.tickets + (int64_t)r * groups + hg, a.splits, &sh_flag)) {
        combine_splits<bf16>(a, r, hg * 16, min(a.Hq, hg * 16 + 16));
        if (tid == 0) a.tickets[(int64_t)r * groups + hg] = 0u;
    }
}

// ---------------------------------------------------------------------------
// general path on CUDA cores: any dtype, any widths; one CTA per (row, split,
// head)
// ---------------------------------------------------------------------------
constexpr int SIMT_MAX_DV_PER_THREAD = 4;   // dv <= 512

template <typename T>
__global__ void __launch_bounds__(AT_THREADS)
attn_simt_kernel(AttnArgs a)
{
    extern __shared__ float qsh[];            // [dqk]
    __shared__ float pw[AT_THREADS];
    __shared__ int64_t prow[AT_THREADS];
    __shared__ float red[AT_THREADS / 32];
    __shared__ int sh_flag;
    griddep_wait();
    griddep_launch();
    const int r = blockIdx.x, split = blockIdx.y, h = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int dqk = a.dqk, dv = a.dv;
    const T* q = static_cast<const T*>(a.q) + ((int64_t)r * a.Hq + h) * dqk;
    for (int d = tid; d < dqk; d += AT_THREADS) qsh[d] = to_f32(q[d]);

    const int64_t n = attn_hist_len(a, r);
    const int n_sel = attn_kept(a, r, n);
    const int per = (a.K + a.splits - 1) / a.splits;
    const int begin = min(split * per, n_sel), end = min(begin + per, n_sel);
    const int64_t base = attn_base(a, r);
    const int32_t* sel = a.idx + (int64_t)r * a.K;
    const T* kp = static_cast<const T*>(a.k);
    const T* vp = static_cast<const T*>(a.v);
    const float sl2 = a.softmax_scale * LOG2E;
    __syncthreads();

    float o[SIMT_MAX_DV_PER_THREAD] = {0, 0, 0, 0};
    float m = -INFINITY, l = 0.0f;
    for (int c0 = begin; c0 < end; c0 += AT_THREADS) {
        const int slot = c0 + tid;
        float logit = -INFINITY;
        int64_t row = -1;
        if (slot < end) {
            const int pos = sel[slot];
            if (pos >= 0 && pos < n) {
                row = base + pos;
                const T* kr = kp + row * a.ld_k;
                float acc = 0.0f;
                for (int d = 0; d < dqk; ++d) acc = fmaf(qsh[d], to_f32(kr[d]), acc);
                logit = acc * sl2;
            }
        }
        float cm = warp_max(logit);
        if (lane == 0) red[warp] = cm;
        __syncthreads();
        cm = red[0];
        for (int w = 1; w < AT_THREADS / 32; ++w) cm = fmaxf(cm, red[w]);
        const float mn = fmaxf(m, cm);
        const float al = (m == -INFINITY) ? 0.0f : exp2f(m - mn);
        const float ref = (mn == -INFINITY) ? 0.0f : mn;
        m = mn;
        const float p = exp2f(logit - ref);
        pw[tid] = p;
        prow[tid] = row;
        __syncthreads();
        float ps = warp_sum(p);
        __syncthreads();                      // everyone has read red[] above
        if (lane == 0) red[warp] = ps;
        __syncthreads();
        float tot = 0.0f;
        for (int w = 0; w < AT_THREADS / 32; ++w) tot += red[w];
        l = l * al + tot;
        const int cnt = min(AT_THREADS, end - c0);
#pragma unroll
        for (int u = 0; u < SIMT_MAX_DV_PER_THREAD; ++u) {
            const int col = tid + u * AT_THREADS;
            if (col >= dv) break;
            float acc = o[u] * al;
            for (int i = 0; i < cnt; ++i)
                if (prow[i] >= 0) acc = fmaf(pw[i], to_f32(vp[prow[i] * a.ld_v + col]), acc);
            o[u] = acc;
        }
        __syncthreads();
    }

    if (a.splits == 1) {
        const float gs = gate_of(a, r, h) / (l > 0.0f ? l : 1.0f);
        T* out = static_cast<T*>(a.out) + ((int64_t)r * a.Hq + h) * dv;
#pragma unroll
        for (int u = 0; u < SIMT_MAX_DV_PER_THREAD; ++u) {
            const int col = tid + u * AT_THREADS;
            if (col < dv) store_out<T>(out + col, o[u] * gs);
        }
        return;
    }
    float* pp = a.part + (((int64_t)r * a.splits + split) * a.Hq + h) * (dv + 2);
#pragma unroll
    for (int u = 0; u < SIMT_MAX_DV_PER_THREAD; ++u) {
        const int col = tid + u * AT_THREADS;
        if (col < dv) pp[col] = o[u];
    }
    if (tid == 0) { pp[dv] = m; pp[dv + 1] = l; }
    if (take_ticket(a.tickets + (int64_t)r * a.Hq + h, a.splits, &sh_flag)) {
        combine_splits<T>(a, r, h, h + 1);
        if (tid == 0) a.tickets[(int64_t)r * a.Hq + h] = 0u;
    }
}

// Kept rows per pipeline stage: 32 for wide rows (the 576-wide latent row),
// so that two stages and two CTAs fit an SM, else 64.
int mma_chunk(const AttnArgs& a)
{
    return (a.dqk >= 256 && a.dqk % 32 == 0) ? 32 : CHUNK;
}

size_t mma_smem_bytes(const AttnArgs& a, int stages)
{
    const size_t ch = (size_t)mma_chunk(a);
    return sizeof(bf16) * ((size_t)16 * (a.dqk + PAD) + (size_t)stages * ch * (a.dqk + PAD) +
                           (a.v_aliases_k ? 0 : (size_t)stages * ch * (a.dv + PAD)) +
                           16 * (ch + PAD));
}

constexpr size_t MMA_SMEM_LIMIT = 200 * 1024;    // leaves room for static shared memory

// Pipeline depth: double buffering (the kernel supports up to 4 buffers)
// unless that leaves room for only one CTA per SM.
int attention_stages(const AttnArgs& a)
{
    // measured: two CTAs per SM beat a deeper pipeline in one CTA (the
    // 576-wide latent row with 64-row stages: 2 stages, one CTA per SM, 241 us
    // per decode step at 64 x 32K; 1 stage, two CTAs per SM, 203 us); with
    // 32-row stages the latent row gets both: two stages, two CTAs per SM
    return mma_smem_bytes(a, 2) <= 104 * 1024 ? 2 : 1;     // + 9 KB static: two CTAs per SM
}

template <int NT>
cudaError_t launch_mma(AttnArgs a, cudaStream_t s)
{
    a.stages = attention_stages(a);
    const size_t smem = mma_smem_bytes(a, a.stages);
    auto kern = mma_chunk(a) == 32 ? attn_mma_kernel<NT, 32> : attn_mma_kernel<NT, CHUNK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();                  // do not leave the error latched
        return e;
    }
    dim3 grid(a.rows, a.splits, (a.Hq + 15) / 16);
    return launch_kernel(kern, grid, dim3(AT_THREADS), smem, s, a.pdl, a);
}

}  // namespace

bool attention_mma_supported(const AttnArgs& a)
{
    if (a.dtype != SA_BF16) return false;
    if (mma_smem_bytes(a, 1) > MMA_SMEM_LIMIT) return false;
    if (a.dqk % 16 != 0 || a.dqk > 576) return false;
    if (a.dv % 64 != 0 || a.dv > 512) return false;
    if (a.v_aliases_k && a.dv > a.dqk) return false;
    return true;
}

// Splits of the kept rows per query row for the decode attention: at most
// about two CTAs per SM (148 SMs) in all, and at least 256 (self-gathering
// kernel) or 128 (shared-tile kernel) kept rows per CTA, so that each CTA's
// pipeline streams long enough to hide its fill. Both measured against more
// and fewer splits.
int attention_splits(int K, int64_t n_cap, int rows, bool gather_kernel)
{
    const int64_t kept = min64(K, n_cap);
    const int target = 2 * 148;
    const int64_t min_per = gather_kernel ? 256 : 128;
    if (kept <= min_per || rows <= 0 || rows >= target) return 1;
    const int want = gather_kernel ? (target + rows - 1) / rows : max(1, target / rows);
    int64_t per = (kept + want - 1) / want;
    per = max64(max64(min_per, (K + MAX_SPLITS - 1) / MAX_SPLITS), per);
    per = (per + CHUNK - 1) / CHUNK * CHUNK;
    return (int)((K + per - 1) / per);
}

// Kernel choice for prefill rows (SA_ATTN_*). Measured at the 128K prefill
// shapes (16 heads per key/value head): 16.3 ms with the default kernel,
// 22.8 ms on tcgen05, whose 64 KB tiles become usable only when the last of
// their 4096 copies lands.
static std::atomic<int> g_prefill_attention{SA_ATTN_AUTO};

int set_prefill_attention_kernel(int which) { return g_prefill_attention.exchange(which); }

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
    if (g_prefill_attention.load(std::memory_order_relaxed) == SA_ATTN_TCGEN05 && attention_tc_supported(a)) {
        const cudaError_t e = launch_attention_tc(a, s);
        if (e != cudaErrorNotSupported) return e;
    }
    if (attention_gather_supported(a)) {
        const cudaError_t e = launch_attention_gather(a, s);
        if (e != cudaErrorNotSupported) return e;
    }
    if (attention_mma_supported(a)) {
        switch (a.dv / 32) {
        case 2: return launch_mma<2>(a, s);
        case 4: return launch_mma<4>(a, s);
        case 6: return launch_mma<6>(a, s);
        case 8: return launch_mma<8>(a, s);
        case 12: return launch_mma<12>(a, s);
        case 16: return launch_mma<16>(a, s);
        default: break;
        }
    }
    dim3 grid(a.rows, a.splits, a.Hq);
    const size_t smem = sizeof(float) * a.dqk;
    if (a.dtype == SA_F32) return launch_kernel(attn_simt_kernel<float>, grid, dim3(AT_THREADS), smem, s, a.pdl, a);
    return launch_kernel(attn_simt_kernel<bf16>, grid, dim3(AT_THREADS), smem, s, a.pdl, a);
}

}  // namespace sa
