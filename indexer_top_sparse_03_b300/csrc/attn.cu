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
#include "attn_common.cuh"
#include "../../include/sparse_attn.h"

namespace sa {
namespace {

constexpr int AT_THREADS = 128;     // 4 warps
constexpr int CHUNK = 64;           // kept rows per pipeline stage
constexpr int PAD = 8;              // bf16 elements of row padding (16 B)

// ---------------------------------------------------------------------------
// bf16 tensor-core path (mma.sync m16n8k16); dv = 32 * NT, NT even
// ---------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(AT_THREADS)
attn_mma_kernel(AttnArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ float red_max[4][16], red_sum[4][16];
    __shared__ int sh_flag;

    griddep_wait();                          // the kept positions
    griddep_launch();
    const int r = blockIdx.x, split = blockIdx.y, hg = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int dqk = a.dqk, dv = a.dv;
    const int qs_ld = dqk + PAD, ks_ld = dqk + PAD, vs_ld = dv + PAD, ps_ld = CHUNK + PAD;

    const int stages = a.stages;
    bf16* Qs = reinterpret_cast<bf16*>(smem_raw);
    bf16* Ks = Qs + 16 * qs_ld;
    bf16* Vs = Ks + stages * CHUNK * ks_ld;
    bf16* Ps = Vs + (a.v_aliases_k ? 0 : stages * CHUNK * vs_ld);
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

    auto issue = [&](int c, int buf) {
        const int kpieces = dqk / 8, vpieces = dv / 8;
        bf16* kdst = Ks + buf * CHUNK * ks_ld;
        for (int i = tid; i < CHUNK * kpieces; i += AT_THREADS) {
            const int row = i / kpieces, pc = i % kpieces;
            const int slot = begin + c * CHUNK + row;
            int pos = slot < end ? sel[slot] : -1;
            const bool ok = pos >= 0 && pos < n;
            const bf16* src = kp + (ok ? (base + pos) * a.ld_k + pc * 8 : 0);
            cp_async16(kdst + row * ks_ld + pc * 8, src, ok);
        }
        if (!a.v_aliases_k) {
            bf16* vdst = Vs + buf * CHUNK * vs_ld;
            for (int i = tid; i < CHUNK * vpieces; i += AT_THREADS) {
                const int row = i / vpieces, pc = i % vpieces;
                const int slot = begin + c * CHUNK + row;
                int pos = slot < end ? sel[slot] : -1;
                const bool ok = pos >= 0 && pos < n;
                const bf16* src = vp + (ok ? (base + pos) * a.ld_v + pc * 8 : 0);
                cp_async16(vdst + row * vs_ld + pc * 8, src, ok);
            }
        }
        cp_async_commit();
    };

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const float sl2 = a.softmax_scale * LOG2E;
    const int nchunks = (cnt + CHUNK - 1) / CHUNK;
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

        const bf16* Kb = Ks + buf * CHUNK * ks_ld;
        const bf16* Vb = a.v_aliases_k ? Kb : Vs + buf * CHUNK * vs_ld;

        // S = Q K^T for this warp's 16 keys
        float s[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
        for (int ks = 0; ks < dqk / 16; ++ks) {
            uint32_t af[4], bfm[4];
            ldsm_x4(af, smem_u32(Qs + ((mat & 1) * 8 + rr) * qs_ld + ks * 16 + (mat >> 1) * 8));
            ldsm_x4(bfm, smem_u32(Kb + (warp * 16 + (mat >> 1) * 8 + rr) * ks_ld + ks * 16 + (mat & 1) * 8));
            mma_16816(s[0], af, bfm[0], bfm[1]);
            mma_16816(s[1], af, bfm[2], bfm[3]);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kc = warp * 16 + nt * 8 + 2 * t4 + e;
                const bool ok = begin + c * CHUNK + kc < end;
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
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t p01 = pack_bf16x2(exp2f(s[nt][0] - ref0), exp2f(s[nt][1] - ref0));
            const uint32_t p23 = pack_bf16x2(exp2f(s[nt][2] - ref1), exp2f(s[nt][3] - ref1));
            const float2 f01 = bf16x2_to_f32x2(p01), f23 = bf16x2_to_f32x2(p23);
            ps0 += f01.x + f01.y;
            ps1 += f23.x + f23.y;
            const int col = warp * 16 + nt * 8 + 2 * t4;
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
        for (int ks = 0; ks < CHUNK / 16; ++ks) {
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

size_t mma_smem_bytes(const AttnArgs& a, int stages)
{
    return sizeof(bf16) * ((size_t)16 * (a.dqk + PAD) + (size_t)stages * CHUNK * (a.dqk + PAD) +
                           (a.v_aliases_k ? 0 : (size_t)stages * CHUNK * (a.dv + PAD)) +
                           16 * (CHUNK + PAD));
}

constexpr size_t MMA_SMEM_LIMIT = 200 * 1024;    // leaves room for static shared memory

// Pipeline depth: double buffering (the kernel supports up to 4 buffers)
// unless that leaves room for only one CTA per SM.
int attention_stages(const AttnArgs& a)
{
    // measured: more CTAs per SM beat a deeper pipeline in one CTA
    // (the 576-wide latent row: 2 stages, one CTA per SM, 241 us per decode
    // step at 64 x 32K; 1 stage, two CTAs per SM, 203 us)
    return mma_smem_bytes(a, 2) <= 110 * 1024 ? 2 : 1;
}

template <int NT>
cudaError_t launch_mma(AttnArgs a, cudaStream_t s)
{
    a.stages = attention_stages(a);
    const size_t smem = mma_smem_bytes(a, a.stages);
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();                  // do not leave the error latched
        return e;
    }
    dim3 grid(a.rows, a.splits, (a.Hq + 15) / 16);
    return launch_kernel(attn_mma_kernel<NT>, grid, dim3(AT_THREADS), smem, s, a.pdl, a);
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

// Splits of the kept rows per query row for the decode attention. The
// self-gathering kernel: about two waves of CTAs on 148 SMs, at least 256
// kept rows per CTA. The shared-tile kernel (wide latent rows, one CTA per SM
// at most two): about four waves, at least 128 kept rows per CTA. Both
// measured against more and fewer splits.
int attention_splits(int K, int64_t n_cap, int rows, bool gather_kernel)
{
    const int64_t kept = min64(K, n_cap);
    const int target = (gather_kernel ? 2 : 4) * 148;
    const int64_t min_per = gather_kernel ? 256 : 128;
    if (kept <= min_per || rows <= 0 || rows >= target) return 1;
    const int want = (target + rows - 1) / rows;
    int64_t per = (kept + want - 1) / want;
    per = max64(max64(min_per, (K + MAX_SPLITS - 1) / MAX_SPLITS), per);
    per = (per + CHUNK - 1) / CHUNK * CHUNK;
    return (int)((K + per - 1) / per);
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s)
{
    if (a.rows <= 0) return cudaSuccess;
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
