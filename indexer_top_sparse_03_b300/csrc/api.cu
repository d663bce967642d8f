// C ABI of the sparse attention library: argument checks, workspace layout and
// the order of the launches. Every check runs on the host before anything is
// enqueued; nothing here allocates device memory or synchronises.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "kernels.h"
#include "../../include/sparse_attn.h"

namespace sa {
bool attention_mma_supported(const AttnArgs& a);
}

namespace {

constexpr size_t WS_ALIGN = 256;

// NVTX range over one entry point or stage (free when no tool is attached)
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
constexpr int MAX_K = 65536;

size_t align_up(size_t x) { return (x + WS_ALIGN - 1) / WS_ALIGN * WS_ALIGN; }
bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
bool valid_dtype(int d) { return d == SA_F32 || d == SA_BF16 || d == SA_FP8_E4M3; }

int status_of(cudaError_t e) { return e == cudaSuccess ? SA_OK : SA_ERR_LAUNCH; }

int check_indexer_shape(int dtype, int Hi, int di)
{
    if (!valid_dtype(dtype)) return SA_ERR_INVALID_ARG;
    if (Hi < 1 || di < 1) return SA_ERR_INVALID_ARG;
    if (Hi > 32 || di % 16 != 0 || di > 256) return SA_ERR_UNSUPPORTED;
    return SA_OK;
}

// ---- prefill workspace layout --------------------------------------------
// kept positions (if not returned) | score rows of one pass (also the scratch
// rows of the fused path's fallback) | fused path: sampled keys, their
// scales, sampled scores, thresholds, segment counts, segment pairs, failure
// list
//
// Rows whose history is long enough take the fused path (indexer filter pass
// + selection among the kept pairs); the plan fixes from which row on, and
// the shape of every fused pass, on the host.
constexpr int SAMPLE_LG = 4;                 // one sampled key per 16 positions

struct FusePlan {
    bool on;
    int64_t t_fuse;          // first fused row
    int64_t rows;            // rows per fused pass
    int tq, lcap, cand_cap;
    int64_t ns, ld_ssc, words;
    int nseg_max;
    size_t seg_words_max;    // max over passes of rows * nseg * cap_seg
};

struct PrefillLayout {
    int64_t rows_per_pass;   // query rows scored per indexer/Top-K pass
    int64_t ld_s;            // score row stride: L rounded up to a multiple of 4 (16-byte rows)
    FusePlan fuse;
    size_t idx_off, scores_off, ksamp_off, kscale_off, ssc_off, thr_off, cnt_off, seg_off, fail_off, total;
};

// pairs a row keeps at its threshold, generously: 16 x (K/16 + 6 sigma + 17)
int64_t fused_expected_pairs(int K)
{
    const double share = K / 16.0;
    return 16 * ((int64_t)ceil(share + 6.0 * sqrt(share) + 16.0) + 1);
}

// segments per row and pairs per segment of the fused pass over rows [t0, t1)
void fused_pass_shape(int64_t t0, int64_t t1, int K, int& nseg, int& cap_seg)
{
    const double per_item = (double)sa::INDEXER_GROUP * 128.0 * (double)fused_expected_pairs(K) / (double)(t0 + 1);
    cap_seg = (int)ceil(2.0 * per_item + 48.0);
    nseg = (int)(((t1 + 127) / 128 + sa::INDEXER_GROUP - 1) / sa::INDEXER_GROUP);
}

// end of the fused pass that starts at t0: passes are aligned to end at L,
// so that only the first one is partial
int64_t fused_pass_end(const FusePlan& f, int64_t L, int64_t t0)
{
    const int64_t len = t0 == f.t_fuse ? (L - f.t_fuse - 1) % f.rows + 1 : f.rows;
    return t0 + len < L ? t0 + len : L;
}

FusePlan fuse_plan(const sa_prefill_args& a, int64_t rows_per_pass)
{
    FusePlan f{};
    sa::IndexerArgs ia{};
    ia.dtype = a.idx_dtype; ia.Hi = a.Hi; ia.di = a.di;
    f.lcap = sa::indexer_filter_lcap(ia);
    if (f.lcap <= 64) return f;
    f.tq = sa::indexer_query_tile(ia);
    const int64_t E = fused_expected_pairs(a.K);
    f.cand_cap = (int)((2 * E + 1023) / 1024 * 1024);
    if (f.cand_cap < 8192) f.cand_cap = 8192;
    if (f.cand_cap > 16384) return f;
    // the first row whose per-item pairs fit the local lists twice over
    int64_t n_req = (int64_t)ceil(2.0 * sa::INDEXER_GROUP * 128.0 * (double)E / (double)(f.lcap - 48));
    if (n_req < 8 * (int64_t)a.K) n_req = 8 * (int64_t)a.K;
    f.t_fuse = n_req - 1;
    if (f.t_fuse >= a.L) return f;
    f.ns = sa::sample_count(a.L - 1, SAMPLE_LG);
    if (f.ns > 16384) return f;              // the threshold step's shared-memory row
    f.ld_ssc = (f.ns + 3) / 4 * 4;
    f.words = (a.L + 31) / 32;
    // rows per fused pass: at most the score pass's rows (the fallback rescores
    // into those rows), and few enough that the pair segments stay <= 256 MB
    const int64_t t_req = f.t_fuse;
    for (f.rows = rows_per_pass < 2048 ? rows_per_pass : 2048;; f.rows /= 2) {
        // start on a pass boundary counted back from L when a whole pass fits
        const int64_t whole = (a.L - t_req) / f.rows;
        f.t_fuse = whole > 0 ? a.L - whole * f.rows : t_req;
        f.nseg_max = 0;
        f.seg_words_max = 0;
        for (int64_t t0 = f.t_fuse; t0 < a.L; t0 = fused_pass_end(f, a.L, t0)) {
            const int64_t t1 = fused_pass_end(f, a.L, t0);
            int nseg, cap;
            fused_pass_shape(t0, t1, a.K, nseg, cap);
            if (cap > f.lcap) return f;
            if (nseg > f.nseg_max) f.nseg_max = nseg;
            const size_t w = (size_t)(t1 - t0) * nseg * cap;
            if (w > f.seg_words_max) f.seg_words_max = w;
        }
        if (f.seg_words_max * 8 <= (size_t(256) << 20) || f.rows <= 128) break;
    }
    sa::FusedSelectArgs probe{};
    probe.cand_cap = f.cand_cap; probe.words = f.words; probe.nseg = f.nseg_max;
    if (sa::fused_select_smem(probe) > 200 * 1024) return f;
    f.on = true;
    return f;
}

PrefillLayout prefill_layout(const sa_prefill_args& a)
{
    PrefillLayout l{};
    const int64_t L = a.L;
    const int64_t budget = int64_t(1) << 30;               // bytes of scores per pass
    l.ld_s = (L + 3) / 4 * 4;
    int64_t rows = budget / (4 * (l.ld_s > 0 ? l.ld_s : 4));
    rows = rows < 1 ? 1 : (rows > L ? L : rows);
    l.rows_per_pass = rows;
    l.fuse = fuse_plan(a, rows);
    size_t off = 0;
    l.idx_off = off;
    if (a.idx_out == nullptr) off += align_up(sizeof(int32_t) * (size_t)L * a.K);
    l.scores_off = off;
    off += align_up(sizeof(float) * (size_t)rows * (size_t)l.ld_s);
    if (l.fuse.on) {
        const FusePlan& f = l.fuse;
        const size_t es = a.idx_dtype == SA_BF16 ? 2 : (a.idx_dtype == SA_FP8_E4M3 ? 1 : 4);
        l.ksamp_off = off;
        off += align_up((size_t)f.ns * a.di * es);
        l.kscale_off = off;
        off += align_up(sizeof(float) * (size_t)f.ns);
        l.ssc_off = off;
        off += align_up(sizeof(float) * (size_t)f.rows * (size_t)f.ld_ssc);
        l.thr_off = off;
        off += align_up(sizeof(uint32_t) * (size_t)f.rows);
        l.cnt_off = off;
        off += align_up(sizeof(unsigned) * (size_t)f.rows * (size_t)f.nseg_max);
        l.seg_off = off;
        off += align_up(sizeof(unsigned long long) * f.seg_words_max);
        l.fail_off = off;
        off += align_up(sizeof(unsigned) * (4 + (size_t)f.rows));
    }
    l.total = off;
    return l;
}

int check_prefill_scalars(const sa_prefill_args* a)
{
    if (!a) return SA_ERR_INVALID_ARG;
    if (a->L < 0 || a->Hq < 1 || a->dqk < 1 || a->dv < 1 || a->K < 1) return SA_ERR_INVALID_ARG;
    int st = check_indexer_shape(a->idx_dtype, a->Hi, a->di);
    if (st != SA_OK) return st;
    if (a->attn_dtype != SA_F32 && a->attn_dtype != SA_BF16) {
        return a->attn_dtype == SA_FP8_E4M3 ? SA_ERR_UNSUPPORTED : SA_ERR_INVALID_ARG;
    }
    if (a->ld_k < a->dqk || a->ld_v < a->dv) return SA_ERR_INVALID_ARG;
    if (a->K > MAX_K || a->Hq > 64) return SA_ERR_UNSUPPORTED;
    if (a->dqk % 8 != 0 || a->dv % 8 != 0 || a->ld_k % 8 != 0 || a->ld_v % 8 != 0) return SA_ERR_UNSUPPORTED;
    if (a->attn_dtype == SA_BF16 ? (a->dqk > 576 || a->dv > 512) : (a->dqk > 256 || a->dv > 512))
        return SA_ERR_UNSUPPORTED;
    if (!(a->softmax_scale == a->softmax_scale)) return SA_ERR_INVALID_ARG;   // NaN
    return SA_OK;
}

int check_prefill(const sa_prefill_args* a)
{
    int st = check_prefill_scalars(a);
    if (st != SA_OK || a->L == 0) return st;
    if (!a->q || !a->k || !a->v || !a->q_idx || !a->k_idx || !a->w || !a->gate || !a->out)
        return SA_ERR_INVALID_ARG;
    if (a->idx_dtype == SA_FP8_E4M3 && (!a->q_scale || !a->k_scale)) return SA_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->q_idx, 16) ||
        !aligned(a->k_idx, 16) || !aligned(a->out, 16) || !aligned(a->w, 4) || !aligned(a->gate, 4))
        return SA_ERR_INVALID_ARG;
    return SA_OK;
}

// ---- decode workspace layout ----------------------------------------------
// scores | zeroed block: key-bin histograms, candidate counters, split-K
// tickets, scan tickets | threshold bins | kept-position bitmaps | candidate
// lists | kept positions (if not returned) | split-K partials
struct DecodeLayout {
    int splits;
    int64_t ld_w, ld_s;
    size_t scores_off, hist_off, cnt_off, tickets_off, row_tickets_off, zero_bytes, split_off, bitmap_off, cand_off,
        idx_off, part_off, total;
};

DecodeLayout decode_layout(const sa_decode_args& a)
{
    DecodeLayout l{};
    // the self-gathering kernel takes bf16 rows of 64 or 128 with separate values
    const bool gather = a.attn_dtype == SA_BF16 && a.dqk == a.dv && (a.dqk == 64 || a.dqk == 128) &&
                        !(a.v_cache == a.k_cache && a.ld_v == a.ld_k);
    l.splits = sa::attention_splits(a.K, a.max_ctx, a.B, gather);
    const size_t B = (size_t)a.B;
    const int64_t ctx = a.max_ctx > 0 ? a.max_ctx : 1;
    l.ld_w = (ctx + 127) / 128 * 4;             // bitmap words per row, a multiple of 4
    l.ld_s = l.ld_w * 32;                       // score row stride, a multiple of 128
    size_t off = 0;
    l.scores_off = off;
    off += align_up(sizeof(float) * B * (size_t)l.ld_s);
    l.hist_off = off;
    off += sizeof(unsigned) * B * 4096;
    l.cnt_off = off;
    off += sizeof(unsigned) * B;
    l.tickets_off = off;
    off += sizeof(unsigned) * B * (size_t)a.Hq;
    l.row_tickets_off = off;
    off += sizeof(unsigned) * B;
    off = align_up(off);
    l.zero_bytes = off - l.hist_off;
    l.split_off = off;
    off += align_up(sizeof(sa::BinSplit) * B);
    l.bitmap_off = off;
    off += align_up(sizeof(uint32_t) * B * (size_t)l.ld_w);
    l.cand_off = off;
    off += align_up(sizeof(unsigned long long) * B * sa::DECODE_CAND_CAP);
    l.idx_off = off;
    if (a.idx_out == nullptr) off += align_up(sizeof(int32_t) * B * a.K);
    l.part_off = off;
    if (l.splits > 1) off += align_up(sizeof(float) * B * l.splits * a.Hq * (a.dv + 2));
    l.total = off;
    return l;
}

int check_decode_scalars(const sa_decode_args* a)
{
    if (!a) return SA_ERR_INVALID_ARG;
    if (a->B < 0 || a->Hq < 1 || a->dqk < 1 || a->dv < 1 || a->K < 1 || a->max_ctx < 0)
        return SA_ERR_INVALID_ARG;
    if (!valid_dtype(a->idx_dtype) || !valid_dtype(a->attn_dtype)) return SA_ERR_INVALID_ARG;
    if (a->Hi < 1 || a->di < 1) return SA_ERR_INVALID_ARG;
    if (a->ld_k < a->dqk || a->ld_v < a->dv) return SA_ERR_INVALID_ARG;
    if (a->attn_dtype != SA_BF16) return SA_ERR_UNSUPPORTED;
    if (a->idx_dtype != SA_BF16 && a->idx_dtype != SA_FP8_E4M3) return SA_ERR_UNSUPPORTED;
    if (a->Hi > 32 || a->di % 32 != 0 || a->di > 256) return SA_ERR_UNSUPPORTED;
    if (a->idx_dtype == SA_FP8_E4M3 && a->di % 64 != 0) return SA_ERR_UNSUPPORTED;
    if (a->dqk % 16 != 0 || a->dv % 16 != 0 || a->dqk > 576 || a->dv > 512) return SA_ERR_UNSUPPORTED;
    if (a->ld_k % 8 != 0 || a->ld_v % 8 != 0 || a->K > MAX_K || a->Hq > 64) return SA_ERR_UNSUPPORTED;
    if (a->max_ctx >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
    if (!(a->softmax_scale == a->softmax_scale)) return SA_ERR_INVALID_ARG;
    return SA_OK;
}

int check_decode(const sa_decode_args* a)
{
    int st = check_decode_scalars(a);
    if (st != SA_OK || a->B == 0) return st;
    if (!a->q || !a->q_idx || !a->w || !a->gate || !a->k_cache || !a->v_cache || !a->k_idx_cache ||
        !a->seq_start || !a->ctx_len || !a->out)
        return SA_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->q_idx, 16) || !aligned(a->k_cache, 16) ||
        !aligned(a->v_cache, 16) || !aligned(a->k_idx_cache, 16) || !aligned(a->out, 16) ||
        !aligned(a->seq_start, 8) || !aligned(a->ctx_len, 4))
        return SA_ERR_INVALID_ARG;
    if (a->idx_dtype == SA_FP8_E4M3 &&
        (!a->q_scale || !a->k_idx_scale || !aligned(a->q_scale, 4) || !aligned(a->k_idx_scale, 4)))
        return SA_ERR_INVALID_ARG;
    return SA_OK;
}

// ---- block-granular prefill ------------------------------------------------
// pooled keys | block scores of one pass | block row lengths | kept blocks |
// kept positions (if not returned) | kept-position counts
struct BlocksLayout {
    int lg;
    int64_t nb, ld_b, rows_per_pass;
    size_t pooled_off, scores_off, rowlen_off, blk_off, idx_off, cnt_off, total;
};

int block_lg(int block_size)
{
    if (block_size < 1 || block_size > 1024 || (block_size & (block_size - 1))) return -1;
    int lg = 0;
    while ((1 << lg) < block_size) ++lg;
    return lg;
}

BlocksLayout blocks_layout(const sa_prefill_args& a, int lg)
{
    BlocksLayout l{};
    l.lg = lg;
    l.nb = ((int64_t)a.L + (1 << lg) - 1) >> lg;
    l.ld_b = (l.nb + 3) / 4 * 4;
    int64_t rows = (int64_t(1) << 30) / (4 * (l.ld_b > 0 ? l.ld_b : 4));
    l.rows_per_pass = rows < 1 ? 1 : (rows > a.L ? a.L : rows);
    const int Kb = a.K >> lg;
    size_t off = 0;
    l.pooled_off = off; off += align_up(sizeof(uint16_t) * (size_t)l.nb * a.di);
    l.scores_off = off; off += align_up(sizeof(float) * (size_t)l.rows_per_pass * l.ld_b);
    l.rowlen_off = off; off += align_up(sizeof(int32_t) * (size_t)l.rows_per_pass);
    l.blk_off = off; off += align_up(sizeof(int32_t) * (size_t)l.rows_per_pass * Kb);
    l.idx_off = off;
    if (a.idx_out == nullptr) off += align_up(sizeof(int32_t) * (size_t)a.L * a.K);
    l.cnt_off = off; off += align_up(sizeof(int32_t) * (size_t)a.L);
    l.total = off;
    return l;
}

int check_blocks(const sa_prefill_args* a, int block_size, bool scalars_only)
{
    int st = scalars_only ? check_prefill_scalars(a) : check_prefill(a);
    if (st != SA_OK) return st;
    const int lg = block_lg(block_size);
    if (lg < 0) return SA_ERR_INVALID_ARG;
    if (a->K % block_size != 0) return SA_ERR_INVALID_ARG;
    if (a->idx_dtype != SA_BF16) return SA_ERR_UNSUPPORTED;
    return SA_OK;
}

}  // namespace

extern "C" {

const char* sa_status_string(int status)
{
    switch (status) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument";
    case SA_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case SA_ERR_WORKSPACE: return "workspace missing or too small";
    case SA_ERR_LAUNCH: return "CUDA launch error";
    default: return "unknown status";
    }
}

int sa_version(void) { return 100; }

int sa_set_prefill_attention_kernel(int which)
{
    if (which != SA_ATTN_AUTO && which != SA_ATTN_TCGEN05) return SA_ERR_INVALID_ARG;
    return sa::set_prefill_attention_kernel(which);
}

int sa_device_errors(unsigned* bits, int reset)
{
    if (!bits) return SA_ERR_INVALID_ARG;
    unsigned idx_bits = 0, attn_bits = 0, dense_bits = 0;
    if (sa::indexer_device_errors(&idx_bits, reset != 0) != cudaSuccess ||
        sa::attention_tc_device_errors(&attn_bits, reset != 0) != cudaSuccess ||
        sa::attention_dense_tc_device_errors(&dense_bits, reset != 0) != cudaSuccess)
        return SA_ERR_LAUNCH;
    *bits = idx_bits | attn_bits | dense_bits;
    return SA_OK;
}

int indexer_score(const void* q_idx, int dtype, const float* q_scale, const float* w,
                  const void* k_idx, const float* k_scale, int T, int N, int Hi, int di,
                  int64_t causal_offset, float* scores, int64_t ld_s, cudaStream_t stream)
{
    if (T < 0 || N < 0) return SA_ERR_INVALID_ARG;
    int st = check_indexer_shape(dtype, Hi, di);
    if (st != SA_OK) return st;
    if (T == 0 || N == 0) return SA_OK;
    if (!q_idx || !w || !k_idx || !scores || ld_s < N) return SA_ERR_INVALID_ARG;
    if (dtype == SA_FP8_E4M3 && (!q_scale || !k_scale)) return SA_ERR_INVALID_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16) || !aligned(scores, 4) || !aligned(w, 4))
        return SA_ERR_INVALID_ARG;
    sa::IndexerArgs a{};
    a.q_idx = q_idx; a.dtype = dtype; a.q_scale = q_scale; a.w = w;
    a.k_idx = k_idx; a.k_scale = k_scale;
    a.T = T; a.N = N; a.Hi = Hi; a.di = di; a.causal_offset = causal_offset;
    a.t_begin = 0; a.scores = scores; a.ld_s = ld_s;
    return status_of(sa::launch_indexer(a, stream));
}

int topk_select(const float* scores, int64_t ld_s, const int32_t* row_len, int T, int K,
                int32_t* idx_out, cudaStream_t stream)
{
    if (T < 0 || K < 1 || ld_s < 1) return SA_ERR_INVALID_ARG;
    if (K > MAX_K) return SA_ERR_UNSUPPORTED;
    if (T == 0) return SA_OK;
    if (!scores || !row_len || !idx_out) return SA_ERR_INVALID_ARG;
    if (!aligned(scores, 4) || !aligned(row_len, 4) || !aligned(idx_out, 4)) return SA_ERR_INVALID_ARG;
    sa::TopkArgs a{};
    a.scores = scores; a.ld_s = ld_s; a.row_len = row_len; a.causal_first = 0;
    a.n_cap = ld_s; a.rows = T; a.K = K; a.idx = idx_out; a.ld_idx = K;
    return status_of(sa::launch_topk(a, stream));
}

size_t sa_prefill_workspace_size(const sa_prefill_args* args)
{
    if (check_prefill_scalars(args) != SA_OK) return 0;
    return prefill_layout(*args).total;
}

int sparse_attn_prefill(const sa_prefill_args* args, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    NvtxRange range("sparse_attn_prefill");
    int st = check_prefill(args);
    if (st != SA_OK) return st;
    const sa_prefill_args& a = *args;
    if (a.L == 0) return SA_OK;
    const PrefillLayout lay = prefill_layout(a);
    if (!ws || ws_bytes < lay.total || !aligned(ws, WS_ALIGN)) return SA_ERR_WORKSPACE;
    char* wsb = static_cast<char*>(ws);
    int32_t* idx = a.idx_out ? a.idx_out : reinterpret_cast<int32_t*>(wsb + lay.idx_off);
    float* scores = reinterpret_cast<float*>(wsb + lay.scores_off);

    const FusePlan& f = lay.fuse;
    bool sampled = false;
    for (int64_t t0 = 0; t0 < a.L;) {
        const bool fused = f.on && t0 >= f.t_fuse;
        int64_t t1 = fused ? fused_pass_end(f, a.L, t0) : t0 + lay.rows_per_pass;
        if (f.on && !fused && t1 > f.t_fuse) t1 = f.t_fuse;
        if (t1 > a.L) t1 = a.L;
        sa::IndexerArgs ia{};
        ia.q_idx = a.q_idx; ia.dtype = a.idx_dtype; ia.q_scale = a.q_scale; ia.w = a.w;
        ia.k_idx = a.k_idx; ia.k_scale = a.k_scale;
        ia.T = (int)t1; ia.N = (int)t1; ia.Hi = a.Hi; ia.di = a.di; ia.causal_offset = 0;
        ia.t_begin = (int)t0; ia.scores = scores; ia.ld_s = lay.ld_s;
        if (!fused) {
            cudaError_t e = sa::launch_indexer(ia, stream);
            if (e != cudaSuccess) return SA_ERR_LAUNCH;
            sa::TopkArgs ta{};
            ta.scores = scores; ta.ld_s = lay.ld_s; ta.row_len = nullptr; ta.causal_first = t0;
            ta.n_cap = t1; ta.rows = (int)(t1 - t0); ta.K = a.K; ta.idx = idx + t0 * a.K; ta.ld_idx = a.K;
            e = sa::launch_topk(ta, stream);
            if (e != cudaSuccess) return SA_ERR_LAUNCH;
        } else {
            void* ksamp = wsb + lay.ksamp_off;
            float* kscale = reinterpret_cast<float*>(wsb + lay.kscale_off);
            float* ssc = reinterpret_cast<float*>(wsb + lay.ssc_off);
            unsigned* fail = reinterpret_cast<unsigned*>(wsb + lay.fail_off);
            if (!sampled) {
                const int es = a.idx_dtype == SA_BF16 ? 2 : (a.idx_dtype == SA_FP8_E4M3 ? 1 : 4);
                if (sa::launch_sample_gather(a.k_idx, a.di * es, a.idx_dtype == SA_FP8_E4M3 ? a.k_scale : nullptr, f.ns,
                                             SAMPLE_LG, ksamp, kscale, stream) != cudaSuccess)
                    return SA_ERR_LAUNCH;
                sampled = true;
            }
            // 1. scores against the sampled keys of every row's history
            sa::IndexerArgs sia = ia;
            sia.k_idx = ksamp; sia.k_scale = a.idx_dtype == SA_FP8_E4M3 ? kscale : nullptr;
            sia.N = (int)f.ns; sia.sample_log2 = SAMPLE_LG; sia.scores = ssc; sia.ld_s = f.ld_ssc;
            if (sa::launch_indexer(sia, stream) != cudaSuccess) return SA_ERR_LAUNCH;
            // 2. thresholds
            sa::FusedSelectArgs fa{};
            fa.t_begin = t0; fa.rows = (int)(t1 - t0); fa.N = t1; fa.K = a.K;
            fa.tq = f.tq; fa.group = sa::INDEXER_GROUP; fa.sample_log2 = SAMPLE_LG; fa.ns = f.ns;
            fa.thr = reinterpret_cast<uint32_t*>(wsb + lay.thr_off);
            fa.seg_cnt = reinterpret_cast<unsigned*>(wsb + lay.cnt_off);
            fa.seg_cand = reinterpret_cast<unsigned long long*>(wsb + lay.seg_off);
            fused_pass_shape(t0, t1, a.K, fa.nseg, fa.cap_seg);
            fa.cand_cap = f.cand_cap; fa.words = f.words;
            fa.idx = idx + t0 * a.K; fa.ld_idx = a.K;
            fa.fail_cnt = fail; fa.fail_list = reinterpret_cast<int*>(fail + 4);
            fa.ia = ia; fa.scratch = scores; fa.ld_scratch = lay.ld_s;
            if (sa::launch_sample_threshold(fa, ssc, f.ld_ssc, f.ns, stream) != cudaSuccess) return SA_ERR_LAUNCH;
            // 3. the filter pass: kept pairs per work item, no scores stored
            sa::IndexerArgs fia = ia;
            fia.scores = nullptr; fia.ld_s = 0;
            fia.thr = fa.thr; fia.seg_cnt = reinterpret_cast<unsigned*>(wsb + lay.cnt_off);
            fia.seg_cand = reinterpret_cast<unsigned long long*>(wsb + lay.seg_off);
            fia.nseg = fa.nseg; fia.cap_seg = fa.cap_seg;
            if (sa::launch_indexer_tc(fia, stream) != cudaSuccess) return SA_ERR_LAUNCH;
            // 4-5. exact selection, then the rows that need the fallback
            if (sa::launch_zero(fail, 16, stream) != cudaSuccess) return SA_ERR_LAUNCH;
            if (sa::launch_fused_select(fa, stream) != cudaSuccess) return SA_ERR_LAUNCH;
        }
        t0 = t1;
    }
    if (a.stage_events && cudaEventRecord(a.stage_events[0], stream) != cudaSuccess) return SA_ERR_LAUNCH;
    // Rows whose history fits in K keep every position, and the next rows keep
    // a large share of theirs: the dense causal kernel computes them (key tiles
    // shared by 8 queries, rows t >= K masked to their kept positions) more
    // cheaply than per-row gathers; the gather kernel takes the rest. A dense
    // row costs in proportion to t, a gathered one to K; the measured
    // crossover is at t = 4K on the tensor-core dense kernel (5K the same, 6K
    // and 3K slower) and at 2K on the mma.sync one.
    const bool aliased = (a.v == a.k) && a.ld_v == a.ld_k;
    int64_t dense_rows = 0;
    if (a.attn_dtype == SA_BF16 && a.dqk == a.dv && !aliased) {
        sa::DenseArgs da{};
        da.q = a.q; da.k = a.k; da.ld_k = a.ld_k; da.v = a.v; da.ld_v = a.ld_v; da.gate = a.gate; da.out = a.out;
        da.Hq = a.Hq; da.D = a.dqk;
        da.softmax_scale = a.softmax_scale; da.idx = idx; da.K = a.K; da.mask_from = a.K;
        da.L = 4 * (int64_t)a.K < a.L ? 4 * (int64_t)a.K : a.L;
        if (!sa::attention_dense_tc_supported(da)) da.L = 2 * (int64_t)a.K < a.L ? 2 * (int64_t)a.K : a.L;
        if (sa::attention_dense_tc_supported(da) || sa::attention_dense_supported(da)) {
            if (sa::launch_attention_dense(da, stream) != cudaSuccess) return SA_ERR_LAUNCH;
            dense_rows = da.L;
        }
    }
    if (dense_rows < a.L) {
        const size_t es = a.attn_dtype == SA_BF16 ? 2 : 4;
        sa::AttnArgs at{};
        at.q = static_cast<const char*>(a.q) + (size_t)dense_rows * a.Hq * a.dqk * es;
        at.k = a.k; at.ld_k = a.ld_k; at.v = a.v; at.ld_v = a.ld_v;
        at.v_aliases_k = aliased;
        at.row_base = nullptr; at.idx = idx + dense_rows * a.K; at.K = a.K; at.ctx_len = nullptr;
        at.causal_first = dense_rows; at.n_cap = a.L; at.gate = a.gate + dense_rows * a.Hq;
        at.rows = (int)(a.L - dense_rows); at.Hq = a.Hq; at.dqk = a.dqk; at.dv = a.dv;
        at.softmax_scale = a.softmax_scale; at.dtype = a.attn_dtype;
        at.out = static_cast<char*>(a.out) + (size_t)dense_rows * a.Hq * a.dv * es;
        at.splits = 1; at.part = nullptr; at.tickets = nullptr;
        if (sa::launch_attention(at, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    }
    if (a.stage_events && cudaEventRecord(a.stage_events[1], stream) != cudaSuccess) return SA_ERR_LAUNCH;
    return SA_OK;
}

int sparse_attn_backward(const sa_backward_args* args, cudaStream_t stream)
{
    NvtxRange range("sparse_attn_backward");
    if (!args) return SA_ERR_INVALID_ARG;
    const sa_backward_args& a = *args;
    if (a.L < 0 || a.Hq < 1 || a.dqk < 1 || a.dv < 1 || a.K < 1) return SA_ERR_INVALID_ARG;
    if (a.dtype != SA_BF16 && a.dtype != SA_F32) return valid_dtype(a.dtype) ? SA_ERR_UNSUPPORTED : SA_ERR_INVALID_ARG;
    if (a.ld_k < a.dqk || a.ld_v < a.dv) return SA_ERR_INVALID_ARG;
    if (!(a.softmax_scale == a.softmax_scale)) return SA_ERR_INVALID_ARG;
    if (a.dqk != a.dv || a.K > MAX_K || a.ld_k % 8 != 0 || a.ld_v % 8 != 0) return SA_ERR_UNSUPPORTED;
    sa::BwdArgs b{};
    b.L = a.L; b.Hq = a.Hq; b.D = a.dqk; b.K = a.K; b.dtype = a.dtype; b.softmax_scale = a.softmax_scale;
    b.q = a.q; b.k = a.k; b.ld_k = a.ld_k; b.v = a.v; b.ld_v = a.ld_v; b.idx = a.idx; b.gate = a.gate;
    b.dout = a.dout; b.dq = a.dq; b.dk = a.dk; b.dv = a.dv_out; b.dgate = a.dgate;
    if (!sa::attention_backward_supported(b)) return SA_ERR_UNSUPPORTED;
    if (a.L == 0) return SA_OK;
    if (!a.q || !a.k || !a.v || !a.idx || !a.gate || !a.dout || !a.dq || !a.dk || !a.dv_out || !a.dgate)
        return SA_ERR_INVALID_ARG;
    if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.dout, 16) ||
        !aligned(a.dk, 16) || !aligned(a.dv_out, 16) || !aligned(a.dq, 4) || !aligned(a.dgate, 4) ||
        !aligned(a.gate, 4) || !aligned(a.idx, 4))
        return SA_ERR_INVALID_ARG;
    return status_of(sa::launch_attention_backward(b, stream));
}

size_t sa_prefill_blocks_workspace_size(const sa_prefill_args* args, int block_size)
{
    if (check_blocks(args, block_size, true) != SA_OK) return 0;
    return blocks_layout(*args, block_lg(block_size)).total;
}

int sparse_attn_prefill_blocks(const sa_prefill_args* args, int block_size, void* ws, size_t ws_bytes,
                               cudaStream_t stream)
{
    NvtxRange range("sparse_attn_prefill_blocks");
    int st = check_blocks(args, block_size, false);
    if (st != SA_OK) return st;
    const sa_prefill_args& a = *args;
    if (a.L == 0) return SA_OK;
    const BlocksLayout lay = blocks_layout(a, block_lg(block_size));
    if (!ws || ws_bytes < lay.total || !aligned(ws, WS_ALIGN)) return SA_ERR_WORKSPACE;
    char* wsb = static_cast<char*>(ws);
    void* pooled = wsb + lay.pooled_off;
    float* scores = reinterpret_cast<float*>(wsb + lay.scores_off);
    int32_t* rowlen = reinterpret_cast<int32_t*>(wsb + lay.rowlen_off);
    int32_t* blk = reinterpret_cast<int32_t*>(wsb + lay.blk_off);
    int32_t* idx = a.idx_out ? a.idx_out : reinterpret_cast<int32_t*>(wsb + lay.idx_off);
    int32_t* cnt = reinterpret_cast<int32_t*>(wsb + lay.cnt_off);
    const int Kb = a.K >> lay.lg;

    if (sa::launch_pool_keys(a.k_idx, a.L, a.di, lay.lg, pooled, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    for (int64_t t0 = 0; t0 < a.L; t0 += lay.rows_per_pass) {
        const int64_t t1 = (t0 + lay.rows_per_pass < a.L) ? t0 + lay.rows_per_pass : a.L;
        const int rows = (int)(t1 - t0);
        sa::IndexerArgs ia{};
        ia.q_idx = a.q_idx; ia.dtype = a.idx_dtype; ia.w = a.w;
        ia.k_idx = pooled; ia.T = (int)t1; ia.N = (int)lay.nb; ia.Hi = a.Hi; ia.di = a.di;
        ia.t_begin = (int)t0; ia.scores = scores; ia.ld_s = lay.ld_b; ia.block_log2 = lay.lg;
        if (sa::launch_indexer(ia, stream) != cudaSuccess) return SA_ERR_LAUNCH;
        if (sa::launch_block_rowlen(t0, rows, lay.lg, rowlen, stream) != cudaSuccess) return SA_ERR_LAUNCH;
        sa::TopkArgs ta{};
        ta.scores = scores; ta.ld_s = lay.ld_b; ta.row_len = rowlen; ta.n_cap = lay.nb;
        ta.rows = rows; ta.K = Kb; ta.idx = blk; ta.ld_idx = Kb;
        if (sa::launch_topk(ta, stream) != cudaSuccess) return SA_ERR_LAUNCH;
        if (sa::launch_expand_blocks(blk, Kb, t0, rows, lay.lg, idx + t0 * a.K, cnt + t0, stream) != cudaSuccess)
            return SA_ERR_LAUNCH;
    }
    if (a.stage_events && cudaEventRecord(a.stage_events[0], stream) != cudaSuccess) return SA_ERR_LAUNCH;
    // as in the token-level prefill, the rows below 4K go through the
    // tensor-core dense kernel masked to their kept positions (every row:
    // the expanded block lists are -1 padded like the token lists)
    const bool aliased = (a.v == a.k) && a.ld_v == a.ld_k;
    int64_t dense_rows = 0;
    if (a.attn_dtype == SA_BF16 && a.dqk == a.dv && !aliased) {
        sa::DenseArgs da{};
        da.q = a.q; da.k = a.k; da.ld_k = a.ld_k; da.v = a.v; da.ld_v = a.ld_v; da.gate = a.gate; da.out = a.out;
        da.Hq = a.Hq; da.D = a.dqk; da.softmax_scale = a.softmax_scale; da.idx = idx; da.K = a.K; da.mask_from = 0;
        da.L = 4 * (int64_t)a.K < a.L ? 4 * (int64_t)a.K : a.L;
        if (sa::attention_dense_tc_supported(da)) {
            if (sa::launch_attention_dense(da, stream) != cudaSuccess) return SA_ERR_LAUNCH;
            dense_rows = da.L;
        }
    }
    if (dense_rows < a.L) {
        const size_t es = a.attn_dtype == SA_BF16 ? 2 : 4;
        sa::AttnArgs at{};
        at.q = static_cast<const char*>(a.q) + (size_t)dense_rows * a.Hq * a.dqk * es;
        at.k = a.k; at.ld_k = a.ld_k; at.v = a.v; at.ld_v = a.ld_v;
        at.v_aliases_k = aliased;
        at.row_base = nullptr; at.idx = idx + dense_rows * a.K; at.K = a.K; at.ctx_len = nullptr;
        at.kept_len = cnt + dense_rows;
        at.causal_first = dense_rows; at.n_cap = a.L; at.gate = a.gate + dense_rows * a.Hq;
        at.rows = (int)(a.L - dense_rows); at.Hq = a.Hq; at.dqk = a.dqk; at.dv = a.dv;
        at.softmax_scale = a.softmax_scale; at.dtype = a.attn_dtype;
        at.out = static_cast<char*>(a.out) + (size_t)dense_rows * a.Hq * a.dv * es;
        at.splits = 1; at.part = nullptr; at.tickets = nullptr;
        if (sa::launch_attention(at, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    }
    if (a.stage_events && cudaEventRecord(a.stage_events[1], stream) != cudaSuccess) return SA_ERR_LAUNCH;
    return SA_OK;
}

size_t sa_prefill_local_workspace_size(const sa_prefill_args* args, int window)
{
    if (check_prefill_scalars(args) != SA_OK || window < 1 || args->attn_dtype != SA_BF16) return 0;
    const sa_prefill_args& a = *args;
    size_t off = prefill_layout(a).total;
    off += align_up(sizeof(int32_t) * (size_t)a.L * window);            // window positions
    off += align_up(sizeof(int32_t) * (size_t)a.L);                     // their counts
    off += align_up(sizeof(float) * (size_t)a.L * a.Hq);                // negated gate logits
    off += align_up(sizeof(uint16_t) * (size_t)a.L * a.Hq * a.dv);      // the local branch's output
    return off;
}

int sparse_attn_prefill_local(const sa_prefill_args* args, int window, void* ws, size_t ws_bytes,
                              cudaStream_t stream)
{
    NvtxRange range("sparse_attn_prefill_local");
    int st = check_prefill(args);
    if (st != SA_OK) return st;
    if (window < 1) return SA_ERR_INVALID_ARG;
    if (args->attn_dtype != SA_BF16) return SA_ERR_UNSUPPORTED;
    const sa_prefill_args& a = *args;
    if (a.L == 0) return SA_OK;
    const size_t need = sa_prefill_local_workspace_size(args, window);
    if (!ws || ws_bytes < need || !aligned(ws, WS_ALIGN)) return SA_ERR_WORKSPACE;
    // the sparse branch, gated by g
    const size_t base = prefill_layout(a).total;
    st = sparse_attn_prefill(args, ws, base, stream);
    if (st != SA_OK) return st;
    char* wsb = static_cast<char*>(ws) + base;
    int32_t* widx = reinterpret_cast<int32_t*>(wsb);
    wsb += align_up(sizeof(int32_t) * (size_t)a.L * window);
    int32_t* wcnt = reinterpret_cast<int32_t*>(wsb);
    wsb += align_up(sizeof(int32_t) * (size_t)a.L);
    float* neg = reinterpret_cast<float*>(wsb);
    wsb += align_up(sizeof(float) * (size_t)a.L * a.Hq);
    void* local = wsb;
    // the local branch, gated by 1 - g = sigmoid(-x), then the sum
    if (sa::launch_window_idx(0, a.L, window, widx, wcnt, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    if (sa::launch_negate(a.gate, neg, (int64_t)a.L * a.Hq, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    sa::AttnArgs at{};
    at.q = a.q; at.k = a.k; at.ld_k = a.ld_k; at.v = a.v; at.ld_v = a.ld_v;
    at.v_aliases_k = (a.v == a.k) && a.ld_v == a.ld_k;
    at.row_base = nullptr; at.idx = widx; at.K = window; at.ctx_len = nullptr; at.kept_len = wcnt;
    at.causal_first = 0; at.n_cap = a.L; at.gate = neg;
    at.rows = a.L; at.Hq = a.Hq; at.dqk = a.dqk; at.dv = a.dv;
    at.softmax_scale = a.softmax_scale; at.dtype = a.attn_dtype; at.out = local;
    at.splits = 1; at.part = nullptr; at.tickets = nullptr;
    if (sa::launch_attention(at, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    if (sa::launch_add_bf16(a.out, local, (int64_t)a.L * a.Hq * a.dv, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    return SA_OK;
}

int attention_dense_causal(const void* q, const void* k, int64_t ld_k, const void* v, int64_t ld_v,
                           const float* gate, void* out, int L, int Hq, int d, float softmax_scale,
                           cudaStream_t stream)
{
    if (L < 0 || Hq < 1 || d < 1 || ld_k < d || ld_v < d) return SA_ERR_INVALID_ARG;
    if (!(softmax_scale == softmax_scale)) return SA_ERR_INVALID_ARG;
    sa::DenseArgs a{};
    a.q = q; a.k = k; a.ld_k = ld_k; a.v = v; a.ld_v = ld_v; a.gate = gate; a.out = out;
    a.L = L; a.Hq = Hq; a.D = d; a.softmax_scale = softmax_scale;
    if (!sa::attention_dense_supported(a)) return SA_ERR_UNSUPPORTED;
    if (L == 0) return SA_OK;
    if (!q || !k || !v || !gate || !out) return SA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(gate, 4))
        return SA_ERR_INVALID_ARG;
    return status_of(sa::launch_attention_dense(a, stream));
}

size_t sa_decode_workspace_size(const sa_decode_args* args)
{
    if (check_decode_scalars(args) != SA_OK) return 0;
    return decode_layout(*args).total;
}

int sparse_attn_decode(const sa_decode_args* args, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    NvtxRange range("sparse_attn_decode");
    int st = check_decode(args);
    if (st != SA_OK) return st;
    const sa_decode_args& a = *args;
    if (a.B == 0) return SA_OK;
    const DecodeLayout lay = decode_layout(a);
    if (!ws || ws_bytes < lay.total || !aligned(ws, WS_ALIGN)) return SA_ERR_WORKSPACE;
    char* wsb = static_cast<char*>(ws);
    float* scores = reinterpret_cast<float*>(wsb + lay.scores_off);
    unsigned* hist = reinterpret_cast<unsigned*>(wsb + lay.hist_off);
    unsigned* cand_cnt = reinterpret_cast<unsigned*>(wsb + lay.cnt_off);
    unsigned* tickets = reinterpret_cast<unsigned*>(wsb + lay.tickets_off);
    int32_t* idx = a.idx_out ? a.idx_out : reinterpret_cast<int32_t*>(wsb + lay.idx_off);
    float* part = reinterpret_cast<float*>(wsb + lay.part_off);

    if (sa::launch_zero(wsb + lay.hist_off, lay.zero_bytes, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    sa::DecodeScanArgs da{};
    da.q_idx = a.q_idx; da.w = a.w; da.k_idx = a.k_idx_cache; da.seq_start = a.seq_start;
    da.fp8 = a.idx_dtype == SA_FP8_E4M3; da.q_scale = a.q_scale; da.k_scale = a.k_idx_scale;
    da.ctx_len = a.ctx_len; da.max_ctx = a.max_ctx; da.B = a.B; da.Hi = a.Hi; da.di = a.di;
    da.scores = scores; da.ld_s = lay.ld_s; da.hist = hist;
    da.row_tickets = reinterpret_cast<unsigned*>(wsb + lay.row_tickets_off); da.K = a.K;
    da.split = reinterpret_cast<sa::BinSplit*>(wsb + lay.split_off);
    if (sa::launch_decode_scan(da, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    if (a.stage_events && cudaEventRecord(a.stage_events[0], stream) != cudaSuccess) return SA_ERR_LAUNCH;

    sa::DecodeSelectArgs sa_{};
    sa_.scores = scores; sa_.ld_s = lay.ld_s; sa_.ctx_len = a.ctx_len;
    sa_.max_ctx = a.max_ctx; sa_.B = a.B; sa_.K = a.K; sa_.split = da.split;
    sa_.bitmap = reinterpret_cast<uint32_t*>(wsb + lay.bitmap_off); sa_.ld_w = lay.ld_w;
    sa_.cand = reinterpret_cast<unsigned long long*>(wsb + lay.cand_off); sa_.cand_cap = sa::DECODE_CAND_CAP;
    sa_.cand_cnt = cand_cnt; sa_.idx = idx;
    if (sa::launch_decode_select(sa_, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    if (a.stage_events && cudaEventRecord(a.stage_events[1], stream) != cudaSuccess) return SA_ERR_LAUNCH;

    sa::AttnArgs at{};
    at.q = a.q; at.k = a.k_cache; at.ld_k = a.ld_k; at.v = a.v_cache; at.ld_v = a.ld_v;
    at.v_aliases_k = (a.v_cache == a.k_cache) && a.ld_v == a.ld_k;
    at.row_base = a.seq_start; at.idx = idx; at.K = a.K; at.ctx_len = a.ctx_len;
    at.causal_first = 0; at.n_cap = a.max_ctx; at.gate = a.gate;
    at.rows = a.B; at.Hq = a.Hq; at.dqk = a.dqk; at.dv = a.dv;
    at.softmax_scale = a.softmax_scale; at.dtype = a.attn_dtype; at.out = a.out;
    at.splits = lay.splits; at.part = part; at.tickets = tickets; at.pdl = true;
    if (sa::launch_attention(at, stream) != cudaSuccess) return SA_ERR_LAUNCH;
    if (a.stage_events && cudaEventRecord(a.stage_events[2], stream) != cudaSuccess) return SA_ERR_LAUNCH;
    return SA_OK;
}

int sparse_attn_decode_host(const sa_decode_args* args, const void* host_in, void* dev_in, size_t in_bytes,
                            void* host_out, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    NvtxRange range("sparse_attn_decode_host");
    if (!host_in || !dev_in || !host_out || in_bytes == 0) return SA_ERR_INVALID_ARG;
    int st = check_decode(args);
    if (st != SA_OK) return st;
    const sa_decode_args& a = *args;
    if (a.B > 0) {
        const DecodeLayout lay = decode_layout(a);
        if (!ws || ws_bytes < lay.total || !aligned(ws, WS_ALIGN)) return SA_ERR_WORKSPACE;
    }
    if (cudaMemcpyAsync(dev_in, host_in, in_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return SA_ERR_LAUNCH;
    st = sparse_attn_decode(args, ws, ws_bytes, stream);
    if (st != SA_OK) return st;
    const size_t es = a.attn_dtype == SA_BF16 ? 2 : 4;
    const size_t out_bytes = (size_t)a.B * a.Hq * a.dv * es;
    if (out_bytes && cudaMemcpyAsync(host_out, a.out, out_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return SA_ERR_LAUNCH;
    return SA_OK;
}

}  // extern "C"
