// Internal launchers of the sparse attention library (host side). Arguments
// are validated by the C-ABI layer (api.cu) before any of these is called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace sa {

// 2D TMA descriptor of a row-major matrix of 1-, 2- or 4-byte elements
// (bytes, bf16, fp32); with swizzle, the box's row bytes (32, 64 or 128)
// pick the swizzle mode (else none).
bool make_tensor_map_2d(CUtensorMap* m, const void* base, int elem_bytes, int64_t rows, int64_t cols,
                        int64_t row_stride_elems, int box_cols, int box_rows, bool swizzle = true);
int device_sm_count();

// Kernel launch, optionally as a programmatic dependent of the previous work
// on the stream (the kernel must call griddep_wait() before touching data
// that work produces or reads).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// The same with thread-block clusters of cluster.x * cluster.y * cluster.z CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                  dim3 cluster, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster.x;
    attr[0].val.clusterDim.y = cluster.y;
    attr[0].val.clusterDim.z = cluster.z;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// Zeroes `bytes` (a multiple of 16) at p; first kernel of the decode step.
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s);

// ---- step 1: indexer (prefill / shared keys) ------------------------------
struct IndexerArgs {
    const void* q_idx;      // [T, Hi, di]
    int dtype;              // SA_F32 / SA_BF16 / SA_FP8_E4M3
    const float* q_scale;   // [T, Hi] or null
    const float* w;         // [T, Hi]
    const void* k_idx;      // [N, di]
    const float* k_scale;   // [N] or null
    int T, N, Hi, di;
    int64_t causal_offset;  // n_t = clamp(t + 1 + causal_offset, 0, N)
    int t_begin;            // first query row handled (rows t_begin .. T-1)
    float* scores;          // row t at scores + (t - t_begin) * ld_s
    int64_t ld_s;
    // sampled keys: k_idx row i is the key sampled from stratum i (see
    // sample_pos); then n_t = min(N, sample_count(t)) instead of the causal n_t
    int sample_log2;        // 0: off
    // pooled keys: k_idx row b is the mean of positions [b 2^lg, (b+1) 2^lg);
    // then n_t = min(N, (t >> lg) + 1): every block holding a visible position
    int block_log2;         // 0: off
    // filter mode (thr != null): no score is stored; a (query t, key j) pair
    // with score_key(s) >= thr[t - t_begin] is appended, as the pair
    // (float bits of s << 32 | ~j), to the segment of its work item: segment g of
    // row r holds seg_cnt[r * nseg + g] entries (its true count, possibly above
    // cap_seg, in which case only cap_seg were kept) at
    // seg_cand + (r * nseg + g) * cap_seg
    const uint32_t* thr;
    unsigned* seg_cnt;
    unsigned long long* seg_cand;
    int nseg, cap_seg;
};

// ---- stratified key sample -------------------------------------------------
// One key per stratum of 2^lg consecutive positions, at a pseudo-random offset
// inside it: offset(i) = fmix32(i ^ SAMPLE_SEED) mod 2^lg, fmix32 being the
// MurmurHash3 32-bit finaliser. A stratified sample keeps every key's
// inclusion probability at 2^-lg whatever the structure of the positions.
constexpr uint32_t SAMPLE_SEED = 0x9E3779B9u;
__host__ __device__ inline uint32_t fmix32(uint32_t h)
{
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}
__host__ __device__ inline int64_t sample_pos(int64_t i, int lg)
{
    return (i << lg) + (int64_t)(fmix32((uint32_t)i ^ SAMPLE_SEED) & ((1u << lg) - 1u));
}
// number of sampled positions <= t
__host__ __device__ inline int64_t sample_count(int64_t t, int lg)
{
    if (t < 0) return 0;
    const int64_t full = (t + 1) >> lg;                      // strata wholly <= t
    const int64_t part = (t + 1) & ((int64_t(1) << lg) - 1);  // positions of the next one <= t
    return full + ((int64_t)(fmix32((uint32_t)full ^ SAMPLE_SEED) & ((1u << lg) - 1u)) < part ? 1 : 0);
}
// keys visible to query row t
__host__ __device__ inline int64_t indexer_row_n(const IndexerArgs& a, int64_t t)
{
    const int64_t n = a.sample_log2 ? sample_count(t, a.sample_log2)
                    : a.block_log2 ? (t < 0 ? 0 : (t >> a.block_log2) + 1) : t + 1 + a.causal_offset;
    return n < 0 ? 0 : (n > a.N ? a.N : n);
}
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s);        // picks one of:
cudaError_t launch_indexer_simt(const IndexerArgs& a, cudaStream_t s);   // any dtype/shape, CUDA cores
cudaError_t launch_indexer_tc(const IndexerArgs& a, cudaStream_t s);     // bf16 / FP8, tensor cores
bool indexer_tc_supported(const IndexerArgs& a);

cudaError_t indexer_device_errors(unsigned* bits, bool reset);   // the tensor-core indexer's error word
int indexer_filter_lcap(const IndexerArgs& a);   // pairs per query and work item in filter mode; 0: none
int indexer_query_tile(const IndexerArgs& a);    // queries per tensor-core tile (256 / Hi)
constexpr int INDEXER_GROUP = 8;                 // key tiles (of 128) per tensor-core work item

// ---- steps 1+2 fused for long causal rows -----------------------------------
struct FusedSelectArgs {
    int64_t t_begin;        // rows t_begin .. t_begin + rows - 1, n_t = min(t + 1, N)
    int rows;
    int64_t N;
    int K;
    int tq, group;          // the filter pass's query-tile height and key tiles per item
    int sample_log2;
    int64_t ns;             // sampled keys
    uint32_t* thr;          // [rows] threshold keys
    const unsigned* seg_cnt;            // [rows][nseg]
    const unsigned long long* seg_cand; // [rows][nseg][cap_seg]
    int nseg, cap_seg;
    int cand_cap;           // pairs of one row staged in shared memory
    int64_t words;          // bitmap words of the longest row
    int32_t* idx;           // row r at idx + r * ld_idx
    int64_t ld_idx;
    unsigned* fail_cnt;     // zeroed before the select
    int* fail_list;         // [rows]
    IndexerArgs ia;         // the full indexer problem (fallback rows are rescored from it)
    float* scratch;         // fallback score rows: row r at scratch + r * ld_scratch
    int64_t ld_scratch;
};
cudaError_t launch_sample_gather(const void* k_idx, int row_bytes, const float* k_scale, int64_t ns, int lg,
                                 void* ksamp, float* ksamp_scale, cudaStream_t s);
size_t fused_threshold_smem(int64_t max_samples);
cudaError_t launch_sample_threshold(const FusedSelectArgs& a, const float* ssc, int64_t ld_ssc, int64_t max_samples,
                                    cudaStream_t s);
size_t fused_select_smem(const FusedSelectArgs& a);
cudaError_t launch_fused_select(const FusedSelectArgs& a, cudaStream_t s);   // select + fallback

// ---- block-granular selection -----------------------------------------------
// mean of each block of 2^lg consecutive key rows (bf16 in, bf16 out, fp32 sum)
cudaError_t launch_pool_keys(const void* k_idx, int64_t N, int di, int lg, void* pooled, cudaStream_t s);
// n_r = ((t0 + r) >> lg) + 1 for rows r < rows
cudaError_t launch_block_rowlen(int64_t t0, int rows, int lg, int32_t* row_len, cudaStream_t s);
// selected blocks (ascending, -1 padded, Kb per row) -> their positions <= t,
// ascending, -1 padded, Kb << lg per row; count[r] = positions written
cudaError_t launch_expand_blocks(const int32_t* blk, int Kb, int64_t t0, int rows, int lg, int32_t* idx,
                                 int32_t* count, cudaStream_t s);

// ---- dense causal attention (the full-attention control branch) ------------
struct DenseArgs {
    const void* q;           // [L, Hq, D] bf16
    const void* k;           // row j at k + j * ld_k
    int64_t ld_k;
    const void* v;
    int64_t ld_v;
    const float* gate;       // [L, Hq]
    void* out;               // [L, Hq, D] bf16
    int64_t L;
    int Hq, D;
    float softmax_scale;
    // optional kept-position mask: rows t >= mask_from attend only to the
    // positions listed in idx[t * K .. t * K + K) (all <= t); null = dense
    const int32_t* idx;
    int K;
    int64_t mask_from;
};
bool attention_dense_supported(const DenseArgs& a);
cudaError_t launch_attention_dense(const DenseArgs& a, cudaStream_t s);   // tcgen05 where it applies
bool attention_dense_tc_supported(const DenseArgs& a);                     // d = 128, 16 heads
cudaError_t launch_attention_dense_tc(const DenseArgs& a, cudaStream_t s);
cudaError_t attention_dense_tc_device_errors(unsigned* bits, bool reset);

// ---- sliding-window local branch ---------------------------------------------
// idx[r] = positions max(0, t - W + 1) .. t (t = t0 + r), ascending, W per row
// (-1 padded); kept[r] = their count
cudaError_t launch_window_idx(int64_t t0, int rows, int W, int32_t* idx, int32_t* kept, cudaStream_t s);
// neg[i] = -x[i] (sigmoid(-x) = 1 - sigmoid(x))
cudaError_t launch_negate(const float* x, float* neg, int64_t n, cudaStream_t s);
// out[i] = round(out[i] + add[i]) for n bf16 elements (fp32 sum)
cudaError_t launch_add_bf16(void* out, const void* add, int64_t n, cudaStream_t s);

// ---- gradients of steps 3-4 over a fixed index set -------------------------
struct BwdArgs {
    int L, Hq, D, K, dtype;  // D = dqk = dv
    float softmax_scale;
    const void* q;           // [L, Hq, D]
    const void* k;           // row j at k + j * ld_k
    int64_t ld_k;
    const void* v;
    int64_t ld_v;
    const int32_t* idx;      // [L, K], < 0 = none
    const float* gate;       // [L, Hq]
    const void* dout;        // [L, Hq, D]
    float* dq;               // [L, Hq, D]
    float* dk;               // [L, D]
    float* dv;               // [L, D]
    float* dgate;            // [L, Hq]
};
bool attention_backward_supported(const BwdArgs& a);
cudaError_t launch_attention_backward(const BwdArgs& a, cudaStream_t s);      // picks one of:
bool attention_backward_tc_supported(const BwdArgs& a);                        // bf16, tensor cores
cudaError_t launch_attention_backward_tc(const BwdArgs& a, cudaStream_t s);   // (dk, dv zeroed by the caller)

// ---- step 2: Top-K over score rows -----------------------------------------
struct TopkArgs {
    const float* scores;    // row r at scores + r * ld_s
    int64_t ld_s;
    const int32_t* row_len; // [rows] or null: then n_r = clamp(causal_first + r + 1, 0, n_cap)
    int64_t causal_first;
    int64_t n_cap;          // upper clamp of every row length
    int rows, K;
    int32_t* idx;           // row r at idx + r * ld_idx
    int64_t ld_idx;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);

// ---- steps 3-4: gathered attention + gate ----------------------------------
struct AttnArgs {
    const void* q;          // [rows, Hq, dqk]
    const void* k;          // key row p at k + (base + p) * ld_k
    int64_t ld_k;
    const void* v;          // value row p at v + (base + p) * ld_v
    int64_t ld_v;
    bool v_aliases_k;       // v == k (latent row): values read from the key tile
    const int64_t* row_base;  // [rows] first packed row per query row, or null (0)
    const int32_t* idx;     // [rows, K] kept positions, ascending, -1 padded
    int K;
    const int32_t* ctx_len; // [rows] history length per row, or null: n = causal_first + r + 1
    const int32_t* kept_len;  // [rows] kept entries per row, or null: min(K, n)
    int64_t causal_first;
    int64_t n_cap;
    const float* gate;      // [rows, Hq]
    int rows, Hq, dqk, dv;
    float softmax_scale;
    int dtype;              // SA_F32 / SA_BF16
    void* out;              // [rows, Hq, dv]
    // split-K (decode): > 1 splits the kept rows across CTAs and merges
    int splits;
    float* part;            // [rows, splits, Hq, dv + 2]
    unsigned* tickets;      // [rows], zero on entry, left zero on exit
    int stages;             // set by the launcher: gather buffers (1 or 2)
    bool pdl;               // launch as a programmatic dependent of the previous kernel
};
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s);          // picks one of:
int set_prefill_attention_kernel(int which);          // SA_ATTN_*; returns the previous choice
bool attention_tc_supported(const AttnArgs& a);       // prefill rows on tcgen05, d = 128
cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t s);
cudaError_t attention_tc_device_errors(unsigned* bits, bool reset);   // its bounded-wait error word
bool attention_gather_supported(const AttnArgs& a);   // cp.async gathers + mma.sync, d = 64 or 128
cudaError_t launch_attention_gather(const AttnArgs& a, cudaStream_t s);
int attention_splits(int K, int64_t n_cap, int rows, bool gather_kernel);

// Bin of the K-th best score of a row, from a 4096-bin histogram of the top
// 12 bits of the scores' order-preserving keys.
struct BinSplit {
    int bin;            // bin of the K-th best key
    unsigned above;     // keys in higher bins (< K)
    unsigned in_bin;    // keys in that bin (above + in_bin >= K)
};

// ---- decode step 1: indexer scan over each sequence's cache --------------
struct DecodeScanArgs {
    const void* q_idx;      // [B, Hi, di] bf16, or e4m3 codes when fp8
    const float* w;         // [B, Hi]
    const void* k_idx;      // packed [rows, di] bf16, or e4m3 codes when fp8
    int fp8;                // e4m3 inputs: q_scale [B, Hi] and k_scale [rows] fp32
    const float* q_scale;
    const float* k_scale;
    const int64_t* seq_start;
    const int32_t* ctx_len;
    int64_t max_ctx;
    int B, Hi, di;
    float* scores;          // [B, ld_s]
    int64_t ld_s;           // a multiple of 128 (rows 512-byte aligned)
    unsigned* hist;         // [B, 4096] key-bin histogram, zero on entry
    unsigned* row_tickets;  // [B], zero on entry
    int K;
    BinSplit* split;        // [B] bin of the K-th best score (rows with n > K)
    int chunk;              // keys per chunk (set by the launcher)
    int b_begin, nb;        // rows of one launch (set by the launcher)
};
cudaError_t launch_decode_scan(const DecodeScanArgs& a, cudaStream_t s);

// ---- decode step 2: Top-K of each sequence's score row --------------------
struct DecodeSelectArgs {
    const float* scores;    // [B, ld_s], ld_s a multiple of 32
    int64_t ld_s;
    const int32_t* ctx_len;
    int64_t max_ctx;
    int B, K;
    const BinSplit* split;  // [B] from the scan
    uint32_t* bitmap;       // [B, ld_w] kept-position bits
    int64_t ld_w;
    unsigned long long* cand;   // [B, cand_cap] (key << 32 | ~position) of the threshold bin
    int cand_cap;
    unsigned* cand_cnt;     // [B], zero on entry
    int32_t* idx;           // [B, K]
};
cudaError_t launch_decode_select(const DecodeSelectArgs& a, cudaStream_t s);
constexpr int DECODE_CAND_CAP = 16384;

}  // namespace sa
