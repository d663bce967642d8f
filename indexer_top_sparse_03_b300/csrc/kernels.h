// Internal launchers of the sparse attention library (host side). Arguments
// are validated by the C-ABI layer (api.cu) before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sa {

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
};
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s);

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
};
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s);
int attention_splits(int K, int64_t n_cap, int rows);

// ---- decode step 1: indexer scan over each sequence's cache --------------
struct DecodeScanArgs {
    const void* q_idx;      // [B, Hi, di] bf16
    const float* w;         // [B, Hi]
    const void* k_idx;      // packed [rows, di] bf16
    const int64_t* seq_start;
    const int32_t* ctx_len;
    int64_t max_ctx;
    int B, Hi, di;
    float* scores;          // [B, max_ctx]
    unsigned* tickets;      // [B] zeroed here for the attention combine
};
cudaError_t launch_decode_scan(const DecodeScanArgs& a, cudaStream_t s);

}  // namespace sa
