/*
 * sparse_attn.h -- C ABI of the B300 (sm_103a) gated sparse attention library.
 *
 * The layer ("Hybrid Attention Architectures: Engineering Trade-offs from
 * Linear Attention to Gated Sparse Attention", section 3.1 and the pseudocode
 * of section 3.3; "From Full Attention to Sparsity", section "Fine-Grained
 * Sparse Attention: Indexer Plus Top-K"):
 *   1. a light indexer scores every causal history position of each query,
 *        s[t,j] = sum_h w[t,h] * max(0, q_idx[t,h,:] . k_idx[j,:])
 *      (no positional encoding, no scale, no bias; the pages leave the
 *      formula open and this is the reading the library implements);
 *   2. Top-K keeps the K highest-scoring positions, an exact tie going to
 *      the lower position; a query with n <= K history positions keeps all n;
 *   3. exact softmax attention runs over the kept key/value rows only;
 *   4. a sigmoid output gate scales each (token, head) output:
 *        out[t,h,:] = sigmoid(gate[t,h]) * attn[t,h,:]
 *      (section 3.3 returns gate * attn_out; output gating, "Sparse Attention
 *      and Hybrid Attention Architecture Design", section 4).
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument named as a tensor is a DEVICE pointer unless its
 *     comment says host. Tensors are dense and row-major unless a row stride
 *     (ld_*) in elements is given. The caller owns every buffer, including the
 *     workspace; the library allocates no device memory and keeps no state
 *     between calls.
 *   - Work is enqueued on `stream` and never synchronised: results are ready
 *     when the stream reaches them. Calls on different streams that share a
 *     workspace race.
 *   - Return value: SA_OK (0) or a negative sa_status. Argument errors are
 *     found on the host before anything is enqueued, so a failed call leaves
 *     the outputs untouched. SA_ERR_LAUNCH reports a CUDA error seen right
 *     after a launch (cudaGetLastError), which may also stem from earlier
 *     asynchronous work on the device.
 *   - Floating point: products are accumulated in fp32; softmax and the gate
 *     are evaluated in fp32; outputs are rounded to nearest-even into the
 *     attention dtype. NaN or infinite inputs give unspecified results.
 *   - FP8 means e4m3 ("fn": no infinities) codes with one fp32 scale per
 *     row; the element's value is code * scale and scales must be positive.
 */
#ifndef SPARSE_ATTN_H
#define SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SA_API __attribute__((visibility("default")))
#else
#define SA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SA_OK = 0,
    SA_ERR_INVALID_ARG = -1,  /* null pointer, negative size, bad stride ... */
    SA_ERR_UNSUPPORTED = -2,  /* valid, but a dtype/shape this build lacks   */
    SA_ERR_WORKSPACE = -3,    /* workspace missing or smaller than required  */
    SA_ERR_LAUNCH = -4        /* a CUDA error right after a launch           */
} sa_status;

typedef enum {
    SA_F32 = 0,          /* IEEE binary32                                    */
    SA_BF16 = 1,         /* bfloat16                                         */
    SA_FP8_E4M3 = 2      /* e4m3 codes + fp32 per-row scales (indexer only)  */
} sa_dtype;

/* Human-readable name of a status code (static storage, never NULL). */
SA_API const char* sa_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
SA_API int sa_version(void);

/*
 * Device-side error bits of the current GPU, ORed since the last reset:
 * SA_DEVERR_WAIT_TIMEOUT = a bounded wait of a tensor-core kernel (the
 * indexer, or the prefill attention) gave up (its outputs are then
 * incomplete; the kernel returned instead of hanging).
 * Synchronises the device. *bits receives the word; reset != 0 clears it.
 * Returns SA_OK or SA_ERR_LAUNCH (the copy failed).
 */
#define SA_DEVERR_WAIT_TIMEOUT 1u
SA_API int sa_device_errors(unsigned* bits, int reset);

/*
 * Kernel for the gathered attention of prefill rows (the exact attention
 * over the kept rows, "Hybrid Attention Architectures...", section 3.1):
 *   SA_ATTN_AUTO     (default) cp.async gathers into per-warp rings, S = Q K^T
 *                    and P V on mma.sync; at 16 query heads per key/value
 *                    head the gather, not the arithmetic, bounds it, and this
 *                    kernel hides the gather latency best;
 *   SA_ATTN_TCGEN05  the tensor-core kernel: tiles of 128 kept rows gathered
 *                    by eight warps into 128-byte-swizzled shared memory,
 *                    S^T and O^T accumulated in TMEM by tcgen05.mma; used
 *                    where it applies (bf16, dqk = dv = 128, Hq a multiple
 *                    of 16), else the default.
 * Process-wide, takes effect for later calls; returns the previous choice,
 * or SA_ERR_INVALID_ARG for an unknown value (the choice is unchanged).
 */
#define SA_ATTN_AUTO 0
#define SA_ATTN_TCGEN05 1
SA_API int sa_set_prefill_attention_kernel(int which);

/*
 * indexer_score -- step 1 alone (exposed for testing).
 *
 *   q_idx   [T, Hi, di]  query-side indexer vectors, dtype `dtype`
 *   q_scale [T, Hi] fp32 per-(token, head) scales; required iff FP8, else
 *           ignored
 *   w       [T, Hi] fp32 head weights (any sign)
 *   k_idx   [N, di]  key-side indexer vectors, dtype `dtype`
 *   k_scale [N] fp32 per-key scales; required iff FP8, else ignored
 *   scores  [T, ld_s] fp32 output, ld_s >= N. Row t is written at positions
 *           j < n_t = clamp(t + 1 + causal_offset, 0, N); positions j >= n_t
 *           are not written. causal_offset = 0 is causal self-attention over
 *           one sequence; causal_offset >= N - 1 scores every key.
 * Supported: dtype F32, BF16 or FP8_E4M3; 1 <= Hi <= 32; di a multiple of 16
 * in [16, 256]. T = 0 or N = 0 is a no-op.
 */
SA_API int indexer_score(const void* q_idx, int dtype, const float* q_scale, const float* w,
                  const void* k_idx, const float* k_scale,
                  int T, int N, int Hi, int di, int64_t causal_offset,
                  float* scores, int64_t ld_s, cudaStream_t stream);

/*
 * topk_select -- step 2 alone (exposed for testing).
 *
 *   scores  [T, ld_s] fp32; row t holds n_t = row_len[t] valid scores
 *   row_len [T] int32 device array; each value is clamped to [0, ld_s]
 *   idx_out [T, K] int32 output: the selected positions of row t in
 *           ascending order, min(K, n_t) of them, then -1 padding.
 * Selection keeps the K largest scores; among equal scores the lower position
 * wins; +0.0 and -0.0 compare equal. Rows with n_t <= K keep 0..n_t-1.
 * Supported: 1 <= K <= 65536, ld_s >= 1.
 */
SA_API int topk_select(const float* scores, int64_t ld_s, const int32_t* row_len, int T, int K,
                int32_t* idx_out, cudaStream_t stream);

/*
 * Causal prefill of one sequence of L tokens (token t attends within 0..t).
 * Attention uses Hq query heads sharing one key/value head (MQA).
 */
typedef struct {
    int L;                 /* tokens (queries == keys)                       */
    int Hq, dqk, dv;       /* query heads; q.k width; value width            */
    int Hi, di;            /* indexer heads and width                        */
    int K;                 /* positions kept per query                       */
    float softmax_scale;   /* logits are softmax_scale * q.k                  */
    int attn_dtype;        /* SA_F32 or SA_BF16: q, k, v and out             */
    int idx_dtype;         /* SA_F32, SA_BF16 or SA_FP8_E4M3: q_idx, k_idx   */
    const void* q;         /* [L, Hq, dqk]                                   */
    const void* k;         /* [L, ld_k], the first dqk columns are the key   */
    int64_t ld_k;
    const void* v;         /* [L, ld_v], the first dv columns are the value;
                              may alias k (latent row)                       */
    int64_t ld_v;
    const void* q_idx;     /* [L, Hi, di]                                    */
    const float* q_scale;  /* [L, Hi] (FP8 only)                             */
    const void* k_idx;     /* [L, di]                                        */
    const float* k_scale;  /* [L] (FP8 only)                                 */
    const float* w;        /* [L, Hi] indexer head weights                   */
    const float* gate;     /* [L, Hq] gate logits; sigmoid applied inside    */
    void* out;             /* [L, Hq, dv] in attn_dtype                      */
    int32_t* idx_out;      /* [L, K] selected positions (ascending, -1 pad),
                              or NULL to keep them in the workspace          */
    const cudaEvent_t* stage_events; /* NULL, or 2 events recorded on the
                              stream after selection (steps 1-2, every pass)
                              and after attention (steps 3-4)               */
} sa_prefill_args;

/* Workspace bytes sparse_attn_prefill needs for these arguments (0 on bad
 * arguments). Only the scalar fields are read. */
SA_API size_t sa_prefill_workspace_size(const sa_prefill_args* args);

/*
 * sparse_attn_prefill -- steps 1-4 for every token of one sequence.
 * ws: device workspace of at least sa_prefill_workspace_size(args) bytes,
 * 256-byte aligned; its contents on entry do not matter.
 * Supported: attn_dtype BF16 with dqk, dv multiples of 16 and <= 576 / 512,
 * or F32 with dqk, dv <= 256; 1 <= Hq <= 64; ld_k >= dqk, ld_v >= dv, both
 * multiples of 8; the indexer limits of indexer_score; 1 <= K <= 65536.
 */
SA_API int sparse_attn_prefill(const sa_prefill_args* args, void* ws, size_t ws_bytes,
                        cudaStream_t stream);

/*
 * sparse_attn_prefill with block-granular selection (the block-level routing
 * of "Sparse Attention and Hybrid Attention Architecture Design": keys are
 * mean-pooled per block, the indexer scores blocks, Top-K keeps blocks, and
 * exact attention runs inside the kept blocks). Blocks are block_size
 * consecutive positions (block b = positions [b*bs, (b+1)*bs)); the pooled
 * indexer key of a block is the mean of its k_idx rows rounded to bf16; query
 * t scores the blocks holding a visible position (b*bs <= t), keeps the
 * K / block_size best (ties: lower block), and attends over the positions
 * <= t of the kept blocks. idx_out, if not NULL, receives [L, K] kept
 * positions (ascending, -1 padded). With block_size 1 this is
 * sparse_attn_prefill.
 * Supported: idx_dtype SA_BF16; block_size a power of two in [1, 1024] that
 * divides K; the other limits of sparse_attn_prefill.
 */
SA_API size_t sa_prefill_blocks_workspace_size(const sa_prefill_args* args, int block_size);
SA_API int sparse_attn_prefill_blocks(const sa_prefill_args* args, int block_size, void* ws, size_t ws_bytes,
                                      cudaStream_t stream);

/*
 * sparse_attn_prefill fused with a sliding-window local branch (the branch
 * fusion of "Sparse Attention and Hybrid Attention Architecture Design":
 * out = g * sparse + (1 - g) * local, g = sigmoid(gate logit) per (token,
 * head)). sparse is the pre-gate output of sparse_attn_prefill; local is
 * exact attention of query t over positions max(0, t - window + 1) .. t.
 * Supported: attn_dtype SA_BF16, window >= 1; the limits of
 * sparse_attn_prefill. ws: at least sa_prefill_local_workspace_size bytes.
 */
SA_API size_t sa_prefill_local_workspace_size(const sa_prefill_args* args, int window);
SA_API int sparse_attn_prefill_local(const sa_prefill_args* args, int window, void* ws, size_t ws_bytes,
                                     cudaStream_t stream);

/*
 * Dense causal attention with the sigmoid output gate: query t attends over
 * every position 0..t (the full-attention layer the sparse one replaces;
 * "From Full Attention to Sparsity" measures the sparse layer against it:
 * sparse attention pays off once the indexer costs less than the attention
 * it saves). q [L, Hq, d], k rows [L, ld_k], v rows [L, ld_v], gate [L, Hq]
 * logits, out [L, Hq, d]. Supported: bf16, d in {64, 128}, 1 <= Hq <= 64,
 * ld_k, ld_v multiples of 8, 16-byte aligned q, k, v, out.
 */
SA_API int attention_dense_causal(const void* q, const void* k, int64_t ld_k, const void* v, int64_t ld_v,
                                  const float* gate, void* out, int L, int Hq, int d, float softmax_scale,
                                  cudaStream_t stream);

/*
 * One decode step for B sequences: the new query of sequence b attends over
 * its ctx_len[b] cached rows, stored at packed rows seq_start[b] ..
 * seq_start[b] + ctx_len[b] - 1 of the caches (append the new token's own
 * row first if it should be visible to itself).
 */
typedef struct {
    int B;                 /* sequences                                      */
    int Hq, dqk, dv;
    int Hi, di;
    int K;
    float softmax_scale;
    int attn_dtype;        /* SA_BF16                                        */
    int idx_dtype;         /* SA_BF16 or SA_FP8_E4M3                         */
    const void* q;         /* [B, Hq, dqk]                                   */
    const void* q_idx;     /* [B, Hi, di]                                    */
    const float* q_scale;  /* [B, Hi] positive row scales (FP8 only)         */
    const float* w;        /* [B, Hi]                                        */
    const float* gate;     /* [B, Hq] gate logits                            */
    const void* k_cache;   /* [rows, ld_k]: keys are the first dqk columns   */
    int64_t ld_k;
    const void* v_cache;   /* [rows, ld_v]: values are the first dv columns;
                              may alias k_cache (latent row)                 */
    int64_t ld_v;
    const void* k_idx_cache;  /* [rows, di] indexer keys                     */
    const float* k_idx_scale; /* [rows] positive row scales (FP8 only)       */
    const int64_t* seq_start; /* [B] device: first packed row of sequence b  */
    const int32_t* ctx_len;   /* [B] device: cached rows of sequence b,
                                 clamped to [0, max_ctx] on the device       */
    int64_t max_ctx;       /* host: an upper bound of every ctx_len[b]       */
    void* out;             /* [B, Hq, dv] in attn_dtype                      */
    int32_t* idx_out;      /* [B, K] selected positions within the sequence
                              (ascending, -1 pad), or NULL                   */
    const cudaEvent_t* stage_events; /* NULL, or 3 events recorded on the
                              stream after step 1 (indexer scan), after step 2
                              (Top-K) and after steps 3-4 (attention, gate);
                              stages fused into one kernel record together  */
} sa_decode_args;

/* Workspace bytes sparse_attn_decode needs (0 on bad arguments). */
SA_API size_t sa_decode_workspace_size(const sa_decode_args* args);

/*
 * sparse_attn_decode -- steps 1-4 for one new token of each sequence, with the
 * attention over the K kept rows split across CTAs and merged by a
 * log-sum-exp combine.
 * ws: device workspace of at least sa_decode_workspace_size(args) bytes,
 * 256-byte aligned; its contents on entry do not matter.
 * Supported: attn_dtype BF16 with dqk, dv multiples of 16, dqk <= 576,
 * dv <= 512; 1 <= Hq <= 64; idx_dtype BF16 with 1 <= Hi <= 32 and di a
 * multiple of 32 in [32, 256], or idx_dtype FP8_E4M3 (e4m3 codes, value =
 * code * row scale; q_scale and k_idx_scale required, 4-byte aligned) with di
 * a multiple of 64 in [64, 256]: the FP8 score is
 * k_idx_scale[j] * sum_h w[b,h] q_scale[b,h] max(0, q8 . k8), as in
 * indexer_score; ld_k, ld_v multiples of 8; 1 <= K <= 65536;
 * 0 <= max_ctx < 2^31.
 */
SA_API int sparse_attn_decode(const sa_decode_args* args, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/*
 * sparse_attn_decode_host -- one decode step whose per-step inputs come from
 * host memory and whose output goes back to host memory, all on `stream`:
 * in_bytes bytes are copied from host_in to dev_in (the caller packs the
 * step's inputs there: args->q, q_idx, w, gate and, for FP8, q_scale point
 * into dev_in, which must hold in_bytes bytes), then sparse_attn_decode runs,
 * then args->out (B * Hq * dv elements of attn_dtype) is copied to host_out.
 * Asynchronous: the caller waits on the stream (or an event recorded after
 * this call) before reading host_out or rewriting host_in. Page-locked host
 * buffers make the copies asynchronous; pageable ones work but block.
 * Errors: SA_ERR_INVALID_ARG for null host_in / dev_in / host_out or
 * in_bytes == 0, else those of sparse_attn_decode (checked before anything
 * is enqueued); SA_ERR_LAUNCH if a copy cannot be enqueued.
 */
SA_API int sparse_attn_decode_host(const sa_decode_args* args, const void* host_in, void* dev_in, size_t in_bytes,
                                   void* host_out, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Gradients of steps 3-4 over a fixed index set (the training path:
 * "Hybrid Attention Architectures...", section 3.1 -- once the indexer has
 * chosen the set, attention over it is ordinary softmax attention -- and
 * section 3.3 -- the gate scales its output). For query row t of one causal
 * sequence, with the positions idx[t, :] (entries < 0 skipped; the kept
 * positions sparse_attn_prefill returns), l_i = softmax_scale * q_h . k_i,
 * p = softmax(l), o_h = sum_i p_i v_i, out_h = sigmoid(gate_h) o_h, the call
 * returns the derivatives of sum(dout * out):
 *   dq [L, Hq, dqk], dgate [L, Hq] (with respect to the gate logits), and
 *   dk [L, dqk], dv [L, dv]: each key / value row's total over every query
 *   that selected it (overwritten; accumulated on the GPU in fp32 in an
 *   order that varies from run to run).
 * All outputs are fp32. Supported: dtype SA_BF16 or SA_F32 (q, k, v, dout),
 * dqk == dv in {64, 128}, 1 <= Hq <= 16, ld_k >= dqk, ld_v >= dv (multiples
 * of 8), v may alias k; 1 <= K <= 65536. The caller owns every buffer; the
 * call allocates nothing and needs no workspace. Errors: SA_ERR_INVALID_ARG
 * (null or misaligned pointers, bad sizes), SA_ERR_UNSUPPORTED (shapes above),
 * SA_ERR_LAUNCH.
 */
typedef struct {
    int L;                 /* query rows = key rows of the sequence           */
    int Hq, dqk, dv;
    int K;                 /* entries per row of idx                          */
    int dtype;             /* SA_BF16 or SA_F32                               */
    float softmax_scale;
    const void* q;         /* [L, Hq, dqk]                                    */
    const void* k;         /* [L, ld_k]                                       */
    int64_t ld_k;
    const void* v;         /* [L, ld_v]                                       */
    int64_t ld_v;
    const int32_t* idx;    /* [L, K] kept positions of each row, -1 = none    */
    const float* gate;     /* [L, Hq] gate logits                             */
    const void* dout;      /* [L, Hq, dv] gradient of the layer output        */
    float* dq;             /* [L, Hq, dqk]                                    */
    float* dk;             /* [L, dqk]                                        */
    float* dv_out;         /* [L, dv]                                         */
    float* dgate;          /* [L, Hq]                                         */
} sa_backward_args;

SA_API int sparse_attn_backward(const sa_backward_args* args, cudaStream_t stream);

/* Bytes of device scratch the library carries for sparse_attn_decode_noalloc. */
#define SA_DECODE_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * sparse_attn_decode_noalloc -- sparse_attn_decode for callers that cannot
 * allocate device memory (plugins whose host owns every allocation, code that
 * must not allocate once serving has started). The paper has no counterpart:
 * this is a deployment convenience, not part of the layer.
 *
 * Same arguments, kernels and results as sparse_attn_decode, but the scratch
 * lives in a fixed array of SA_DECODE_NOALLOC_SCRATCH_BYTES inside the
 * library, held on every GPU that loads the library until the process exits.
 * Calls whose sa_decode_workspace_size(args) exceeds that size return
 * SA_ERR_WORKSPACE and enqueue nothing. Nothing is allocated. All calls share
 * the array, which keeps the previous call's contents (the step clears what
 * must start at zero); calls whose GPU work overlaps (other streams or host
 * threads) race and give wrong results. The first call on each device looks
 * up the array's device address; make it before any stream capture begins.
 */
SA_API int sparse_attn_decode_noalloc(const sa_decode_args* args, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H */
