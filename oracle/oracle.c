/*
 * fp64 CPU oracle for the gated sparse attention layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file: only tests/, the package smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header, table or constant with the
 * CUDA library, and it never reads a value the CUDA library produced.
 *
 * What it computes is the plain definition of the layer described on
 * "Hybrid Attention Architectures: Engineering Trade-offs from Linear Attention
 * to Gated Sparse Attention", section 3.1 (score every history position,
 * keep the K highest, exact attention over that candidate set only) and
 * section 3.3 (the gate scales the attention output), with the indexer
 * carrying no positional encoding ("From Full Attention to Sparsity",
 * section "Fine-Grained Sparse Attention: Indexer Plus Top-K").
 *
 * The pages give no formula for the indexer. The one used is
 *     s[r, j] = sum_h w[r, h] * max(0, sum_d q_idx[r, h, d] * k_idx[j, d])
 * with no scale and no bias. Every step below is evaluated in IEEE double
 * precision, one row at a time, in the order the definition states; the only
 * library routines used are qsort and exp.
 *
 * Stored formats are decoded here from their bit-level definitions:
 *   f32  : IEEE binary32 (exact in double)
 *   bf16 : the upper 16 bits of an IEEE binary32 (exact in double)
 *   e4m3 : 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no
 *          infinities, S.1111.111 is NaN (the "fn" variant); the value
 *          times its fp32 scale is exact in double (4 + 24 significant bits).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_E4M3 = 2 };

/* ------------------------------------------------------------------ */
/* decoding of the stored element formats                             */
/* ------------------------------------------------------------------ */

double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_f64(uint8_t bits)
{
    int sign = bits >> 7;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9); /* subnormal: (m/8) * 2^(1-7) */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

static double load_elem(const void* base, int dtype, int64_t i)
{
    switch (dtype) {
    case OR_F32: return (double)((const float*)base)[i];
    case OR_BF16: return oracle_bf16_to_f64(((const uint16_t*)base)[i]);
    case OR_E4M3: return oracle_e4m3_to_f64(((const uint8_t*)base)[i]);
    default: return NAN;
    }
}

/* ------------------------------------------------------------------ */
/* a tiny row-parallel runner                                          */
/* ------------------------------------------------------------------ */

typedef void (*row_fn)(void* ctx, int64_t row);

typedef struct {
    row_fn fn;
    void* ctx;
    int64_t nrows;
    int tid, nthreads;
} worker_arg;

static void* worker_main(void* p)
{
    worker_arg* a = (worker_arg*)p;
    for (int64_t r = a->tid; r < a->nrows; r += a->nthreads)
        a->fn(a->ctx, r);
    return NULL;
}

static int resolve_threads(int nthreads, int64_t nrows)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > nrows) nthreads = (int)(nrows > 0 ? nrows : 1);
    return nthreads;
}

static void run_rows(row_fn fn, void* ctx, int64_t nrows, int nthreads)
{
    nthreads = resolve_threads(nthreads, nrows);
    if (nthreads == 1) {
        for (int64_t r = 0; r < nrows; ++r) fn(ctx, r);
        return;
    }
    pthread_t th[256];
    worker_arg args[256];
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn; args[t].ctx = ctx; args[t].nrows = nrows;
        args[t].tid = t; args[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, worker_main, &args[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* the number of threads a call with this many rows would use */
int oracle_threads_used(int nthreads, int64_t nrows)
{
    return resolve_threads(nthreads, nrows);
}

/* ------------------------------------------------------------------ */
/* indexer score                                                       */
/* ------------------------------------------------------------------ */
/*
 * For task r: query row qrow[r] of q_idx ([*, Hi, di]) and w ([*, Hi]) is
 * scored against keys key_start[r] .. key_start[r] + n[r] - 1 of k_idx
 * ([*, di]); the n[r] scores go to out[out_off[r] + j].
 * FP8 inputs carry one fp32 scale per (query row, head) and one per key row;
 * the element value is code * scale (NULL scales mean 1).
 */
typedef struct {
    const void* q_idx; int dtype; const float* q_scale; const float* w;
    const void* k_idx; const float* k_scale;
    int Hi, di;
    const int64_t *qrow, *key_start, *n, *out_off;
    double* out;
} indexer_ctx;

static void indexer_row(void* p, int64_t r)
{
    indexer_ctx* c = (indexer_ctx*)p;
    const int Hi = c->Hi, di = c->di;
    const int64_t t = c->qrow[r];
    double* q = (double*)malloc(sizeof(double) * (size_t)Hi * di);
    double* wt = (double*)malloc(sizeof(double) * (size_t)Hi);
    for (int h = 0; h < Hi; ++h) {
        double qs = c->q_scale ? (double)c->q_scale[t * Hi + h] : 1.0;
        for (int d = 0; d < di; ++d)
            q[h * di + d] = load_elem(c->q_idx, c->dtype, (t * Hi + h) * (int64_t)di + d) * qs;
        wt[h] = (double)c->w[t * Hi + h];
    }
    for (int64_t j = 0; j < c->n[r]; ++j) {
        const int64_t kr = c->key_start[r] + j;
        const double ks = c->k_scale ? (double)c->k_scale[kr] : 1.0;
        double s = 0.0;
        for (int h = 0; h < Hi; ++h) {
            double dot = 0.0;
            for (int d = 0; d < di; ++d)
                dot += q[h * di + d] * (load_elem(c->k_idx, c->dtype, kr * (int64_t)di + d) * ks);
            s += wt[h] * (dot > 0.0 ? dot : 0.0);
        }
        c->out[c->out_off[r] + j] = s;
    }
    free(q);
    free(wt);
}

int oracle_indexer(const void* q_idx, int dtype, const float* q_scale, const float* w,
                   const void* k_idx, const float* k_scale, int Hi, int di,
                   int64_t ntasks, const int64_t* qrow, const int64_t* key_start,
                   const int64_t* n, const int64_t* out_off, double* out, int nthreads)
{
    if (dtype < OR_F32 || dtype > OR_E4M3 || Hi <= 0 || di <= 0) return -1;
    indexer_ctx c = { q_idx, dtype, q_scale, w, k_idx, k_scale, Hi, di,
                      qrow, key_start, n, out_off, out };
    run_rows(indexer_row, &c, ntasks, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Top-K                                                               */
/* ------------------------------------------------------------------ */
/*
 * For task r the scores s[s_off[r] .. s_off[r] + n[r] - 1] are ranked by
 * (score descending, position ascending) and the first min(K, n[r]) positions
 * go to idx[r*K ...] in that order; the rest of the K slots hold -1.
 * Keeping "the K highest-scoring positions" is section 3.1 of the first page;
 * the lower position wins an exact tie.
 */
typedef struct { double s; int64_t j; } scored_pos;

static int by_score_then_pos(const void* a, const void* b)
{
    const scored_pos* x = (const scored_pos*)a;
    const scored_pos* y = (const scored_pos*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

typedef struct {
    const double* s; const int64_t *s_off, *n; int K; int32_t* idx;
} topk_ctx;

static void topk_row(void* p, int64_t r)
{
    topk_ctx* c = (topk_ctx*)p;
    const int64_t n = c->n[r];
    int32_t* out = c->idx + r * (int64_t)c->K;
    scored_pos* a = (scored_pos*)malloc(sizeof(scored_pos) * (size_t)(n > 0 ? n : 1));
    for (int64_t j = 0; j < n; ++j) {
        a[j].s = c->s[c->s_off[r] + j];
        a[j].j = j;
    }
    qsort(a, (size_t)n, sizeof(scored_pos), by_score_then_pos);
    for (int64_t k = 0; k < c->K; ++k)
        out[k] = k < n ? (int32_t)a[k].j : -1;
    free(a);
}

int oracle_topk(const double* s, int64_t ntasks, const int64_t* s_off, const int64_t* n,
                int K, int32_t* idx, int nthreads)
{
    if (K <= 0) return -1;
    for (int64_t r = 0; r < ntasks; ++r)
        for (int64_t j = 0; j < n[r]; ++j)
            if (!isfinite(s[s_off[r] + j])) return -2;
    topk_ctx c = { s, s_off, n, K, idx };
    run_rows(topk_row, &c, ntasks, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* exact attention over a supplied index set, then the sigmoid gate    */
/* ------------------------------------------------------------------ */
/*
 * For task r, query row qrow[r] of q ([*, Hq, dqk]) attends, per head h,
 * over the key rows key_start[r] + idx[r*K + i] for every slot i whose index
 * is >= 0 (slots holding -1 are skipped; a slot may not repeat a position).
 * Key row p supplies k = k_cache[p*ld_k + 0 .. dqk-1] and
 * v = v_cache[p*ld_v + 0 .. dv-1] (v may alias k: the latent layout).
 *   l_i = scale * q.k_i, m = max l, p_i = exp(l_i - m) / sum exp(l - m),
 *   o = sum p_i v_i, g = 1 / (1 + exp(-gate[qrow, h])), out = g * o.
 * pre (if not NULL) receives o before the gate, out receives g * o, both
 * [ntasks, Hq, dv] doubles.
 */
typedef struct {
    const void* q; int dtype; int Hq, dqk, dv;
    const void* kc; int64_t ld_k; const void* vc; int64_t ld_v;
    const int64_t *qrow, *key_start; const int32_t* idx; int K;
    double scale; const float* gate;
    double *out, *pre;
} attend_ctx;

static void attend_row(void* p, int64_t r)
{
    attend_ctx* c = (attend_ctx*)p;
    const int64_t t = c->qrow[r];
    const int32_t* sel = c->idx + r * (int64_t)c->K;
    double* logit = (double*)malloc(sizeof(double) * (size_t)c->K);
    double* q = (double*)malloc(sizeof(double) * (size_t)c->dqk);
    double* o = (double*)malloc(sizeof(double) * (size_t)c->dv);
    for (int h = 0; h < c->Hq; ++h) {
        for (int d = 0; d < c->dqk; ++d)
            q[d] = load_elem(c->q, c->dtype, (t * c->Hq + h) * (int64_t)c->dqk + d);
        double m = -INFINITY;
        for (int i = 0; i < c->K; ++i) {
            if (sel[i] < 0) continue;
            const int64_t kr = c->key_start[r] + sel[i];
            double dot = 0.0;
            for (int d = 0; d < c->dqk; ++d)
                dot += q[d] * load_elem(c->kc, c->dtype, kr * c->ld_k + d);
            logit[i] = c->scale * dot;
            if (logit[i] > m) m = logit[i];
        }
        double denom = 0.0;
        for (int e = 0; e < c->dv; ++e) o[e] = 0.0;
        for (int i = 0; i < c->K; ++i) {
            if (sel[i] < 0) continue;
            const int64_t kr = c->key_start[r] + sel[i];
            const double pi = exp(logit[i] - m);
            denom += pi;
            for (int e = 0; e < c->dv; ++e)
                o[e] += pi * load_elem(c->vc, c->dtype, kr * c->ld_v + e);
        }
        const double g = 1.0 / (1.0 + exp(-(double)c->gate[t * c->Hq + h]));
        double* dst = c->out + (r * c->Hq + h) * (int64_t)c->dv;
        double* pdst = c->pre ? c->pre + (r * c->Hq + h) * (int64_t)c->dv : NULL;
        for (int e = 0; e < c->dv; ++e) {
            const double oe = denom > 0.0 ? o[e] / denom : 0.0;
            if (pdst) pdst[e] = oe;
            dst[e] = g * oe;
        }
    }
    free(logit);
    free(q);
    free(o);
}

int oracle_attend(const void* q, int dtype, int Hq, int dqk, int dv,
                  const void* k_cache, int64_t ld_k, const void* v_cache, int64_t ld_v,
                  int64_t ntasks, const int64_t* qrow, const int64_t* key_start,
                  const int32_t* idx, int K, double scale, const float* gate,
                  double* out, double* pre, int nthreads)
{
    if (dtype != OR_F32 && dtype != OR_BF16) return -1;
    if (Hq <= 0 || dqk <= 0 || dv <= 0 || K <= 0) return -1;
    attend_ctx c = { q, dtype, Hq, dqk, dv, k_cache, ld_k, v_cache, ld_v,
                     qrow, key_start, idx, K, scale, gate, out, pre };
    run_rows(attend_row, &c, ntasks, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* gradients of the gated attention over a fixed index set             */
/* ------------------------------------------------------------------ */
/*
 * The training path of the layer ("Hybrid Attention Architectures...",
 * section 3.1: the selected set is fixed once the indexer has chosen it, and
 * attention over it is ordinary softmax attention; the gate of section 3.3
 * scales its output). For task r (query row t = qrow[r], keys key_start[r] +
 * idx[r, i], idx < 0 skipped), with l_i = scale * q_h . k_i, p = softmax(l),
 * o_h = sum_i p_i v_i, g_h = 1 / (1 + exp(-x_h)) and out_h = g_h o_h, the
 * derivatives of sum(dout * out) are, by the chain rule:
 *     dx_h  = g_h (1 - g_h) (dout_h . o_h)
 *     do_h  = g_h dout_h
 *     dp_i  = do_h . v_i,   D_h = sum_i p_i dp_i
 *     dl_i  = p_i (dp_i - D_h)
 *     dq_h  = scale sum_i dl_i k_i
 *     dk_i += scale sum_h dl_i q_h,   dv_i += sum_h p_i do_h
 * dq [ntasks, Hq, dqk] and dgate [ntasks, Hq] are per task; dk [nk, dqk] and
 * dv [nk, dv] collect every task's share (rows of the key and value arrays,
 * which the caller zeroes). dq and dgate run row-parallel; the shared dk and
 * dv are accumulated afterwards, one task after the other, in task order.
 */
typedef struct {
    const void* q; int dtype; int Hq, dqk, dv;
    const void* kc; int64_t ld_k; const void* vc; int64_t ld_v;
    const int64_t *qrow, *key_start; const int32_t* idx; int K;
    double scale; const float* gate; const void* dout;
    double *dq, *dk, *dvo, *dgate;
} backward_ctx;

/* p (softmax weights) and dl (logit gradients) of one (task, head); o is
 * the pre-gate output; returns dout . o */
static double backward_head(const backward_ctx* c, int64_t r, int h, double* q, double* p, double* dl,
                            double* o, double* dout, double* g_out)
{
    const int64_t t = c->qrow[r];
    const int32_t* sel = c->idx + r * (int64_t)c->K;
    for (int d = 0; d < c->dqk; ++d) q[d] = load_elem(c->q, c->dtype, (t * c->Hq + h) * (int64_t)c->dqk + d);
    for (int e = 0; e < c->dv; ++e) dout[e] = load_elem(c->dout, c->dtype, (r * c->Hq + h) * (int64_t)c->dv + e);
    double m = -INFINITY;
    for (int i = 0; i < c->K; ++i) {
        if (sel[i] < 0) continue;
        const int64_t kr = c->key_start[r] + sel[i];
        double dot = 0.0;
        for (int d = 0; d < c->dqk; ++d) dot += q[d] * load_elem(c->kc, c->dtype, kr * c->ld_k + d);
        p[i] = c->scale * dot;
        if (p[i] > m) m = p[i];
    }
    double denom = 0.0;
    for (int i = 0; i < c->K; ++i) {
        if (sel[i] < 0) continue;
        p[i] = exp(p[i] - m);
        denom += p[i];
    }
    for (int e = 0; e < c->dv; ++e) o[e] = 0.0;
    for (int i = 0; i < c->K; ++i) {
        if (sel[i] < 0) continue;
        p[i] /= denom;
        const int64_t kr = c->key_start[r] + sel[i];
        for (int e = 0; e < c->dv; ++e) o[e] += p[i] * load_elem(c->vc, c->dtype, kr * c->ld_v + e);
    }
    const double g = 1.0 / (1.0 + exp(-(double)c->gate[t * c->Hq + h]));
    double dout_o = 0.0;
    for (int e = 0; e < c->dv; ++e) dout_o += dout[e] * o[e];
    /* D = do . o with do = g * dout */
    const double D = g * dout_o;
    for (int i = 0; i < c->K; ++i) {
        if (sel[i] < 0) continue;
        const int64_t kr = c->key_start[r] + sel[i];
        double dp = 0.0;
        for (int e = 0; e < c->dv; ++e) dp += g * dout[e] * load_elem(c->vc, c->dtype, kr * c->ld_v + e);
        dl[i] = p[i] * (dp - D);
    }
    *g_out = g;
    return dout_o;
}

static void backward_row(void* pc, int64_t r)
{
    backward_ctx* c = (backward_ctx*)pc;
    const int32_t* sel = c->idx + r * (int64_t)c->K;
    double* q = (double*)malloc(sizeof(double) * (size_t)c->dqk);
    double* o = (double*)malloc(sizeof(double) * (size_t)c->dv);
    double* dout = (double*)malloc(sizeof(double) * (size_t)c->dv);
    double* p = (double*)malloc(sizeof(double) * (size_t)c->K);
    double* dl = (double*)malloc(sizeof(double) * (size_t)c->K);
    for (int h = 0; h < c->Hq; ++h) {
        double g;
        const double dout_o = backward_head(c, r, h, q, p, dl, o, dout, &g);
        c->dgate[r * c->Hq + h] = g * (1.0 - g) * dout_o;
        double* dq = c->dq + (r * c->Hq + h) * (int64_t)c->dqk;
        for (int d = 0; d < c->dqk; ++d) dq[d] = 0.0;
        for (int i = 0; i < c->K; ++i) {
            if (sel[i] < 0) continue;
            const int64_t kr = c->key_start[r] + sel[i];
            for (int d = 0; d < c->dqk; ++d) dq[d] += c->scale * dl[i] * load_elem(c->kc, c->dtype, kr * c->ld_k + d);
        }
    }
    free(q); free(o); free(dout); free(p); free(dl);
}

int oracle_attend_backward(const void* q, int dtype, int Hq, int dqk, int dv,
                           const void* k_cache, int64_t ld_k, const void* v_cache, int64_t ld_v,
                           int64_t ntasks, const int64_t* qrow, const int64_t* key_start,
                           const int32_t* idx, int K, double scale, const float* gate, const void* dout,
                           double* dq, double* dk, double* dvo, double* dgate, int nthreads)
{
    if (dtype != OR_F32 && dtype != OR_BF16) return -1;
    if (Hq <= 0 || dqk <= 0 || dv <= 0 || K <= 0) return -1;
    backward_ctx c = { q, dtype, Hq, dqk, dv, k_cache, ld_k, v_cache, ld_v, qrow, key_start, idx, K,
                       scale, gate, dout, dq, dk, dvo, dgate };
    run_rows(backward_row, &c, ntasks, nthreads);
    /* the shared key and value rows, one task after the other */
    double* qv = (double*)malloc(sizeof(double) * (size_t)dqk);
    double* o = (double*)malloc(sizeof(double) * (size_t)dv);
    double* dov = (double*)malloc(sizeof(double) * (size_t)dv);
    double* p = (double*)malloc(sizeof(double) * (size_t)K);
    double* dl = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t r = 0; r < ntasks; ++r) {
        const int32_t* sel = idx + r * (int64_t)K;
        for (int h = 0; h < Hq; ++h) {
            double g;
            (void)backward_head(&c, r, h, qv, p, dl, o, dov, &g);
            for (int i = 0; i < K; ++i) {
                if (sel[i] < 0) continue;
                const int64_t kr = key_start[r] + sel[i];
                for (int d = 0; d < dqk; ++d) dk[kr * dqk + d] += scale * dl[i] * qv[d];
                for (int e = 0; e < dv; ++e) dvo[kr * dv + e] += p[i] * g * dov[e];
            }
        }
    }
    free(qv); free(o); free(dov); free(p); free(dl);
    return 0;
}
