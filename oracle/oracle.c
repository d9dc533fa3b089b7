/*
 * Plain fp64 CPU oracle for ragged softmax attention.  TEST INFRASTRUCTURE
 * ONLY: the tests, the smoke check and the benchmark's CPU baseline call it;
 * the product path never does.  It shares no code with the CUDA library.
 *
 * What it computes is the plain definition of softmax attention, per query
 * row, written out with no blocking, no online recurrence and no KV split:
 *
 *   s_j  = scale * <q, k_j>                       (scores; "Flywheel Attention",
 *                                                   section 1, P = softmax(QK^T);
 *                                                   "Writing Page Attention with
 *                                                   PyPTO", section 1.1, QK^T/sqrt(128))
 *   m    = max_j s_j
 *   l    = sum_j exp(s_j - m)
 *   out  = sum_j exp(s_j - m) v_j / l             (O = PV)
 *   lse  = m + ln l                               (natural-log log-sum-exp)
 *   absv = sum_j exp(s_j - m) |v_j| / l           (optional output: the same
 *                                                   weights on the magnitudes
 *                                                   of the values)
 *
 * absv is not part of attention; it is the scale of the rounding error a
 * kernel may make legitimately.  Rounding every weight exp(s_j - m) to a
 * format with unit roundoff u before the PV product ("Writing Page Attention
 * with PyPTO", section 6.3 casts P to BF16 for the matmul) moves each output
 * column by at most about 2 u absv, whichever sum the kernel divides by.
 *
 * over the keys the row may see.  Rows with no visible key give out = 0 and
 * lse = -inf ("TokenSpeed-MLA 2.0.1", SM107 decode section: rows with no
 * visible keys produce zero output and -inf LSE).
 *
 * Paged decode ("Writing Page Attention with PyPTO", sections 1.2-1.3 and 5.2):
 *   query head h reads KV head h / G with G = Hq / Hkv (consecutive query heads
 *   share a KV head: KV head 1 serves query heads 5-9 when G = 5); logical key
 *   j of batch row b lives in physical page block_table[b, j / page_size] at
 *   slot j % page_size.  With q_len > 1 query tokens the rows are causal and
 *   bottom-right aligned: token t sees keys 0 .. n - q_len + t.
 *
 * Sliding window (oracle_paged_decode_window; "TokenSpeed-MLA 2.0.1",
 *   window_left): with window_left = W >= 0, token t sees only keys
 *   max(0, n - q_len + t - W) .. n - q_len + t, i.e. its own position and the
 *   W positions before it.  Keys before the window are not gathered at all, so
 *   their block-table entries are never read.  W < 0: no window.
 *
 * Causal or not (oracle_paged_decode_masked; "TokenSpeed-MLA 2.0.1":
 *   causal_mask supports causal and non-causal decode, and window_left bounds
 *   row i's history to keys from max(0, K - q_len - window_left + i) up to
 *   its bound): token t's own position is pos = n - q_len + t; causal, it sees
 *   keys up to pos, otherwise all n; a window of W starts at max(0, pos - W)
 *   either way.
 *
 * Varlen prefill ("TokenSpeed-MLA 2.0.1", capability summary: ragged varlen
 * prefill without padding, Q and KV packs described by separate cumulative
 * sequence lengths, causal or not):
 *   sequence i owns query rows cu_q[i] .. cu_q[i+1]-1 and keys cu_k[i] ..
 *   cu_k[i+1]-1; with causal masking row r (0-based inside the sequence) sees
 *   keys 0 .. r + Lk - Lq (bottom-right alignment, as the page's benchmark
 *   command selects with --bottom_right_align).
 *
 * FP8 KV cache (oracle_paged_decode_kv8; "TokenSpeed-MLA 2.0.1": decode on
 * FP8 inputs writes BF16 output): keys and values are OCP FP8 E4M3 bytes with
 * one scale each for the whole cache, k_j = k_scale * e4m3(K byte), v_j =
 * v_scale * e4m3(V byte); the attention itself is the same definition.
 *
 * Inputs are BF16 bit patterns (uint16) or E4M3 bytes; each is widened
 * exactly to double.
 * Strides are in elements.  Every function returns 0 on success or a negative
 * code for an out-of-range index (an invalid page number, a bad row id).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("FN" variant): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent 0 encodes subnormals m * 2^-9; the
 * pattern S.1111.111 is NaN; there is no infinity (S.1111.110 = 448 is the
 * largest finite value). */
double oracle_e4m3_to_double(uint8_t b) {
    int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* One query row against an explicit list of key/value row pointers. */
static void attend_row(const uint16_t *q, int64_t q_dstride,
                       const uint16_t *const *krows, int64_t k_dstride,
                       const uint16_t *const *vrows, int64_t v_dstride,
                       int64_t nkeys, int dk, int dv, double scale,
                       double *s /* scratch [nkeys] */, double *out, double *lse, double *absv) {
    if (nkeys <= 0) {
        for (int d = 0; d < dv; ++d) out[d] = 0.0;
        if (absv) for (int d = 0; d < dv; ++d) absv[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        double acc = 0.0;
        for (int d = 0; d < dk; ++d)
            acc += bf16_to_double(q[d * q_dstride]) * bf16_to_double(krows[j][d * k_dstride]);
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int d = 0; d < dv; ++d) out[d] = 0.0;
    if (absv) for (int d = 0; d < dv; ++d) absv[d] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < dv; ++d) out[d] += p * bf16_to_double(vrows[j][d * v_dstride]);
        if (absv) for (int d = 0; d < dv; ++d) absv[d] += p * fabs(bf16_to_double(vrows[j][d * v_dstride]));
    }
    for (int d = 0; d < dv; ++d) out[d] /= l;
    if (absv) for (int d = 0; d < dv; ++d) absv[d] /= l;
    *lse = m + log(l);
}

/* The same row with FP8 E4M3 key and value rows and their scales. */
static void attend_row_kv8(const uint16_t *q, int64_t q_dstride,
                           const uint8_t *const *krows, int64_t k_dstride, double k_scale,
                           const uint8_t *const *vrows, int64_t v_dstride, double v_scale,
                           int64_t nkeys, int dk, int dv, double scale,
                           double *s, double *out, double *lse, double *absv) {
    if (nkeys <= 0) {
        for (int d = 0; d < dv; ++d) out[d] = 0.0;
        if (absv) for (int d = 0; d < dv; ++d) absv[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        double acc = 0.0;
        for (int d = 0; d < dk; ++d)
            acc += bf16_to_double(q[d * q_dstride]) * (k_scale * oracle_e4m3_to_double(krows[j][d * k_dstride]));
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int d = 0; d < dv; ++d) out[d] = 0.0;
    if (absv) for (int d = 0; d < dv; ++d) absv[d] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < dv; ++d) out[d] += p * (v_scale * oracle_e4m3_to_double(vrows[j][d * v_dstride]));
        if (absv)
            for (int d = 0; d < dv; ++d)
                absv[d] += p * fabs(v_scale * oracle_e4m3_to_double(vrows[j][d * v_dstride]));
    }
    for (int d = 0; d < dv; ++d) out[d] /= l;
    if (absv) for (int d = 0; d < dv; ++d) absv[d] /= l;
    *lse = m + log(l);
}

/* ------------------------------------------------------------------ decode */

typedef struct {
    const uint16_t *q; const int64_t *qs;        /* [B, q_len, Hq, Dk] */
    const void *k; const int64_t *ks;            /* [P, ps, Hkv, Dk]: BF16, or E4M3 when kv8 */
    const void *v; const int64_t *vs;            /* [P, ps, Hkv, Dv]   */
    int kv8; double k_scale, v_scale;
    int window_left;                             /* < 0: none */
    int causal;                                  /* 0: every token sees all n keys */
    const int32_t *bt; int64_t bt_stride;        /* [B, max_pages]     */
    const int32_t *seq_lens;                     /* [B]                */
    int B, q_len, Hq, Hkv, Dk, Dv, ps, num_pages, max_pages;
    double scale;
    const int64_t *rows; int64_t n_rows;
    double *out, *lse, *absv;                    /* absv may be NULL */
    int64_t begin, end;
    int status;
} decode_job;

static void *decode_worker(void *arg) {
    decode_job *J = (decode_job *)arg;
    int G = J->Hq / J->Hkv;
    int64_t cap = (int64_t)J->max_pages * J->ps;
    double *s = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
    const void **kr = (const void **)malloc(sizeof(void *) * (size_t)(cap > 0 ? cap : 1));
    const void **vr = (const void **)malloc(sizeof(void *) * (size_t)(cap > 0 ? cap : 1));
    const size_t esz = J->kv8 ? 1 : 2;                   /* bytes per K/V element */
    if (!s || !kr || !vr) { J->status = -3; goto done; }
    for (int64_t i = J->begin; i < J->end; ++i) {
        int64_t row = J->rows ? J->rows[i] : i;
        if (row < 0 || row >= (int64_t)J->B * J->q_len * J->Hq) { J->status = -2; break; }
        int h = (int)(row % J->Hq);
        int t = (int)((row / J->Hq) % J->q_len);
        int b = (int)(row / ((int64_t)J->Hq * J->q_len));
        int g = h / G;                                   /* consecutive heads share a KV head */
        int64_t n = J->seq_lens[b];
        int64_t pos = n - J->q_len + t;                  /* the token's own key position */
        int64_t visible = J->causal ? pos + 1 : n;       /* bottom-right causal for q_len > 1 */
        if (visible > n) visible = n;
        if (visible < 0) visible = 0;
        if (n > cap) { J->status = -1; break; }
        int64_t first = 0;                               /* sliding window: keys first .. visible - 1 */
        if (J->window_left >= 0) {
            first = pos - J->window_left;
            if (first < 0) first = 0;
            if (first > visible) first = visible;
        }
        for (int64_t j = first; j < visible; ++j) {
            int32_t page = J->bt[(int64_t)b * J->bt_stride + j / J->ps];
            if (page < 0 || page >= J->num_pages) { J->status = -1; goto done; }
            int64_t slot = j % J->ps;
            kr[j] = (const char *)J->k + esz * (size_t)(page * J->ks[0] + slot * J->ks[1] + (int64_t)g * J->ks[2]);
            vr[j] = (const char *)J->v + esz * (size_t)(page * J->vs[0] + slot * J->vs[1] + (int64_t)g * J->vs[2]);
        }
        const uint16_t *qrow = J->q + b * J->qs[0] + t * J->qs[1] + h * J->qs[2];
        if (J->kv8)
            attend_row_kv8(qrow, J->qs[3], (const uint8_t *const *)(kr + first), J->ks[3], J->k_scale,
                           (const uint8_t *const *)(vr + first), J->vs[3], J->v_scale, visible - first, J->Dk,
                           J->Dv, J->scale, s, J->out + i * J->Dv, J->lse + i,
                           J->absv ? J->absv + i * J->Dv : NULL);
        else
            attend_row(qrow, J->qs[3], (const uint16_t *const *)(kr + first), J->ks[3],
                       (const uint16_t *const *)(vr + first), J->vs[3], visible - first, J->Dk, J->Dv, J->scale, s,
                       J->out + i * J->Dv, J->lse + i, J->absv ? J->absv + i * J->Dv : NULL);
    }
done:
    free(s); free(kr); free(vr);
    return NULL;
}

static int paged_decode_any(const uint16_t *q, const int64_t *q_stride,
                            const void *k_cache, const int64_t *k_stride,
                            const void *v_cache, const int64_t *v_stride,
                            int kv8, double k_scale, double v_scale, int causal, int window_left,
                            const int32_t *block_table, int64_t bt_stride,
                            const int32_t *seq_lens,
                            int B, int q_len, int Hq, int Hkv, int Dk, int Dv,
                            int page_size, int num_pages, int max_pages, double scale,
                            const int64_t *rows, int64_t n_rows,
                            double *out, double *lse, double *absv, int n_threads) {
    if (Hkv <= 0 || Hq % Hkv != 0 || page_size <= 0) return -4;
    if (n_threads < 1) n_threads = 1;
    if (n_rows < n_threads) n_threads = (int)(n_rows > 0 ? n_rows : 1);
    decode_job *jobs = (decode_job *)calloc((size_t)n_threads, sizeof(decode_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -3; }
    for (int w = 0; w < n_threads; ++w) {
        decode_job *J = &jobs[w];
        J->q = q; J->qs = q_stride; J->k = k_cache; J->ks = k_stride; J->v = v_cache; J->vs = v_stride;
        J->kv8 = kv8; J->k_scale = k_scale; J->v_scale = v_scale; J->window_left = window_left; J->causal = causal;
        J->bt = block_table; J->bt_stride = bt_stride; J->seq_lens = seq_lens;
        J->B = B; J->q_len = q_len; J->Hq = Hq; J->Hkv = Hkv; J->Dk = Dk; J->Dv = Dv;
        J->ps = page_size; J->num_pages = num_pages; J->max_pages = max_pages; J->scale = scale;
        J->rows = rows; J->n_rows = n_rows; J->out = out; J->lse = lse; J->absv = absv;
        J->begin = n_rows * w / n_threads; J->end = n_rows * (w + 1) / n_threads;
        pthread_create(&tid[w], NULL, decode_worker, J);
    }
    int status = 0;
    for (int w = 0; w < n_threads; ++w) {
        pthread_join(tid[w], NULL);
        if (jobs[w].status) status = jobs[w].status;
    }
    free(jobs); free(tid);
    return status;
}

int oracle_paged_decode(const uint16_t *q, const int64_t *q_stride,
                        const uint16_t *k_cache, const int64_t *k_stride,
                        const uint16_t *v_cache, const int64_t *v_stride,
                        const int32_t *block_table, int64_t bt_stride,
                        const int32_t *seq_lens,
                        int B, int q_len, int Hq, int Hkv, int Dk, int Dv,
                        int page_size, int num_pages, int max_pages, double scale,
                        const int64_t *rows, int64_t n_rows,
                        double *out, double *lse, double *absv, int n_threads) {
    return paged_decode_any(q, q_stride, k_cache, k_stride, v_cache, v_stride, 0, 1.0, 1.0, 1, -1, block_table,
                            bt_stride, seq_lens, B, q_len, Hq, Hkv, Dk, Dv, page_size, num_pages, max_pages,
                            scale, rows, n_rows, out, lse, absv, n_threads);
}

int oracle_paged_decode_kv8(const uint16_t *q, const int64_t *q_stride,
                            const uint8_t *k_cache, const int64_t *k_stride,
                            const uint8_t *v_cache, const int64_t *v_stride,
                            double k_scale, double v_scale,
                            const int32_t *block_table, int64_t bt_stride,
                            const int32_t *seq_lens,
                            int B, int q_len, int Hq, int Hkv, int Dk, int Dv,
                            int page_size, int num_pages, int max_pages, double scale,
                            const int64_t *rows, int64_t n_rows,
                            double *out, double *lse, double *absv, int n_threads) {
    return paged_decode_any(q, q_stride, k_cache, k_stride, v_cache, v_stride, 1, k_scale, v_scale, 1, -1, block_table,
                            bt_stride, seq_lens, B, q_len, Hq, Hkv, Dk, Dv, page_size, num_pages, max_pages,
                            scale, rows, n_rows, out, lse, absv, n_threads);
}

/* Either cache type (kv8 = 1: E4M3 bytes with scales) and a sliding window. */
int oracle_paged_decode_window(const uint16_t *q, const int64_t *q_stride,
                               const void *k_cache, const int64_t *k_stride,
                               const void *v_cache, const int64_t *v_stride,
                               int kv8, double k_scale, double v_scale, int window_left,
                               const int32_t *block_table, int64_t bt_stride,
                               const int32_t *seq_lens,
                               int B, int q_len, int Hq, int Hkv, int Dk, int Dv,
                               int page_size, int num_pages, int max_pages, double scale,
                               const int64_t *rows, int64_t n_rows,
                               double *out, double *lse, double *absv, int n_threads) {
    return paged_decode_any(q, q_stride, k_cache, k_stride, v_cache, v_stride, kv8, k_scale, v_scale, 1, window_left,
                            block_table, bt_stride, seq_lens, B, q_len, Hq, Hkv, Dk, Dv, page_size, num_pages,
                            max_pages, scale, rows, n_rows, out, lse, absv, n_threads);
}

/* Either cache type, causal or not, and a sliding window (W < 0: none). */
int oracle_paged_decode_masked(const uint16_t *q, const int64_t *q_stride,
                               const void *k_cache, const int64_t *k_stride,
                               const void *v_cache, const int64_t *v_stride,
                               int kv8, double k_scale, double v_scale, int causal, int window_left,
                               const int32_t *block_table, int64_t bt_stride,
                               const int32_t *seq_lens,
                               int B, int q_len, int Hq, int Hkv, int Dk, int Dv,
                               int page_size, int num_pages, int max_pages, double scale,
                               const int64_t *rows, int64_t n_rows,
                               double *out, double *lse, double *absv, int n_threads) {
    return paged_decode_any(q, q_stride, k_cache, k_stride, v_cache, v_stride, kv8, k_scale, v_scale, causal,
                            window_left, block_table, bt_stride, seq_lens, B, q_len, Hq, Hkv, Dk, Dv, page_size,
                            num_pages, max_pages, scale, rows, n_rows, out, lse, absv, n_threads);
}

/* ----------------------------------------------------------------- prefill */

typedef struct {
    const uint16_t *q; const int64_t *qs;        /* [total_q, Hq, Dk]  */
    const uint16_t *k; const int64_t *ks;        /* [total_k, Hkv, Dk] */
    const uint16_t *v; const int64_t *vs;        /* [total_k, Hkv, Dv] */
    const int32_t *cu_q, *cu_k;                  /* [B + 1]            */
    int B, Hq, Hkv, Dk, Dv, causal;
    int64_t total_q, max_k;
    double scale;
    const int64_t *rows; int64_t n_rows;
    double *out, *lse, *absv;                    /* absv may be NULL */
    int64_t begin, end;
    int status;
} prefill_job;

static void *prefill_worker(void *arg) {
    prefill_job *J = (prefill_job *)arg;
    int G = J->Hq / J->Hkv;
    int64_t cap = J->max_k > 0 ? J->max_k : 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)cap);
    const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)cap);
    const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)cap);
    if (!s || !kr || !vr) { J->status = -3; goto done; }
    for (int64_t i = J->begin; i < J->end; ++i) {
        int64_t row = J->rows ? J->rows[i] : i;
        if (row < 0 || row >= J->total_q * J->Hq) { J->status = -2; break; }
        int h = (int)(row % J->Hq);
        int64_t tok = row / J->Hq;
        int seq = -1;
        for (int b = 0; b < J->B; ++b)
            if (tok >= J->cu_q[b] && tok < J->cu_q[b + 1]) { seq = b; break; }
        if (seq < 0) { J->status = -2; break; }
        int64_t Lq = J->cu_q[seq + 1] - J->cu_q[seq];
        int64_t Lk = J->cu_k[seq + 1] - J->cu_k[seq];
        int64_t r = tok - J->cu_q[seq];
        int64_t visible = Lk;
        if (J->causal) {
            visible = r + Lk - Lq + 1;                   /* bottom-right alignment */
            if (visible > Lk) visible = Lk;
            if (visible < 0) visible = 0;
        }
        int g = h / G;
        for (int64_t j = 0; j < visible; ++j) {
            int64_t kt = J->cu_k[seq] + j;
            kr[j] = J->k + kt * J->ks[0] + (int64_t)g * J->ks[1];
            vr[j] = J->v + kt * J->vs[0] + (int64_t)g * J->vs[1];
        }
        const uint16_t *qrow = J->q + tok * J->qs[0] + (int64_t)h * J->qs[1];
        attend_row(qrow, J->qs[2], kr, J->ks[2], vr, J->vs[2], visible, J->Dk, J->Dv,
                   J->scale, s, J->out + i * J->Dv, J->lse + i, J->absv ? J->absv + i * J->Dv : NULL);
    }
done:
    free(s); free(kr); free(vr);
    return NULL;
}

int oracle_varlen_prefill(const uint16_t *q, const int64_t *q_stride,
                          const uint16_t *k, const int64_t *k_stride,
                          const uint16_t *v, const int64_t *v_stride,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                          int B, int Hq, int Hkv, int Dk, int Dv, int causal, double scale,
                          const int64_t *rows, int64_t n_rows,
                          double *out, double *lse, double *absv, int n_threads) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -4;
    int64_t max_k = 0;
    for (int b = 0; b < B; ++b) {
        int64_t L = (int64_t)cu_seqlens_k[b + 1] - cu_seqlens_k[b];
        if (L < 0 || cu_seqlens_q[b + 1] < cu_seqlens_q[b]) return -1;
        if (L > max_k) max_k = L;
    }
    if (n_threads < 1) n_threads = 1;
    if (n_rows < n_threads) n_threads = (int)(n_rows > 0 ? n_rows : 1);
    prefill_job *jobs = (prefill_job *)calloc((size_t)n_threads, sizeof(prefill_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -3; }
    for (int w = 0; w < n_threads; ++w) {
        prefill_job *J = &jobs[w];
        J->q = q; J->qs = q_stride; J->k = k; J->ks = k_stride; J->v = v; J->vs = v_stride;
        J->cu_q = cu_seqlens_q; J->cu_k = cu_seqlens_k;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->Dk = Dk; J->Dv = Dv; J->causal = causal;
        J->total_q = cu_seqlens_q[B]; J->max_k = max_k; J->scale = scale;
        J->rows = rows; J->n_rows = n_rows; J->out = out; J->lse = lse; J->absv = absv;
        J->begin = n_rows * w / n_threads; J->end = n_rows * (w + 1) / n_threads;
        pthread_create(&tid[w], NULL, prefill_worker, J);
    }
    int status = 0;
    for (int w = 0; w < n_threads; ++w) {
        pthread_join(tid[w], NULL);
        if (jobs[w].status) status = jobs[w].status;
    }
    free(jobs); free(tid);
    return status;
}

/* ------------------------------------------------------------------ append
 *
 * KV-cache append ("Writing Page Attention with PyPTO", sections 4.2-4.3):
 * the K and V rows of query token t of batch row b go to cache token row
 *   layer_base + max(slot_mapping[b * q_len + t], 0)
 * -- the warm-up slot -1 is clamped to 0 before the layer base is added, so a
 * layer never writes into the previous layer's last row.  Token row r lives
 * at page r / ps, slot r % ps of a [pages, ps, Hkv, D] cache.  A BF16 cache
 * takes the BF16 bits unchanged.  An E4M3 cache takes the code of the FP32
 * quotient x / scale (IEEE single-precision division) rounded to the nearest
 * E4M3 value, ties to an even code, finite overflow saturating to +-448, NaN
 * to S.1111.111 -- the plain reading of "FP8 inputs" with one scale per cache
 * ("TokenSpeed-MLA 2.0.1", decode).  Writes go in (b, t) order; rows that
 * several tokens address (repeated warm-up slots) keep the last one.
 */
uint8_t oracle_e4m3_from_float(float x) {
    if (isnan(x)) return signbit(x) ? 0xFF : 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double best_d = INFINITY;
    for (int code = 0; code <= 0x7E; ++code) {        /* every finite non-negative code */
        double d = fabs(oracle_e4m3_to_double((uint8_t)code) - a);
        if (d < best_d || (d == best_d && (code & 1) == 0)) { best = code; best_d = d; }
    }
    return sign | (uint8_t)best;
}

int oracle_kv_append(const uint16_t *k_new, const int64_t *kn_stride,
                     const uint16_t *v_new, const int64_t *vn_stride,
                     const int32_t *slot_mapping, int64_t layer_base,
                     void *k_cache, const int64_t *k_stride,
                     void *v_cache, const int64_t *v_stride,
                     int kv8, float k_scale, float v_scale,
                     int B, int q_len, int Hkv, int Dk, int Dv, int ps, int64_t num_pages) {
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < q_len; ++t) {
            int64_t slot = slot_mapping[(int64_t)b * q_len + t];
            if (slot < 0) slot = 0;                      /* clamp first ... */
            int64_t row = layer_base + slot;             /* ... then add the layer base */
            if (row < 0 || row >= num_pages * ps) return -1;
            int64_t page = row / ps, off = row % ps;
            for (int h = 0; h < Hkv; ++h) {
                for (int pass = 0; pass < 2; ++pass) {
                    const uint16_t *src = pass ? v_new : k_new;
                    const int64_t *ss = pass ? vn_stride : kn_stride;
                    const int64_t *cs = pass ? v_stride : k_stride;
                    int D = pass ? Dv : Dk;
                    float sc = pass ? v_scale : k_scale;
                    for (int d = 0; d < D; ++d) {
                        uint16_t bits = src[b * ss[0] + t * ss[1] + h * ss[2] + d * ss[3]];
                        int64_t at = page * cs[0] + off * cs[1] + (int64_t)h * cs[2] + (int64_t)d * cs[3];
                        if (kv8) {
                            float x = (float)bf16_to_double(bits);
                            ((uint8_t *)(pass ? v_cache : k_cache))[at] = oracle_e4m3_from_float(x / sc);
                        } else {
                            ((uint16_t *)(pass ? v_cache : k_cache))[at] = bits;
                        }
                    }
                }
            }
        }
    }
    return 0;
}
