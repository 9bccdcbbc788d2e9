/*
 * fp64 CPU oracle for the attention forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this file's library.  It shares no code, header or constant with the CUDA
 * path and is deliberately slow and plain: one query row at a time, two
 * passes over the keys, every sum in float64 in key order.
 *
 * What it computes (the plain definition of masked scaled dot-product
 * attention):
 *
 *   Attention(Q,K,V) = softmax(Q K^T * scale + mask) V
 *     -- hotelren.com "AI attention: essence and evolution", sec. 2.1
 *        (softmax-attention derivation, scaling by sqrt(d_k)) and ch.1 code
 *        (masked_fill with -inf, then softmax, then the product with V);
 *        cnnetsun.cn "Transformer QKV bottlenecks on long sequences",
 *        sec. 1 (underlying principle).
 *   The softmax is evaluated with the max shift and the log-sum-exp
 *     -- aicoding.csdn.net "Why attention stalls large-model training",
 *        sec. 2.2 (softmax numerical-stability traps, chunked logsumexp).
 *   A key j is visible to query i iff j < key_len[b] (key-padding mask,
 *     lshu.cn "Self-attention meets the compute wall", sec. 4.1 and 5.2) and,
 *     when causal, j <= i (only earlier positions and itself; hotelren.com
 *     sec. 2.1 note 2, lshu.cn sec. 3.1) and, when a sliding window of w > 0
 *     positions is given, j > i - w (the window of the last w positions up to
 *     the query; aicoding.csdn.net sec. 4.3, sliding-window attention with
 *     w = 512, and hotelren.com ch.1, local window attention at O(n w)).
 *
 * For each batch b, head h and query row i:
 *   s_j   = scale * sum_t q[i,t] k[j,t]          (visible j only)
 *   m     = max_j s_j
 *   l     = sum_j exp(s_j - m)
 *   O[i]  = (sum_j exp(s_j - m) v[j]) / l
 *   lse   = m + ln l                              (natural log)
 * A row with no visible key gets O = 0 and lse = -inf.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    const double *q, *k, *v;
    int64_t B, H, Nq, Nk, d;
    double scale;
    int causal;
    int64_t window;
    const int32_t *key_lens;
    const int64_t *rows;
    int64_t n_rows;
    double *out, *lse;
    int64_t first, last; /* half-open range of work items (b, h, row) */
} oracle_job;

static int key_visible(int64_t i, int64_t j, int64_t key_len, int causal, int64_t window)
{
    if (j >= key_len) return 0;
    if (causal && j > i) return 0;
    if (window > 0 && j <= i - window) return 0;
    return 1;
}

static void oracle_row(const oracle_job *jb, int64_t item, double *s)
{
    const int64_t n_rows = jb->n_rows, Nq = jb->Nq, N = jb->Nk, d = jb->d;
    const int64_t bh = item / n_rows, r = item % n_rows;
    const int64_t b = bh / jb->H;
    const int64_t i = jb->rows ? jb->rows[r] : r;
    const int64_t key_len = jb->key_lens ? (int64_t)jb->key_lens[b] : N;
    const double *q = jb->q + (bh * Nq + i) * d;
    const double *K = jb->k + bh * N * d;
    const double *V = jb->v + bh * N * d;
    double *o = jb->out + item * d;

    /* pass 1: scaled logits of the visible keys and their maximum */
    double m = -INFINITY;
    int64_t n_visible = 0;
    for (int64_t j = 0; j < N; ++j) {
        if (!key_visible(i, j, key_len, jb->causal, jb->window)) continue;
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += q[t] * K[j * d + t];
        s[j] = jb->scale * dot;
        if (s[j] > m) m = s[j];
        ++n_visible;
    }
    for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
    if (n_visible == 0) {
        jb->lse[item] = -INFINITY;
        return;
    }
    /* pass 2: exponentials, their sum, and the weighted sum of V rows */
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (!key_visible(i, j, key_len, jb->causal, jb->window)) continue;
        const double w = exp(s[j] - m);
        l += w;
        for (int64_t t = 0; t < d; ++t) o[t] += w * V[j * d + t];
    }
    for (int64_t t = 0; t < d; ++t) o[t] /= l;
    jb->lse[item] = m + log(l);
}

static void *oracle_worker(void *arg)
{
    oracle_job *jb = (oracle_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    if (!s) return (void *)1;
    for (int64_t it = jb->first; it < jb->last; ++it) oracle_row(jb, it, s);
    free(s);
    return NULL;
}

/*
 * q: float64 [B, H, Nq, d]; k, v: float64 [B, H, Nk, d]; all C-contiguous.
 * Query i and key j share one position axis starting at 0 (the causal rule
 * j <= i compares them directly); self-attention has Nq == Nk.
 * key_lens: int32 [B] or NULL (all Nk keys visible); used as given.
 * window: > 0 limits query i to keys j > i - window; <= 0 means no window.
 * rows: the query rows to compute (same for every (b, h)), or NULL for
 *       0..Nq-1 (then n_rows must equal Nq).
 * out: float64 [B, H, n_rows, d]; lse: float64 [B, H, n_rows].
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
int oracle_attn_fwd(const double *q, const double *k, const double *v,
                    int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                    double scale, int causal, int64_t window, const int32_t *key_lens,
                    const int64_t *rows, int64_t n_rows,
                    double *out, double *lse, int n_threads)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0 || n_rows < 0) return -1;
    if (!rows && n_rows != Nq) return -1;
    const int64_t items = B * H * n_rows;
    if (items == 0) return 0;
    if (!q || !k || !v || !out || !lse) return -1;
    for (int64_t r = 0; rows && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= Nq) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > items) n_threads = (int)items;

    oracle_job jobs[256];
    pthread_t tids[256];
    int started[256] = {0};
    int rc = 0;
    for (int t = 0; t < n_threads; ++t) {
        oracle_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v;
        jb->B = B; jb->H = H; jb->Nq = Nq; jb->Nk = Nk; jb->d = d;
        jb->scale = scale; jb->causal = causal; jb->window = window; jb->key_lens = key_lens;
        jb->rows = rows; jb->n_rows = n_rows; jb->out = out; jb->lse = lse;
        jb->first = items * t / n_threads;
        jb->last = items * (t + 1) / n_threads;
        if (t == 0) continue; /* the calling thread runs job 0 */
        started[t] = pthread_create(&tids[t], NULL, oracle_worker, jb) == 0;
        if (!started[t]) rc = -1;
    }
    if (oracle_worker(&jobs[0]) != NULL) rc = -1;
    for (int t = 1; t < n_threads; ++t) {
        void *ret = NULL;
        if (started[t]) {
            pthread_join(tids[t], &ret);
            if (ret != NULL) rc = -1;
        }
    }
    return rc; /* -1 also when a worker could not start: its rows are undone */
}
