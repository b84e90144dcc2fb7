/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this library. The product path (the CUDA library
 * and its Python binding) never calls it, and this file includes nothing from
 * the product path.
 *
 * What it computes, for every batch b, query head h and query row i (inputs fp16,
 * bf16 or fp32, d innermost; Q and O [B,H,Nq,d], K and V [B,Hkv,Nk,d]; query head h reads key/value
 * head h / (H / Hkv), grouped-query attention, Hkv = H being multi-head attention;
 * self-attention is Nq = Nk = N):
 *
 *   allowed set   A_i = { j : j < L_b  and  (not causal or j <= i + Nk - Nq) }
 *                 L_b = clamp(key_lengths[b], 0, Nk), or Nk when no lengths are given
 *   scores        s_ij = sm_scale * sum_c q_ic k_jc                      (j in A_i)
 *   row max       m_i  = max_{j in A_i} s_ij
 *   normaliser    l_i  = sum_{j in A_i} exp(s_ij - m_i)
 *   probabilities P_ij = exp(s_ij - m_i) / l_i   (0 outside A_i)
 *   output        O_i  = sum_j P_ij v_j
 *   logsumexp     lse_i = m_i + ln l_i
 *   empty A_i     O_i = 0, lse_i = -inf
 *
 * Sources, by page and section:
 *   - "Tensor Parallelism with CUDA - Standard Attention", section "Step 1: QK^T"
 *     (S = QK^T/sqrt(d), one dot product per query/key pair), "Step 2: Softmax"
 *     (row-wise softmax, max subtracted for stability) and "Step 3: PV"
 *     (O_i = sum_j P_ij V_j).
 *   - "Naive Attention Kernel", section "1. Standard Attention: Step by Step"
 *     (scale, additive mask, softmax, PV; masks here are 0 / -inf, which is the
 *     same as leaving the key out of the sum).
 *   - "Self-Attention Kernel & Inference Engine from Scratch", section
 *     "Online Softmax Formulation" (the three steps max, normaliser, divide).
 *   - "cuda-reranker" README, masking paragraph of the optimisation log: padded
 *     keys are excluded from each row's softmax.
 *   - causal: query i attends to keys j <= i (square, top-left aligned), the
 *     plain reading of the causal block skip in "Engineering Decisions &
 *     Trade-offs" of the portfolio page. With Nq != Nk (cross-attention, one of
 *     the README's "natural extensions") the diagonal is aligned at the last
 *     rows: query i sees keys j <= i + Nk - Nq, so the last query sees every
 *     key. The pages fix no alignment; this is the reading taken.
 *   - grouped-query attention (the other "natural extension"): query heads are
 *     split into Hkv consecutive groups of H / Hkv heads, each sharing one K, V.
 *   - logsumexp is not on the pages; it is the natural log of the softmax
 *     normaliser over the scaled, allowed scores.
 *
 * The score row is held explicitly (one row of S at a time, never the N x N
 * matrix) and the softmax is the two-pass definition. Inputs are decoded from
 * IEEE-754 binary16 (or bfloat16, or binary32) to double exactly, so input rounding
 * is not an error source.
 * Work is split across POSIX threads over (batch*head, block of query rows).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = f * 2^-24; exponent 31: inf (f == 0) or NaN;
 * otherwise value = (1024 + f) * 2^(e - 25). Exact in double. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25);
    return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * exponent 0: subnormal, value = f * 2^-133; exponent 255: inf (f == 0) or NaN;
 * otherwise value = (128 + f) * 2^(e - 134). Exact in double. */
double oracle_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -133);
    else if (e == 255)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + f), e - 134);
    return sign ? -mag : mag;
}

static double g_half_table[65536];
static double g_bf16_table[65536];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;

static void build_half_table(void)
{
    for (uint32_t h = 0; h < 65536u; ++h) {
        g_half_table[h] = oracle_half_to_double((uint16_t)h);
        g_bf16_table[h] = oracle_bf16_to_double((uint16_t)h);
    }
}

/* Key j is in query i's allowed set; off = Nk - Nq places the causal diagonal. */
static int allowed(int64_t i, int64_t j, int64_t L, int causal, int64_t off)
{
    if (j >= L)
        return 0; /* key padding: keys at or past the valid length are excluded */
    if (causal && j > i + off)
        return 0; /* causal: query i sees keys j <= i + Nk - Nq only */
    return 1;
}

/* One query row. q: [d]; K, V: [N, d] decoded (N keys); s: scratch [N]; o: [d] out. */
static void attention_row(const double *q, const double *K, const double *V, int64_t N, int64_t d,
                          double sm_scale, int64_t i, int64_t L, int causal, int64_t off,
                          double *s, double *o, double *lse)
{
    int any = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j) {
        if (!allowed(i, j, L, causal, off))
            continue;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += q[c] * K[j * d + c];
        s[j] = sm_scale * dot;
        if (!any || s[j] > m)
            m = s[j];
        any = 1;
    }
    for (int64_t c = 0; c < d; ++c)
        o[c] = 0.0;
    if (!any) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j)
        if (allowed(i, j, L, causal, off))
            l += exp(s[j] - m);
    for (int64_t j = 0; j < N; ++j) {
        if (!allowed(i, j, L, causal, off))
            continue;
        double p = exp(s[j] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            o[c] += p * V[j * d + c];
    }
    *lse = m + log(l);
}

typedef struct {
    const void *q, *k, *v;
    int dtype;          /* 0: binary16, 1: bfloat16 (16-bit patterns), 2: binary32 */
    int64_t B, H, N, d; /* N: query rows per head */
    int64_t Hkv, Nk;    /* key/value heads per batch, keys per head */
    const double *dec;  /* decode table of the input format (fp16 or bf16) */
    double sm_scale;
    int causal;
    const int32_t *key_lengths;
    const int64_t *rows; /* sorted flat row ids ((b*H + h)*N + i), or NULL = every row */
    int64_t n_rows;
    double *o, *lse;
    /* work items: (head, contiguous run of rows) */
    const int64_t *item_begin; /* index into the row list (or flat row id when rows == NULL) */
    int64_t n_items;
    int64_t next_item;
    pthread_mutex_t lock;
    int failed;
} job_t;

static int64_t row_id(const job_t *J, int64_t t) { return J->rows ? J->rows[t] : t; }

/* Element idx of an input tensor, decoded exactly to double. */
static double load_elem(const job_t *J, const void *base, int64_t idx)
{
    if (J->dtype == 2) {
        float f;
        memcpy(&f, (const unsigned char *)base + idx * 4, sizeof f);
        return (double)f;
    }
    return J->dec[((const uint16_t *)base)[idx]];
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const int64_t N = J->N, d = J->d, Nk = J->Nk, G = J->H / J->Hkv;
    const size_t kv_elems = (size_t)(Nk > 0 ? Nk * d : 1);
    double *K = (double *)malloc(kv_elems * sizeof(double));
    double *V = (double *)malloc(kv_elems * sizeof(double));
    double *s = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    double *q = (double *)malloc((size_t)d * sizeof(double));
    int64_t decoded_head = -1;
    if (!K || !V || !s || !q) {
        pthread_mutex_lock(&J->lock);
        J->failed = 1;
        pthread_mutex_unlock(&J->lock);
        free(K); free(V); free(s); free(q);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t it = J->next_item++;
        pthread_mutex_unlock(&J->lock);
        if (it >= J->n_items)
            break;
        int64_t t0 = J->item_begin[it], t1 = J->item_begin[it + 1];
        for (int64_t t = t0; t < t1; ++t) {
            int64_t r = row_id(J, t);
            int64_t bh = r / N, i = r % N, b = bh / J->H, h = bh % J->H;
            int64_t kvh = b * J->Hkv + h / G; /* the key/value head query head h reads */
            if (kvh != decoded_head) {
                for (int64_t e = 0; e < Nk * d; ++e) {
                    K[e] = load_elem(J, J->k, kvh * Nk * d + e);
                    V[e] = load_elem(J, J->v, kvh * Nk * d + e);
                }
                decoded_head = kvh;
            }
            for (int64_t c = 0; c < d; ++c)
                q[c] = load_elem(J, J->q, r * d + c);
            int64_t L = Nk;
            if (J->key_lengths) {
                L = J->key_lengths[b];
                if (L < 0) L = 0;
                if (L > Nk) L = Nk;
            }
            double lse;
            attention_row(q, K, V, Nk, d, J->sm_scale, i, L, J->causal, Nk - N, s, J->o + t * d,
                          &lse);
            if (J->lse)
                J->lse[t] = lse;
        }
    }
    free(K); free(V); free(s); free(q);
    return NULL;
}

/*
 * Computes O (and lse) for the listed query rows, or for all B*H*Nq rows when
 * rows == NULL. q: [B,H,Nq,d]; k, v: [B,Hkv,Nk,d], H a multiple of Hkv; elements
 * are dtype 0: IEEE binary16, 1: bfloat16 (16-bit patterns), 2: IEEE binary32. key_lengths: [B] or NULL. rows: flat row ids (b*H + h)*Nq + i in
 * ascending order, n_rows of them. o: [n_rows, d] doubles (or [B,H,Nq,d] when
 * rows == NULL); lse: [n_rows] or NULL. n_threads <= 0 uses one thread. Returns 0
 * on success, -1 on bad arguments, -2 when memory runs out.
 */
int oracle_attn_ex(const void *q, const void *k, const void *v, int64_t B, int64_t H,
                   int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int dtype, double sm_scale,
                   int causal, const int32_t *key_lengths, const int64_t *rows, int64_t n_rows,
                   double *o, double *lse, int n_threads)
{
    const int64_t N = Nq;
    if (!q || !k || !v || !o || B < 0 || H < 0 || N < 0 || Nk < 0 || d <= 0 || Hkv < 1 ||
        H % Hkv != 0 || dtype < 0 || dtype > 2)
        return -1;
    int64_t total = B * H * N;
    if (!rows)
        n_rows = total;
    if (n_rows < 0)
        return -1;
    for (int64_t t = 0; rows && t < n_rows; ++t)
        if (rows[t] < 0 || rows[t] >= total || (t > 0 && rows[t] < rows[t - 1]))
            return -1;
    if (n_rows == 0)
        return 0;
    pthread_once(&g_table_once, build_half_table);

    /* Items: runs of at most 64 rows that stay within one head. */
    int64_t cap = n_rows + 1;
    int64_t *begin = (int64_t *)malloc((size_t)(cap + 1) * sizeof(int64_t));
    if (!begin)
        return -2;
    int64_t n_items = 0;
    int64_t t = 0;
    while (t < n_rows) {
        begin[n_items++] = t;
        int64_t head = (rows ? rows[t] : t) / N;
        int64_t u = t + 1;
        while (u < n_rows && u - t < 64 && (rows ? rows[u] : u) / N == head)
            ++u;
        t = u;
    }
    begin[n_items] = n_rows;

    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v;
    J.B = B; J.H = H; J.N = N; J.d = d;
    J.Hkv = Hkv; J.Nk = Nk;
    J.dtype = dtype;
    J.dec = dtype == 1 ? g_bf16_table : g_half_table;
    J.sm_scale = sm_scale;
    J.causal = causal;
    J.key_lengths = key_lengths;
    J.rows = rows;
    J.n_rows = n_rows;
    J.o = o;
    J.lse = lse;
    J.item_begin = begin;
    J.n_items = n_items;
    pthread_mutex_init(&J.lock, NULL);

    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > 1024)
        n_threads = 1024;
    if (n_threads > n_items)
        n_threads = (int)n_items;
    pthread_t *th = (pthread_t *)malloc((size_t)n_threads * sizeof(pthread_t));
    int started = 0;
    if (th) {
        for (int w = 0; w < n_threads; ++w) {
            if (pthread_create(&th[w], NULL, worker, &J) != 0)
                break;
            ++started;
        }
    }
    if (started == 0)
        worker(&J);
    for (int w = 0; w < started; ++w)
        pthread_join(th[w], NULL);
    free(th);
    free(begin);
    pthread_mutex_destroy(&J.lock);
    return J.failed ? -2 : 0;
}

/* Self-attention (Nq = Nk = N, Hkv = H): q, k, v all [B,H,N,d]; see oracle_attn_ex. */
int oracle_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B, int64_t H,
                int64_t N, int64_t d, double sm_scale, int causal, const int32_t *key_lengths,
                const int64_t *rows, int64_t n_rows, double *o, double *lse, int n_threads)
{
    return oracle_attn_ex(q, k, v, B, H, H > 0 ? H : 1, N, N, d, 0, sm_scale, causal, key_lengths,
                          rows, n_rows, o, lse, n_threads);
}
