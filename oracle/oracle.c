/*
 * oracle.c -- plain, slow, fp64 CPU oracle for unified-max split-KV decode attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py load this library. The CUDA path shares no code,
 * header, table or helper with it, and neither side includes or links the other.
 *
 * What it follows (web pages, cited by title and section):
 *   [theory]  opt.ai.kr, "FlashDecoding++ async softmax -- theory":
 *             section 1: decode attention is one query token against a K/V cache that grows,
 *                        so every step reads the whole cache; Flash-Decoding cuts that cache
 *                        into splits that run in parallel.
 *             section 3: the ordinary softmax shifted by the running max (first formula);
 *                        the same softmax shifted by a unified max phi fixed in advance
 *                        (second formula), so every block works alone and only a plain sum
 *                        is left at the end; a block whose score crosses the phi criterion
 *                        stops and is recomputed with the ordinary online softmax.
 *   [export]  opt.ai.kr, "FlashDecoding++ export strategy", section 2: the KV cache is split
 *             inside attention and each chunk carries its own partial sum and normaliser.
 *   [3dgen]   hwan-h-heo.github.io, "Optimizing sparse 3D generation inference", section 2.2:
 *             softmax rows sum to one, so value rows that are all equal to v0 give v0.
 *
 * Readings where the pages leave a step open:
 *   R1  The windowed quantity x is the scaled score s = scale * <q, k> (the softmax input of
 *       [theory] s3), in the same units as phi.
 *   R2  A score is in the window iff lo <= s - phi <= hi (closed). The pages name only the
 *       upper (overflow) side; the lower side guards a split whose scores all lie far below
 *       phi. NaN is outside.
 *   R3  One decision per (sequence b, query head h, split j): each query head is its own
 *       softmax row.
 *   R4  A recomputed split is expressed in its own max frame m_j, so the final combine
 *       rescales every split by exp(m_j - M), M = max_j m_j; when nothing fell back every
 *       m_j = phi and this is exactly the plain sum of [theory] s3.
 *   R5  Only tokens t < L_b take part. L_b == 0 gives an all-zero output row.
 *   R6  scale, phi, lo and hi are the float32 values the caller passes, widened to double.
 *   R7  phi may be given per query head (a float32 per head); the same steps then use each
 *       head's own value. A single phi is the case where every head has the same value.
 *   R8  "phi is set by observing the distribution in advance" ([theory] s3) is read as: on
 *       sample inputs, phi_h is a value that keeps the most row-splits of head h inside the
 *       window; among all values that do, the middle of the widest closed run of them.
 *   R9  Several query tokens per sequence ([theory] s3 quotes the method for prefill as well as
 *       decode): the Tq query tokens are the sequence's last Tq positions, so query token i sees
 *       the keys t < L_b - Tq + 1 + i (causal). The splits stay those of the sequence's keys; a
 *       query row's last splits may hold fewer of its keys or none. A row with no key is zero.
 *   R10 The flat GEMM of [theory] s2 (2) and s4 is a decode-time linear layer: a few rows of
 *       activations (M, the batch of query tokens) times a weight matrix that does not change
 *       (N x K). Read as y = x W^T with x [M][K] and W [N][K] row-major (a linear layer's weight
 *       as stored), C[m][n] = sum_k x[m][k] W[n][k]. The pages give no layout or dtype; bf16 in,
 *       as for the cache.
 *   R11 "The block stops and is recomputed with the ordinary online softmax" ([theory] s3) is read
 *       as a statement about the block's result: its partial is the online softmax's. Taking the
 *       block's tiles in order and testing each tile's scores before using them, the tiles before
 *       the first one holding a score outside the window are all inside it, so their phi-frame
 *       sums are the online softmax's sums in the frame phi (the two formulas of s3 agree for any
 *       shift); from that tile on the block continues with the running max, starting from phi when
 *       some sum is already held and from nothing otherwise. or_inplace_partial restates these
 *       steps for one softmax row, so that the tests can hold them against the plain definition.
 *
 * Precision: every value is widened exactly to double (bf16 and fp32 both widen exactly);
 * all arithmetic is double. Threads: rows are independent, and are spread over pthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ----------------------------------------------------------------------------------------- */
/* problem description (the oracle's own struct; the CUDA side has a separate one)           */
/* ----------------------------------------------------------------------------------------- */

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_MODE_NORMAL = 0, OR_MODE_FORCE_FAST = 1, OR_MODE_FORCE_ONLINE = 2 };

/* flag bits of one (b, h, j) decision */
enum { OR_FLAG_OUT = 1, OR_FLAG_ABOVE = 2, OR_FLAG_BELOW = 4, OR_FLAG_NAN = 8 };

typedef struct {
    int batch;            /* B */
    int num_q_heads;      /* Hq */
    int num_kv_heads;     /* Hkv, Hq % Hkv == 0, G = Hq / Hkv query heads share one kv head */
    int head_dim;         /* d */
    int dtype;            /* OR_F32 or OR_BF16 (bf16 given as raw uint16 bit patterns) */
    int paged;            /* 0: K,V are [B][max_seq_len][Hkv][d]; 1: [blocks][block_size][Hkv][d] */
    int max_seq_len;      /* contiguous: the token stride of the cache */
    int block_size;       /* paged only */
    int max_blocks_per_seq; /* paged only: row length of block_table */
    float scale, phi, lo, hi;
    int q_tokens;         /* Tq >= 1 query tokens per sequence, the last Tq positions (R9) */
} or_problem;

/* Query rows (R9). q and out are [B][Tq][Hq][d], i.e. [B*Tq][Hq][d]: "query row" bi = b*Tq + i
 * is query token i of sequence b. It sees the keys t < L_b - Tq + 1 + i (causal within the last
 * Tq positions; all L_b keys for Tq = 1). */
static int or_tq(const or_problem* p) { return p->q_tokens > 1 ? p->q_tokens : 1; }

static int or_key_limit(const or_problem* p, const int32_t* seq_lens, int bi)
{
    int tq = or_tq(p), L = seq_lens[bi / tq];
    int lim = L - tq + 1 + bi % tq;
    if (L <= 0 || lim < 0) return 0;
    return lim;
}

/* ----------------------------------------------------------------------------------------- */
/* element access                                                                            */
/* ----------------------------------------------------------------------------------------- */

static double or_widen(const void* base, int dtype, size_t i)
{
    if (dtype == OR_BF16) {
        /* bf16 is the upper half of an IEEE binary32 pattern */
        uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[i];
}

/* Element offset of K/V row (b, t, g). Contiguous: token t of sequence b at [b][t][g][:].
 * Paged: token t lives in slot t % block_size of physical block block_table[b][t / block_size]. */
static size_t or_kv_offset(const or_problem* p, const int32_t* table, int b, int t, int g)
{
    size_t d = (size_t)p->head_dim, hkv = (size_t)p->num_kv_heads;
    if (!p->paged)
        return (((size_t)b * (size_t)p->max_seq_len + (size_t)t) * hkv + (size_t)g) * d;
    int32_t blk = table[(size_t)b * (size_t)p->max_blocks_per_seq + (size_t)(t / p->block_size)];
    size_t slot = (size_t)(t % p->block_size);
    return (((size_t)blk * (size_t)p->block_size + slot) * hkv + (size_t)g) * d;
}

/* s_t = scale * sum_i q[bi,h,i] * k[b,t,g(h),i]  for t < L, g(h) = floor(h / G), b = bi / Tq
 * ([theory] s1) */
static void or_scores(const or_problem* p, const void* q, const void* k, const int32_t* table,
                      int bi, int h, int L, double* s)
{
    int d = p->head_dim, G = p->num_q_heads / p->num_kv_heads, g = h / G, b = bi / or_tq(p);
    size_t qoff = ((size_t)bi * (size_t)p->num_q_heads + (size_t)h) * (size_t)d;
    double scale = (double)p->scale;
    for (int t = 0; t < L; ++t) {
        size_t koff = or_kv_offset(p, table, b, t, g);
        double dot = 0.0;
        for (int i = 0; i < d; ++i)
            dot += or_widen(q, p->dtype, qoff + (size_t)i) * or_widen(k, p->dtype, koff + (size_t)i);
        s[t] = scale * dot;
    }
}

/* ----------------------------------------------------------------------------------------- */
/* thread pool over rows                                                                      */
/* ----------------------------------------------------------------------------------------- */

typedef void (*or_row_fn)(void* ctx, int row_index);

typedef struct {
    or_row_fn fn;
    void* ctx;
    int n_rows;
    int n_threads;
    int tid;
} or_job;

static void* or_worker(void* arg)
{
    or_job* j = (or_job*)arg;
    for (int r = j->tid; r < j->n_rows; r += j->n_threads)
        j->fn(j->ctx, r);
    return NULL;
}

static int or_resolve_threads(int n_threads, int n_rows)
{
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    if (n_threads > n_rows) n_threads = n_rows > 0 ? n_rows : 1;
    if (n_threads > 512) n_threads = 512;
    return n_threads;
}

/* Runs fn over rows [0, n_rows) on n_threads threads; returns the thread count used. */
static int or_parallel_rows(or_row_fn fn, void* ctx, int n_rows, int n_threads)
{
    n_threads = or_resolve_threads(n_threads, n_rows);
    if (n_threads == 1) {
        for (int r = 0; r < n_rows; ++r) fn(ctx, r);
        return 1;
    }
    pthread_t th[512];
    or_job jobs[512];
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].n_rows = n_rows;
        jobs[t].n_threads = n_threads; jobs[t].tid = t;
        if (pthread_create(&th[t], NULL, or_worker, &jobs[t]) != 0) break;
        ++started;
    }
    if (started < n_threads) {
        /* a thread could not start: finish its share here */
        for (int t = started; t < n_threads; ++t) or_worker(&jobs[t]);
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    return n_threads;
}

/* ----------------------------------------------------------------------------------------- */
/* 1. exact attention: the plain definition, max-shifted ([theory] s3, first formula)        */
/* ----------------------------------------------------------------------------------------- */

typedef struct {
    const or_problem* p;
    const void *q, *k, *v;
    const int32_t* table;
    const int32_t* seq_lens;
    const int32_t* rows;   /* pairs (b, h); NULL means row r = (r / Hq, r % Hq) */
    double* out;           /* [n_rows][d] */
    int use_phi;           /* 0: shift by max_t s_t ; 1: shift by phi ([theory] s3, second formula) */
    double phi_override;   /* shift used when use_phi == 2 */
} or_attn_ctx;

/* Row r -> (query row bi, head h); explicit rows are (bi, h) pairs. */
static void or_row_bh(const or_problem* p, const int32_t* rows, int r, int* b, int* h)
{
    if (rows) { *b = rows[2 * r]; *h = rows[2 * r + 1]; }
    else { *b = r / p->num_q_heads; *h = r % p->num_q_heads; }
}

static void or_attn_row(void* vctx, int r)
{
    or_attn_ctx* c = (or_attn_ctx*)vctx;
    const or_problem* p = c->p;
    int bi, h;
    or_row_bh(p, c->rows, r, &bi, &h);
    int d = p->head_dim, G = p->num_q_heads / p->num_kv_heads, g = h / G, b = bi / or_tq(p);
    int L = or_key_limit(p, c->seq_lens, bi);
    double* o = c->out + (size_t)r * (size_t)d;
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    if (L <= 0) return;                                   /* R5 */

    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    or_scores(p, c->q, c->k, c->table, bi, h, L, s);

    double shift;
    if (c->use_phi == 1) shift = (double)p->phi;
    else if (c->use_phi == 2) shift = c->phi_override;
    else {
        shift = s[0];
        for (int t = 1; t < L; ++t) if (s[t] > shift) shift = s[t];
    }
    double Z = 0.0;
    for (int t = 0; t < L; ++t) {
        double w = exp(s[t] - shift);
        Z += w;
        size_t voff = or_kv_offset(p, c->table, b, t, g);
        for (int i = 0; i < d; ++i) o[i] += w * or_widen(c->v, p->dtype, voff + (size_t)i);
    }
    for (int i = 0; i < d; ++i) o[i] /= Z;
    free(s);
}

/* out[r][:] = softmax(scale * q K^T) V for each requested row, shifted by the row max.
 * Returns the number of threads used. */
int or_attention(const or_problem* p, const void* q, const void* k, const void* v,
                 const int32_t* block_table, const int32_t* seq_lens,
                 const int32_t* rows, int n_rows, double* out, int n_threads)
{
    or_attn_ctx c = { p, q, k, v, block_table, seq_lens, rows, out, 0, 0.0 };
    return or_parallel_rows(or_attn_row, &c, n_rows, n_threads);
}

/* Same definition with the shift fixed in advance ([theory] s3, second formula):
 * w_t = exp(s_t - shift) / sum_u exp(s_u - shift). shift = p->phi when use_given == 0,
 * else the value `shift`. Algebraically equal to or_attention wherever exp stays finite. */
int or_attention_shifted(const or_problem* p, const void* q, const void* k, const void* v,
                         const int32_t* block_table, const int32_t* seq_lens,
                         const int32_t* rows, int n_rows, int use_given, double shift,
                         double* out, int n_threads)
{
    or_attn_ctx c = { p, q, k, v, block_table, seq_lens, rows, out, use_given ? 2 : 1, shift };
    return or_parallel_rows(or_attn_row, &c, n_rows, n_threads);
}

/* ----------------------------------------------------------------------------------------- */
/* 2. the split scheduler, restated                                                           */
/* ----------------------------------------------------------------------------------------- */

/* Split length actually used. split_len > 0 is taken as given. split_len == 0 asks for an
 * automatic choice: spread sum_b L_b * Hkv (token, kv-head) pairs over units_per_sm * num_sms
 * units, round the length up to a multiple of `granule`, then clamp it to
 * [min_split, max(min_split, max_seq_len rounded up to granule)].
 * (The pages give no sizing rule; this policy is the library's own and is restated here.) */
int or_split_len(const int32_t* seq_lens, int batch, int num_kv_heads, int max_seq_len,
                 int split_len, int num_sms, int units_per_sm, int granule, int min_split)
{
    if (split_len > 0) return split_len;
    long long total = 0;
    for (int b = 0; b < batch; ++b) {
        long long L = seq_lens[b];
        if (L < 0) L = 0;
        if (L > max_seq_len) L = max_seq_len;
        total += L;
    }
    long long units = (long long)units_per_sm * (long long)num_sms;
    if (units < 1) units = 1;
    long long pairs = total * (long long)num_kv_heads;
    long long S = (pairs + units - 1) / units;
    S = ((S + granule - 1) / granule) * granule;
    long long hi = ((long long)max_seq_len + granule - 1) / granule * granule;
    if (hi < min_split) hi = min_split;
    if (S < min_split) S = min_split;
    if (S > hi) S = hi;
    return (int)S;
}

/* n_b = ceil(L_b / S) splits for sequence b; split_off[b] = sum of n_c for c < b
 * (split_off has batch + 1 entries). Unit order is b-major, then kv head g, then split j, so
 * the first unit of sequence b is num_kv_heads * split_off[b]. Returns the unit count. */
long long or_plan(const int32_t* seq_lens, int batch, int num_kv_heads, int max_seq_len, int S,
                  int32_t* nsplit, int32_t* split_off)
{
    long long off = 0;
    for (int b = 0; b < batch; ++b) {
        long long L = seq_lens[b];
        if (L < 0) L = 0;
        if (L > max_seq_len) L = max_seq_len;
        int n = (int)((L + S - 1) / S);
        nsplit[b] = n;
        split_off[b] = (int32_t)off;
        off += n;
    }
    split_off[batch] = (int32_t)off;
    return off * (long long)num_kv_heads;
}

/* ----------------------------------------------------------------------------------------- */
/* 3. window decisions per (b, h, j)                                                          */
/* ----------------------------------------------------------------------------------------- */

typedef struct {
    const or_problem* p;
    const void *q, *k;
    const int32_t* table;
    const int32_t* seq_lens;
    int S, max_splits;
    uint8_t* flags;         /* [B][Hq][max_splits] */
    double* row_margin;     /* [B*Hq]: min over valid t of min(|x - lo|, |x - hi|), x = s - phi */
    const float* phi_heads; /* [Hq] or NULL (p->phi for every head) */
} or_flag_ctx;

/* The unified max of head h: the head's own value when per-head values are given (R7). */
static double or_phi(const or_problem* p, const float* phi_heads, int h)
{
    return phi_heads ? (double)phi_heads[h] : (double)p->phi;
}

static uint8_t or_classify(double x, double lo, double hi)
{
    if (x != x) return OR_FLAG_OUT | OR_FLAG_NAN;                      /* R2: NaN is outside */
    if (x > hi) return OR_FLAG_OUT | OR_FLAG_ABOVE;                    /* [theory] s3 overflow side */
    if (x < lo) return OR_FLAG_OUT | OR_FLAG_BELOW;                    /* R2 lower side */
    return 0;
}

static void or_flag_row(void* vctx, int r)
{
    or_flag_ctx* c = (or_flag_ctx*)vctx;
    const or_problem* p = c->p;
    int bi = r / p->num_q_heads, h = r % p->num_q_heads;
    int L = or_key_limit(p, c->seq_lens, bi);
    uint8_t* f = c->flags + (size_t)r * (size_t)c->max_splits;
    for (int j = 0; j < c->max_splits; ++j) f[j] = 0;
    double margin = INFINITY;
    if (L > 0) {
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        or_scores(p, c->q, c->k, c->table, bi, h, L, s);
        double phi = or_phi(p, c->phi_heads, h), lo = (double)p->lo, hi = (double)p->hi;
        for (int t = 0; t < L; ++t) {
            double x = s[t] - phi;
            int j = t / c->S;
            if (j < c->max_splits) f[j] |= or_classify(x, lo, hi);
            double m1 = fabs(x - lo), m2 = fabs(x - hi);
            double m = m1 < m2 ? m1 : m2;
            if (m < margin) margin = m;
        }
        free(s);
    }
    if (c->row_margin) c->row_margin[r] = margin;
}

/* flags[b][h][j] for every row; entries with j >= n_b stay 0. row_margin and phi_heads may be
 * NULL. */
int or_window_flags(const or_problem* p, const void* q, const void* k,
                    const int32_t* block_table, const int32_t* seq_lens, int S, int max_splits,
                    uint8_t* flags, double* row_margin, const float* phi_heads, int n_threads)
{
    or_flag_ctx c = { p, q, k, block_table, seq_lens, S, max_splits, flags, row_margin, phi_heads };
    return or_parallel_rows(or_flag_row, &c, p->batch * or_tq(p) * p->num_q_heads, n_threads);
}

/* ----------------------------------------------------------------------------------------- */
/* 4. the method's own steps in fp64 (test-only restatement of the split decomposition)       */
/* ----------------------------------------------------------------------------------------- */
/*
 * For each row (b, h) and split j covering tokens [jS, min((j+1)S, L_b)):
 *   fast partial in the phi frame ([theory] s3, second formula; [export] s2 per-chunk sums):
 *       o_j = sum_t exp(s_t - phi) v_t,  l_j = sum_t exp(s_t - phi),  m_j = phi
 *   decision (R2, R3): flag_j = any t in the split with s_t - phi outside [lo, hi]
 *   recompute when flagged (mode normal) or always (mode force_online), with the ordinary
 *   online softmax ([theory] s3, first formula, max tracked while running):
 *       m <- max(m, s_t); o, l scaled by exp(m_old - m); o += exp(s_t - m) v_t; l += exp(s_t - m)
 *       giving (o_j, l_j, m_j = split max)
 *   combine (R4): M = max_j m_j, out = sum_j exp(m_j - M) o_j / sum_j exp(m_j - M) l_j
 *       (a plain sum whenever every m_j = phi).
 * Partials are written when part_o / part_l / part_m are not NULL, indexed [row][j].
 */

typedef struct {
    const or_problem* p;
    const void *q, *k, *v;
    const int32_t* table;
    const int32_t* seq_lens;
    const int32_t* rows;
    int S, max_splits, mode;
    double* out;       /* [n_rows][d] */
    double* part_o;    /* [n_rows][max_splits][d] or NULL */
    double* part_l;    /* [n_rows][max_splits] or NULL */
    double* part_m;    /* [n_rows][max_splits] or NULL */
    uint8_t* flags;    /* [n_rows][max_splits] or NULL */
    const float* phi_heads;   /* [Hq] or NULL */
} or_split_ctx;

static void or_split_row(void* vctx, int r)
{
    or_split_ctx* c = (or_split_ctx*)vctx;
    const or_problem* p = c->p;
    int bi, h;
    or_row_bh(p, c->rows, r, &bi, &h);
    int d = p->head_dim, G = p->num_q_heads / p->num_kv_heads, g = h / G, b = bi / or_tq(p);
    /* the splits are the sequence's (n_b = ceil(L_b / S)); this row's keys stop at L (R9), so
     * its last splits may hold fewer tokens, or none */
    int Lseq = c->seq_lens[b], L = or_key_limit(p, c->seq_lens, bi);
    double* out = c->out + (size_t)r * (size_t)d;
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    int n = Lseq > 0 ? (Lseq + c->S - 1) / c->S : 0;
    if (n > c->max_splits) n = c->max_splits;
    if (n == 0 || L <= 0) return;

    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    double* o = (double*)calloc((size_t)n * (size_t)d, sizeof(double));
    double* l = (double*)calloc((size_t)n, sizeof(double));
    double* m = (double*)calloc((size_t)n, sizeof(double));
    uint8_t* f = (uint8_t*)calloc((size_t)n, 1);
    or_scores(p, c->q, c->k, c->table, bi, h, L, s);
    double phi = or_phi(p, c->phi_heads, h), lo = (double)p->lo, hi = (double)p->hi;

    for (int j = 0; j < n; ++j) {
        int t0 = j * c->S, t1 = t0 + c->S < L ? t0 + c->S : L;
        double* oj = o + (size_t)j * (size_t)d;
        /* fast partial against the unified max */
        for (int t = t0; t < t1; ++t) {
            double w = exp(s[t] - phi);
            l[j] += w;
            size_t voff = or_kv_offset(p, c->table, b, t, g);
            for (int i = 0; i < d; ++i) oj[i] += w * or_widen(c->v, p->dtype, voff + (size_t)i);
            f[j] |= or_classify(s[t] - phi, lo, hi);
        }
        m[j] = phi;
        int redo = (c->mode == OR_MODE_FORCE_ONLINE) ||
                   (c->mode == OR_MODE_NORMAL && (f[j] & OR_FLAG_OUT));
        if (redo) {
            /* ordinary online softmax over the same split */
            double mm = -INFINITY, ll = 0.0;
            for (int i = 0; i < d; ++i) oj[i] = 0.0;
            for (int t = t0; t < t1; ++t) {
                double mnew = s[t] > mm ? s[t] : mm;
                double corr = exp(mm - mnew);           /* exp(-inf) = 0 on the first token */
                ll *= corr;
                for (int i = 0; i < d; ++i) oj[i] *= corr;
                double w = exp(s[t] - mnew);
                ll += w;
                size_t voff = or_kv_offset(p, c->table, b, t, g);
                for (int i = 0; i < d; ++i) oj[i] += w * or_widen(c->v, p->dtype, voff + (size_t)i);
                mm = mnew;
            }
            l[j] = ll;
            m[j] = mm;
        }
    }
    /* combine: max-rescaled sum, a plain sum when every m_j == phi */
    double M = m[0];
    for (int j = 1; j < n; ++j) if (m[j] > M) M = m[j];
    double lam = 0.0;
    for (int j = 0; j < n; ++j) {
        double e = exp(m[j] - M);
        lam += e * l[j];
        for (int i = 0; i < d; ++i) out[i] += e * o[(size_t)j * (size_t)d + (size_t)i];
    }
    for (int i = 0; i < d; ++i) out[i] /= lam;

    for (int j = 0; j < n; ++j) {
        size_t pj = (size_t)r * (size_t)c->max_splits + (size_t)j;
        if (c->part_o)
            for (int i = 0; i < d; ++i) c->part_o[pj * (size_t)d + (size_t)i] = o[(size_t)j * (size_t)d + (size_t)i];
        if (c->part_l) c->part_l[pj] = l[j];
        if (c->part_m) c->part_m[pj] = m[j];
        if (c->flags) c->flags[pj] = f[j];
    }
    free(s); free(o); free(l); free(m); free(f);
}

int or_split_method(const or_problem* p, const void* q, const void* k, const void* v,
                    const int32_t* block_table, const int32_t* seq_lens,
                    const int32_t* rows, int n_rows, int S, int max_splits, int mode,
                    double* out, double* part_o, double* part_l, double* part_m, uint8_t* flags,
                    const float* phi_heads, int n_threads)
{
    or_split_ctx c = { p, q, k, v, block_table, seq_lens, rows, S, max_splits, mode,
                       out, part_o, part_l, part_m, flags, phi_heads };
    return or_parallel_rows(or_split_row, &c, n_rows, n_threads);
}

/* One softmax row's partial by R11: scores s[n] (already scaled), values v[n][d], tiles of `tile`
 * tokens. Writes o[d], *l and *m (the frame: phi, or the last running max) and returns 1 if the row
 * switched to the running max. */
int or_inplace_partial(const double* s, const double* v, int n, int d, int tile, double phi,
                       double lo, double hi, double* o, double* l, double* m)
{
    if (n < 0 || d < 1 || tile < 1) return -1;
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    double ll = 0.0, mm = phi;
    int online = 0;
    for (int t0 = 0; t0 < n; t0 += tile) {
        int t1 = t0 + tile < n ? t0 + tile : n;
        if (!online) {
            /* the tile's scores are tested before any of them is used */
            int out = 0;
            for (int t = t0; t < t1; ++t) out |= or_classify(s[t] - phi, lo, hi) & OR_FLAG_OUT;
            if (out) {
                online = 1;
                if (!(ll > 0.0)) mm = -INFINITY;    /* nothing held yet: the plain online start */
            }
        }
        for (int t = t0; t < t1; ++t) {
            if (online) {
                double mnew = s[t] > mm ? s[t] : mm;
                double corr = mm == -INFINITY ? 0.0 : exp(mm - mnew);
                ll *= corr;
                for (int i = 0; i < d; ++i) o[i] *= corr;
                mm = mnew;
            }
            double w = exp(s[t] - mm);
            ll += w;
            for (int i = 0; i < d; ++i) o[i] += w * v[(size_t)t * (size_t)d + (size_t)i];
        }
    }
    *l = ll;
    *m = mm;
    return online;
}

/* ----------------------------------------------------------------------------------------- */
/* 5. calibration of phi from observed scores                                                 */
/* ----------------------------------------------------------------------------------------- */
/*
 * [theory] s3: phi is set in advance by observing the score distribution; a block whose scores
 * leave the window falls back. Read plainly (R8): record, on sample inputs, the range
 * [min s, max s] of every row-split (b, h, j). The split keeps the fast path iff every score
 * satisfies lo <= s - phi <= hi, i.e. iff phi lies in [max s - hi, min s - lo]. For head h, phi_h
 * is a value inside the most such intervals; of all values that reach that count, the middle of
 * the widest closed run. A head none of whose splits can be kept gets the fallback value.
 */

typedef struct {
    const or_problem* p;
    const void *q, *k;
    const int32_t* table;
    const int32_t* seq_lens;
    int S, max_splits;
    double *smin, *smax;    /* [B][Hq][max_splits] */
} or_range_ctx;

static void or_range_row(void* vctx, int r)
{
    or_range_ctx* c = (or_range_ctx*)vctx;
    const or_problem* p = c->p;
    int bi = r / p->num_q_heads, h = r % p->num_q_heads;
    int L = or_key_limit(p, c->seq_lens, bi);
    double* lo = c->smin + (size_t)r * (size_t)c->max_splits;
    double* hi = c->smax + (size_t)r * (size_t)c->max_splits;
    for (int j = 0; j < c->max_splits; ++j) { lo[j] = NAN; hi[j] = NAN; }
    if (L <= 0) return;
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    or_scores(p, c->q, c->k, c->table, bi, h, L, s);
    for (int t = 0; t < L; ++t) {
        int j = t / c->S;
        if (j >= c->max_splits) break;
        if (t % c->S == 0 || s[t] < lo[j]) lo[j] = s[t];
        if (t % c->S == 0 || s[t] > hi[j]) hi[j] = s[t];
    }
    free(s);
}

/* smin / smax [B][Hq][max_splits]: the least and greatest score of each row-split over its valid
 * tokens; NaN for j >= n_b. */
int or_score_ranges(const or_problem* p, const void* q, const void* k, const int32_t* block_table,
                    const int32_t* seq_lens, int S, int max_splits, double* smin, double* smax,
                    int n_threads)
{
    or_range_ctx c = { p, q, k, block_table, seq_lens, S, max_splits, smin, smax };
    return or_parallel_rows(or_range_row, &c, p->batch * or_tq(p) * p->num_q_heads, n_threads);
}

static int or_cmp_double(const void* a, const void* b)
{
    double x = *(const double*)a, y = *(const double*)b;
    return x < y ? -1 : (x > y ? 1 : 0);
}

/* Number of intervals [a_i, b_i] that contain x. */
static int or_stab(const double* a, const double* bb, int n, double x)
{
    int c = 0;
    for (int i = 0; i < n; ++i) c += (a[i] <= x && x <= bb[i]);
    return c;
}

/* phi_out[h] (and count_out[h], the splits it keeps; may be NULL) from the score ranges of the
 * row-splits j < nsplit[b], over all sequences b. Plain method: the kept count is constant on
 * each endpoint and on each open gap between consecutive endpoints, so those are evaluated one by
 * one, and the widest run of consecutive ones at the best count gives phi_h. */
int or_pick_phi(const double* smin, const double* smax, const int32_t* nsplit, int batch,
                int num_q_heads, int max_splits, double lo, double hi, double fallback,
                double* phi_out, int32_t* count_out)
{
    size_t cap = (size_t)batch * (size_t)max_splits;
    double* a = (double*)malloc(sizeof(double) * (cap + 1));
    double* bb = (double*)malloc(sizeof(double) * (cap + 1));
    double* x = (double*)malloc(sizeof(double) * (2 * cap + 1));
    int* cnt = (int*)malloc(sizeof(int) * (4 * cap + 2));
    for (int h = 0; h < num_q_heads; ++h) {
        int n = 0;
        for (int b = 0; b < batch; ++b) {
            int nb = nsplit[b] < max_splits ? nsplit[b] : max_splits;
            for (int j = 0; j < nb; ++j) {
                size_t r = ((size_t)b * (size_t)num_q_heads + (size_t)h) * (size_t)max_splits + (size_t)j;
                double lo_phi = smax[r] - hi, hi_phi = smin[r] - lo;
                if (lo_phi == lo_phi && hi_phi == hi_phi && lo_phi <= hi_phi) {
                    a[n] = lo_phi;
                    bb[n] = hi_phi;
                    ++n;
                }
            }
        }
        if (n == 0) {
            phi_out[h] = fallback;
            if (count_out) count_out[h] = 0;
            continue;
        }
        int m = 0;
        for (int i = 0; i < n; ++i) { x[m++] = a[i]; x[m++] = bb[i]; }
        qsort(x, (size_t)m, sizeof(double), or_cmp_double);
        int u = 0;
        for (int i = 0; i < m; ++i) if (u == 0 || x[i] != x[u - 1]) x[u++] = x[i];
        /* elements in order: point x0, gap (x0, x1), point x1, ..., point x_{u-1} */
        int ne = 2 * u - 1, best = 0;
        for (int e = 0; e < ne; ++e) {
            double at = (e % 2 == 0) ? x[e / 2] : 0.5 * (x[e / 2] + x[e / 2 + 1]);
            cnt[e] = or_stab(a, bb, n, at);
            if (cnt[e] > best) best = cnt[e];
        }
        double best_w = -1.0, best_mid = 0.0;
        for (int e = 0; e < ne;) {
            if (cnt[e] != best) { ++e; continue; }
            int f = e;
            while (f + 1 < ne && cnt[f + 1] == best) ++f;
            /* a run starts and ends on points (a gap at best count implies both its points) */
            double left = x[e / 2], right = x[(f + 1) / 2];
            if (right - left > best_w) { best_w = right - left; best_mid = 0.5 * (left + right); }
            e = f + 1;
        }
        phi_out[h] = best_mid;
        if (count_out) count_out[h] = best;
    }
    free(a); free(bb); free(x); free(cnt);
    return 0;
}

/* ----------------------------------------------------------------------------------------- */
/* 5. flat GEMM of a decode-time linear layer ([theory] s2 (2), s4; R10)                      */
/* ----------------------------------------------------------------------------------------- */

typedef struct {
    int M, N, K, dtype;
    const void* x;            /* [M][K] */
    const void* w;            /* [N][K] */
    const int32_t* entries;   /* (m, n) pairs, or NULL for every (m, n) */
    double* out;              /* [n_entries] or [M][N] */
} or_gemm_ctx;

/* One output row of work: entry r, or row m = r of the full product. */
static void or_gemm_row(void* vctx, int r)
{
    const or_gemm_ctx* c = (const or_gemm_ctx*)vctx;
    if (c->entries) {
        const int m = c->entries[2 * r], n = c->entries[2 * r + 1];
        double acc = 0.0;
        for (int k = 0; k < c->K; ++k)
            acc += or_widen(c->x, c->dtype, (size_t)m * c->K + k) *
                   or_widen(c->w, c->dtype, (size_t)n * c->K + k);
        c->out[r] = acc;
        return;
    }
    for (int n = 0; n < c->N; ++n) {
        double acc = 0.0;
        for (int k = 0; k < c->K; ++k)
            acc += or_widen(c->x, c->dtype, (size_t)r * c->K + k) *
                   or_widen(c->w, c->dtype, (size_t)n * c->K + k);
        c->out[(size_t)r * c->N + n] = acc;
    }
}

/* C[m][n] = sum_k x[m][k] * W[n][k] in double, k ascending, on the widened inputs (R10). With
 * entries == NULL, out is the whole [M][N] product; otherwise out[i] is entry i's (m, n).
 * Returns the thread count used, or -1 on a bad argument. */
int or_flat_gemm(int M, int N, int K, int dtype, const void* x, const void* w,
                 const int32_t* entries, int n_entries, double* out, int n_threads)
{
    if (M < 0 || N < 0 || K < 0 || !out || (M > 0 && K > 0 && !x) || (N > 0 && K > 0 && !w))
        return -1;
    if (entries) {
        for (int i = 0; i < n_entries; ++i)
            if (entries[2 * i] < 0 || entries[2 * i] >= M || entries[2 * i + 1] < 0 ||
                entries[2 * i + 1] >= N)
                return -1;
    }
    or_gemm_ctx c = {M, N, K, dtype, x, w, entries, out};
    return or_parallel_rows(or_gemm_row, &c, entries ? n_entries : M, n_threads);
}

/* Number of threads or_* calls use for n_threads == 0 (the host's online CPUs). */
int or_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
