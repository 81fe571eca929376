/*
 * FP64 CPU oracle for causal grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only tests/, __graft_entry__.smoke() and the cpu_baseline / reference leg of
 * bench.py load it.  It shares no code, header or table with the CUDA library.
 *
 * What it computes is the plain definition of attention, written out with no
 * blocking, no online softmax and no fusion:
 *
 *   s_j   = scale * sum_d q[i,h,d] * k[j,g,d]          for j in V(i)
 *   m     = max_j s_j
 *   w_j   = exp(s_j - m)
 *   out[i,h,d] = sum_j w_j v[j,g,d] / sum_j w_j
 *
 * with g = h / (Hq / Hkv) the KV head shared by a group of query heads, and
 * V(i) the set of keys row i may see:
 *
 *   dense   ("[Kernel][SM70] Default long-prefill GQA architecture", Purpose):
 *           bottom-right causal alignment, V(i) = {0 .. KV - Q + i}.
 *   paged   ("[Perf] Ship the qualified SM70 long-context layout ...", What /
 *           Changes): the same with KV := ctx_len and Q := R tail rows; key t
 *           lives in physical page block_table[t / page], slot t % page, and
 *           K, V = decode_e4m3(byte) * kscale / vscale.
 *   sparse  ("[Kernel][SM70] Repair #378 on latest main", Changes): V(i) is the
 *           union over the row's selected four-token blocks b of
 *           {4b .. 4b+3}, intersected with {0 .. p_i}, p_i = ctx_len - rows + i
 *           (positions past the row are clamped away; block ids outside
 *           0 .. p_i/4 select nothing).  Its keys and values come from an fp16
 *           page cache, or from an E4M3 page cache read as in the paged
 *           variant (the E4M3 storage of the second page applied to this
 *           workload).
 *
 * Inputs arrive as raw fp16 bit patterns and E4M3 bytes; each is decoded here
 * to its exact double value.  Output is double, never rounded to fp16.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE binary16 bits -> exact double. */
static double half_to_double(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return s ? -v : v;
}

/* OCP FP8 E4M3 ("fn" flavour): 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, largest finite 448, subnormals
 * m/8 * 2^-6.  The pages only say "E4M3"; this is the common reading. */
double oracle_e4m3_decode(uint8_t b) {
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) {
        v = ldexp((double)m / 8.0, -6);
    } else {
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    }
    return s ? -v : v;
}

/* ---------------------------------------------------------------------- */
/* The attention of one (row, head) over an explicit ascending key list.   */
/* ---------------------------------------------------------------------- */

typedef struct {
    /* key j's K / V vector for KV head g, decoded to double into dst[D] */
    void (*fetch_k)(const void* ctx, int j, int g, double* dst);
    void (*fetch_v)(const void* ctx, int j, int g, double* dst);
    const void* ctx;
    int D;
} kv_source;

/* Two-pass softmax attention.  keys[0..n) is the visible set in ascending
 * order; qd[D] the query vector; out[D] receives the result.  Scratch buffers
 * s[n], kbuf[D], vbuf[D] are caller-provided.  If probs != NULL the
 * normalised weights w_j / sum w are written there. */
static void attend(const kv_source* src, const double* qd, int g, const int* keys, int n,
                   double scale, double* s, double* kbuf, double* vbuf, double* out,
                   double* probs) {
    const int D = src->D;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) return;
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
        src->fetch_k(src->ctx, keys[t], g, kbuf);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * kbuf[d];
        s[t] = scale * dot;
        if (s[t] > m) m = s[t];
    }
    double denom = 0.0;
    for (int t = 0; t < n; ++t) {
        double w = exp(s[t] - m);
        s[t] = w;
        denom += w;
    }
    for (int t = 0; t < n; ++t) {
        src->fetch_v(src->ctx, keys[t], g, vbuf);
        double w = s[t];
        for (int d = 0; d < D; ++d) out[d] += w * vbuf[d];
    }
    for (int d = 0; d < D; ++d) out[d] /= denom;
    if (probs) {
        for (int t = 0; t < n; ++t) probs[t] = s[t] / denom;
    }
}

/* ---------------------------------------------------------------------- */
/* Key / value sources                                                      */
/* ---------------------------------------------------------------------- */

typedef struct {
    const uint16_t* k;  /* [KV, Hkv, D] fp16 bits */
    const uint16_t* v;
    int Hkv, D;
} dense_ctx;

static void dense_fetch_k(const void* c, int j, int g, double* dst) {
    const dense_ctx* x = (const dense_ctx*)c;
    const uint16_t* p = x->k + ((size_t)j * x->Hkv + g) * x->D;
    for (int d = 0; d < x->D; ++d) dst[d] = half_to_double(p[d]);
}
static void dense_fetch_v(const void* c, int j, int g, double* dst) {
    const dense_ctx* x = (const dense_ctx*)c;
    const uint16_t* p = x->v + ((size_t)j * x->Hkv + g) * x->D;
    for (int d = 0; d < x->D; ++d) dst[d] = half_to_double(p[d]);
}

typedef struct {
    const uint8_t* kc;  /* [num_pages, page, Hkv, D] E4M3 bytes */
    const uint8_t* vc;
    double kscale, vscale;
    const int32_t* table;
    int page, Hkv, D;
} paged_ctx;

static const uint8_t* paged_row(const paged_ctx* x, const uint8_t* cache, int j, int g) {
    int phys = x->table[j / x->page];
    size_t tok = (size_t)phys * x->page + (size_t)(j % x->page);
    return cache + (tok * x->Hkv + g) * x->D;
}
static void paged_fetch_k(const void* c, int j, int g, double* dst) {
    const paged_ctx* x = (const paged_ctx*)c;
    const uint8_t* p = paged_row(x, x->kc, j, g);
    for (int d = 0; d < x->D; ++d) dst[d] = oracle_e4m3_decode(p[d]) * x->kscale;
}
static void paged_fetch_v(const void* c, int j, int g, double* dst) {
    const paged_ctx* x = (const paged_ctx*)c;
    const uint8_t* p = paged_row(x, x->vc, j, g);
    for (int d = 0; d < x->D; ++d) dst[d] = oracle_e4m3_decode(p[d]) * x->vscale;
}

typedef struct {
    const uint16_t* kc;  /* [num_pages, page, Hkv, D] fp16 bits */
    const uint16_t* vc;
    const int32_t* table;
    int page, Hkv, D;
} paged16_ctx;

static const uint16_t* paged16_row(const paged16_ctx* x, const uint16_t* cache, int j, int g) {
    int phys = x->table[j / x->page];
    size_t tok = (size_t)phys * x->page + (size_t)(j % x->page);
    return cache + (tok * x->Hkv + g) * x->D;
}
static void paged16_fetch_k(const void* c, int j, int g, double* dst) {
    const paged16_ctx* x = (const paged16_ctx*)c;
    const uint16_t* p = paged16_row(x, x->kc, j, g);
    for (int d = 0; d < x->D; ++d) dst[d] = half_to_double(p[d]);
}
static void paged16_fetch_v(const void* c, int j, int g, double* dst) {
    const paged16_ctx* x = (const paged16_ctx*)c;
    const uint16_t* p = paged16_row(x, x->vc, j, g);
    for (int d = 0; d < x->D; ++d) dst[d] = half_to_double(p[d]);
}

/* ---------------------------------------------------------------------- */
/* Row-parallel driver                                                      */
/* ---------------------------------------------------------------------- */

enum { VAR_DENSE = 0, VAR_PAGED = 1, VAR_SPARSE = 2 };

typedef struct {
    int variant;
    kv_source src;
    const uint16_t* q;   /* [rows_total, Hq, D] fp16 bits */
    int rows_total, n_ctx, Hq, Hkv, D;
    double scale;
    /* sparse selection */
    const int32_t* sel_idx;
    const int32_t* sel_cnt;
    int max_sel;
    /* work list */
    const int* rows;
    int nrows;
    double* out;         /* [nrows, Hq, D] */
    int next;            /* shared work counter */
    pthread_mutex_t lock;
} job;

/* Visible key set of query row i, ascending; returns its size. */
static int visible_keys(const job* jb, int i, int* keys, unsigned char* mark) {
    int p = jb->n_ctx - jb->rows_total + i;  /* absolute position of row i */
    int n = 0;
    if (jb->variant != VAR_SPARSE) {
        for (int j = 0; j <= p; ++j) keys[n++] = j;
        return n;
    }
    memset(mark, 0, (size_t)p + 1);
    int cnt = jb->sel_cnt[i];
    for (int t = 0; t < cnt; ++t) {
        int b = jb->sel_idx[(size_t)i * jb->max_sel + t];
        if (b < 0) continue;
        for (int u = 0; u < 4; ++u) {
            long long j = 4LL * b + u;
            if (j <= p) mark[j] = 1;
        }
    }
    for (int j = 0; j <= p; ++j)
        if (mark[j]) keys[n++] = j;
    return n;
}

static void* worker(void* arg) {
    job* jb = (job*)arg;
    const int D = jb->D;
    int* keys = (int*)malloc(sizeof(int) * (size_t)(jb->n_ctx + 1));
    unsigned char* mark = (unsigned char*)malloc((size_t)jb->n_ctx + 1);
    double* s = (double*)malloc(sizeof(double) * (size_t)(jb->n_ctx + 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    double* kb = (double*)malloc(sizeof(double) * (size_t)D);
    double* vb = (double*)malloc(sizeof(double) * (size_t)D);
    for (;;) {
        pthread_mutex_lock(&jb->lock);
        int w = jb->next++;
        pthread_mutex_unlock(&jb->lock);
        if (w >= jb->nrows) break;
        int i = jb->rows[w];
        int n = visible_keys(jb, i, keys, mark);
        for (int h = 0; h < jb->Hq; ++h) {
            int g = h / (jb->Hq / jb->Hkv);
            const uint16_t* qp = jb->q + ((size_t)i * jb->Hq + h) * D;
            for (int d = 0; d < D; ++d) qd[d] = half_to_double(qp[d]);
            double* o = jb->out + ((size_t)w * jb->Hq + h) * D;
            attend(&jb->src, qd, g, keys, n, jb->scale, s, kb, vb, o, NULL);
        }
    }
    free(keys); free(mark); free(s); free(qd); free(kb); free(vb);
    return NULL;
}

static int run_job(job* jb, int nthreads) {
    if (jb->Hq <= 0 || jb->Hkv <= 0 || jb->Hq % jb->Hkv) return 1;
    if (jb->rows_total < 1 || jb->rows_total > jb->n_ctx) return 1;
    for (int w = 0; w < jb->nrows; ++w)
        if (jb->rows[w] < 0 || jb->rows[w] >= jb->rows_total) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    jb->next = 0;
    pthread_mutex_init(&jb->lock, NULL);
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, jb);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&jb->lock);
    return 0;
}

/* Dense causal prefill: q [Q,Hq,D], k/v [KV,Hkv,D] fp16 bits; rows[] selects
 * which query rows to compute; out [nrows,Hq,D] double.  Returns 0 or 1. */
int oracle_dense(const uint16_t* q, const uint16_t* k, const uint16_t* v, int Q, int KV,
                 int Hq, int Hkv, int D, double scale, const int* rows, int nrows,
                 double* out, int nthreads) {
    dense_ctx c = {k, v, Hkv, D};
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.variant = VAR_DENSE;
    jb.src.fetch_k = dense_fetch_k;
    jb.src.fetch_v = dense_fetch_v;
    jb.src.ctx = &c;
    jb.src.D = D;
    jb.q = q; jb.rows_total = Q; jb.n_ctx = KV; jb.Hq = Hq; jb.Hkv = Hkv; jb.D = D;
    jb.scale = scale; jb.rows = rows; jb.nrows = nrows; jb.out = out;
    return run_job(&jb, nthreads);
}

/* Paged E4M3 verifier tail: R query rows at the end of ctx_len keys stored in
 * an E4M3 page cache [num_pages, page, Hkv, D] addressed through block_table
 * (logical page -> physical page). */
int oracle_paged_e4m3(const uint16_t* q, const uint8_t* kc, const uint8_t* vc, double kscale,
                      double vscale, const int32_t* block_table, int page, int ctx_len, int R,
                      int Hq, int Hkv, int D, double scale, const int* rows, int nrows,
                      double* out, int nthreads) {
    paged_ctx c = {kc, vc, kscale, vscale, block_table, page, Hkv, D};
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.variant = VAR_PAGED;
    jb.src.fetch_k = paged_fetch_k;
    jb.src.fetch_v = paged_fetch_v;
    jb.src.ctx = &c;
    jb.src.D = D;
    jb.q = q; jb.rows_total = R; jb.n_ctx = ctx_len; jb.Hq = Hq; jb.Hkv = Hkv; jb.D = D;
    jb.scale = scale; jb.rows = rows; jb.nrows = nrows; jb.out = out;
    return run_job(&jb, nthreads);
}

/* Selected-block sparse paged prefill over an fp16 page cache. */
int oracle_sparse_blocks(const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                         const int32_t* block_table, const int32_t* sel_idx,
                         const int32_t* sel_cnt, int max_sel, int page, int ctx_len,
                         int rows_total, int Hq, int Hkv, int D, double scale, const int* rows,
                         int nrows, double* out, int nthreads) {
    paged16_ctx c = {kc, vc, block_table, page, Hkv, D};
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.variant = VAR_SPARSE;
    jb.src.fetch_k = paged16_fetch_k;
    jb.src.fetch_v = paged16_fetch_v;
    jb.src.ctx = &c;
    jb.src.D = D;
    jb.q = q; jb.rows_total = rows_total; jb.n_ctx = ctx_len; jb.Hq = Hq; jb.Hkv = Hkv;
    jb.D = D; jb.scale = scale; jb.sel_idx = sel_idx; jb.sel_cnt = sel_cnt;
    jb.max_sel = max_sel; jb.rows = rows; jb.nrows = nrows; jb.out = out;
    for (int w = 0; w < nrows; ++w) {
        int i = rows[w];
        if (i < 0 || i >= rows_total || sel_cnt[i] < 0 || sel_cnt[i] > max_sel) return 1;
    }
    return run_job(&jb, nthreads);
}

/* Selected-block sparse paged prefill over an E4M3 page cache: the sparse
 * visible sets, keys and values decode(byte) * kscale / vscale. */
int oracle_sparse_blocks_e4m3(const uint16_t* q, const uint8_t* kc, const uint8_t* vc,
                              double kscale, double vscale, const int32_t* block_table,
                              const int32_t* sel_idx, const int32_t* sel_cnt, int max_sel,
                              int page, int ctx_len, int rows_total, int Hq, int Hkv, int D,
                              double scale, const int* rows, int nrows, double* out,
                              int nthreads) {
    paged_ctx c = {kc, vc, kscale, vscale, block_table, page, Hkv, D};
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.variant = VAR_SPARSE;
    jb.src.fetch_k = paged_fetch_k;
    jb.src.fetch_v = paged_fetch_v;
    jb.src.ctx = &c;
    jb.src.D = D;
    jb.q = q; jb.rows_total = rows_total; jb.n_ctx = ctx_len; jb.Hq = Hq; jb.Hkv = Hkv;
    jb.D = D; jb.scale = scale; jb.sel_idx = sel_idx; jb.sel_cnt = sel_cnt;
    jb.max_sel = max_sel; jb.rows = rows; jb.nrows = nrows; jb.out = out;
    for (int w = 0; w < nrows; ++w) {
        int i = rows[w];
        if (i < 0 || i >= rows_total || sel_cnt[i] < 0 || sel_cnt[i] > max_sel) return 1;
    }
    return run_job(&jb, nthreads);
}

/* Normalised attention weights of one (row, head) of the dense variant over
 * its visible keys 0 .. KV - Q + row; probs[] must hold KV entries.  Returns
 * the number of visible keys, or -1 on bad arguments. */
int oracle_dense_probs(const uint16_t* q, const uint16_t* k, const uint16_t* v, int Q, int KV,
                       int Hq, int Hkv, int D, double scale, int row, int head,
                       double* probs) {
    if (row < 0 || row >= Q || head < 0 || head >= Hq || Q > KV || Hq % Hkv) return -1;
    dense_ctx c = {k, v, Hkv, D};
    kv_source src = {dense_fetch_k, dense_fetch_v, &c, D};
    int n = KV - Q + row + 1;
    int* keys = (int*)malloc(sizeof(int) * (size_t)n);
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    double* kb = (double*)malloc(sizeof(double) * (size_t)D);
    double* vb = (double*)malloc(sizeof(double) * (size_t)D);
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < n; ++j) keys[j] = j;
    const uint16_t* qp = q + ((size_t)row * Hq + head) * D;
    for (int d = 0; d < D; ++d) qd[d] = half_to_double(qp[d]);
    attend(&src, qd, head / (Hq / Hkv), keys, n, scale, s, kb, vb, o, probs);
    free(keys); free(s); free(qd); free(kb); free(vb); free(o);
    return n;
}
