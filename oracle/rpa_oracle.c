/*
 * rpa_oracle.c -- plain, slow, fp64 CPU oracle for ragged paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant table with the CUDA
 * library.
 *
 * What it computes is the plain definition the "ragged_paged.zig" page
 * reaches with its blockwise online softmax (sections flashAttention and run):
 * for every sequence s, every query token i of s and every query head qh,
 *
 *   kv head      h   = qh / G,  G = num_q_heads / num_kv_heads     (GQA group)
 *   position     p   = kv_len - q_len + i                      (row_ids)
 *   key j        K_j = dec(kv_pages[page_indices[s, j/ps], j%ps, 2h,   :]) * k_scale
 *   value j      V_j = dec(kv_pages[page_indices[s, j/ps], j%ps, 2h+1, :]) * v_scale
 *   logit        x_j = sm_scale * <q_i, K_j>,  then cap*tanh(x_j/cap) if soft_cap
 *   allowed(j)   j < kv_len, and (not causal or j <= p),
 *                and (no window or not (p - sliding_window >= j))
 *   o            = sum_j w_j V_j / sum_j w_j,  w_j = exp(x_j - max x) on allowed j
 *
 * Attention sinks (the "from_qwen_ops.rs" page, flat_softmax_rows_at, on
 * `sinks`): when set, query head qh has one extra logit s_qh that joins its
 * row's softmax and carries no value: the row maximum starts from s_qh and
 * exp(s_qh - max) joins the denominator,
 *   o            = sum_j w_j V_j / (sum_j w_j + exp(s_qh - m)),
 *   m            = max(s_qh, max x),  w_j = exp(x_j - m).
 * The sink is a logit of the softmax as it stands: it is neither scaled by
 * sm_scale nor soft-capped (those act on the q.k products).
 *
 * Readings where the page is silent or literal-but-quirky (kept in one place):
 *  - masked keys get weight exactly 0 (the page adds mask_value, whose exp
 *    underflows to 0 whenever a row has an allowed key);
 *  - keys j >= kv_len are always excluded, also when not causal;
 *  - a row with no allowed key is 0 (the page's l_safe guard);
 *  - dequant is exact fp64 x*scale (the page rounds it to the q dtype);
 *  - tokens not covered by [cu_q_lens[0], cu_q_lens[num_seqs]) are 0.
 *
 * Latent attention over a paged latent cache (the "from_qwen_ops.rs" page,
 * "The latent-attention family at whole-tile widths": a latent of 512 and a
 * rope part of 64, sixteen or more heads of 576), when latent is set: every
 * slot of a page holds one row of head_dim elements per kv head (kv_pages
 * [total_num_pages, page_size, num_kv_heads, head_dim]); key j of kv head h is
 * that whole row, and its value is the row's first v_head_dim elements:
 *   K_j = dec(kv_pages[pg, sl, h, 0:head_dim]) * k_scale,
 *   V_j = dec(kv_pages[pg, sl, h, 0:v_head_dim]) * v_scale,
 * and o is [num_q_tokens, num_q_heads, v_head_dim].  Everything else (masks,
 * soft cap, sinks, GQA grouping) is as above.
 *
 * Element types ("ragged_paged.zig", Cfg: q_dtype f32 / f16 / bf16; kv_dtype
 * bf16 / f16 / f8e4m3fn / f8e5m2 / i8).  Every stored value is decoded exactly
 * to fp64 from its format's definition and used as it is: the page's casts to
 * the q dtype before its matmuls are not reproduced (the oracle is the exact
 * definition; the GPU's operand rounding is within the tolerance).
 *  - f32: IEEE-754 binary32;
 *  - bf16: the upper half of an IEEE binary32;
 *  - f16: IEEE-754 binary16: 1 sign, 5 exponent bits (bias 15), 10 mantissa
 *    bits, subnormals, infinities and NaN at exponent 31;
 *  - e4m3fn (OCP FP8): bias 7, 3 mantissa bits, subnormals, no infinities,
 *    S.1111.111 = NaN, max 448;
 *  - e5m2 (OCP FP8): bias 15, 2 mantissa bits, subnormals, infinities and NaN
 *    at exponent 31 (the upper byte of a binary16), max 57344;
 *  - i8: two's-complement integers -128..127.
 * The k_scale / v_scale dequant factors multiply the decoded K / V values.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int64_t num_q_tokens, num_q_heads, num_kv_heads, head_dim;
    int64_t total_num_pages, page_size, max_num_seqs, pages_per_seq;
    int32_t kv_dtype; /* OracleKv: element type of kv_pages */
    int32_t is_causal;
    double sm_scale;
    int32_t has_soft_cap;
    int32_t has_k_scale;
    double soft_cap;
    double k_scale;
    int32_t has_v_scale;
    int32_t has_sliding_window;
    double v_scale;
    int64_t sliding_window;
    int32_t has_sinks;
    const double* sinks; /* [num_q_heads] sink logits when has_sinks */
    int32_t q_dtype;     /* OracleQ: element type of q */
    int32_t latent;      /* 1: latent cache layout (one row per kv head; V = its first v_head_dim) */
    int64_t v_head_dim;  /* width of V and o (head_dim unless latent) */
} OracleCfg;

enum { OR_OK = 0, OR_INVALID_ARG = 1, OR_BAD_PAGE_INDEX = 4, OR_BAD_LENGTHS = 5 };
typedef enum { OKV_BF16 = 0, OKV_E4M3 = 1, OKV_F16 = 2, OKV_E5M2 = 3, OKV_I8 = 4 } OracleKv;
typedef enum { OQ_BF16 = 0, OQ_F16 = 1, OQ_F32 = 2 } OracleQ;

/* bf16: the 16 stored bits are the upper half of an IEEE-754 binary32. */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp8 e4m3fn (OCP FP8): 1 sign, 4 exponent (bias 7), 3 mantissa bits. */
double oracle_e4m3_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7); /* subnormal */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* f16 (IEEE binary16): 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double oracle_f16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 10) & 0x1F;
    int m = b & 0x3FF;
    double v;
    if (e == 0x1F) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m / 1024.0, 1 - 15); /* subnormal */
    else v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -v : v;
}

/* fp8 e5m2 (OCP FP8): 1 sign, 5 exponent (bias 15), 2 mantissa bits. */
double oracle_e5m2_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1F;
    int m = b & 0x3;
    double v;
    if (e == 0x1F) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m / 4.0, 1 - 15); /* subnormal */
    else v = ldexp(1.0 + (double)m / 4.0, e - 15);
    return sign ? -v : v;
}

/* f32 (IEEE binary32) */
static double f32_to_f64(const void* p) {
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

/* Mask of the page (flashAttention): a key is dropped when it is past the
 * sequence, when causal and j > p, or when p - sliding_window >= j. */
static int key_allowed(const OracleCfg* c, int64_t kv_len, int64_t p, int64_t j) {
    if (j >= kv_len) return 0;
    if (c->is_causal && j > p) return 0;
    if (c->has_sliding_window && p - c->sliding_window >= j) return 0;
    return 1;
}

/* Element d of the K row (is_v = 0) or V row (is_v = 1) of kv head h in a page slot. */
static double kv_elem(const OracleCfg* c, const void* kv, int64_t page, int64_t slot, int64_t h, int is_v,
                      int64_t d) {
    int64_t idx;
    if (c->latent) /* [N, ps, Hkv, D]: K and V share the row */
        idx = ((page * c->page_size + slot) * c->num_kv_heads + h) * c->head_dim + d;
    else /* [N, ps, 2 Hkv, D]: combined head 2h = K, 2h + 1 = V */
        idx = ((page * c->page_size + slot) * (2 * c->num_kv_heads) + 2 * h + is_v) * c->head_dim + d;
    switch (c->kv_dtype) {
        case OKV_E4M3: return oracle_e4m3_to_f64(((const uint8_t*)kv)[idx]);
        case OKV_E5M2: return oracle_e5m2_to_f64(((const uint8_t*)kv)[idx]);
        case OKV_I8: return (double)((const int8_t*)kv)[idx];
        case OKV_F16: return oracle_f16_to_f64(((const uint16_t*)kv)[idx]);
        default: return oracle_bf16_to_f64(((const uint16_t*)kv)[idx]);
    }
}

static double q_elem(const OracleCfg* c, const void* q, int64_t idx) {
    switch (c->q_dtype) {
        case OQ_F32: return f32_to_f64((const float*)q + idx);
        case OQ_F16: return oracle_f16_to_f64(((const uint16_t*)q)[idx]);
        default: return oracle_bf16_to_f64(((const uint16_t*)q)[idx]);
    }
}

/* Lengths / page-table validity, stated as the preconditions of the method.
 * Returns OR_OK, OR_BAD_LENGTHS or OR_BAD_PAGE_INDEX (lengths checked first). */
int rpa_oracle_validate(const OracleCfg* c, const int32_t* kv_lens, const int32_t* page_indices,
                        const int32_t* cu_q_lens, int32_t num_seqs) {
    if (num_seqs < 0 || num_seqs > c->max_num_seqs) return OR_BAD_LENGTHS;
    if (cu_q_lens[0] < 0) return OR_BAD_LENGTHS;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int64_t q0 = cu_q_lens[s], q1 = cu_q_lens[s + 1], kl = kv_lens[s];
        if (q1 < q0) return OR_BAD_LENGTHS;
        if (kl < 0 || kl > c->pages_per_seq * c->page_size) return OR_BAD_LENGTHS;
        if (q1 - q0 > kl) return OR_BAD_LENGTHS;
    }
    if (cu_q_lens[num_seqs] > c->num_q_tokens) return OR_BAD_LENGTHS;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int64_t kl = kv_lens[s];
        int64_t np = (kl + c->page_size - 1) / c->page_size;
        for (int64_t j = 0; j < np; ++j) {
            int32_t pg = page_indices[(int64_t)s * c->pages_per_seq + j];
            if (pg < 0 || pg >= c->total_num_pages) return OR_BAD_PAGE_INDEX;
        }
    }
    return OR_OK;
}

/* One output row: query token t (of sequence s, local index i), query head qh.
 * scratch holds kv_len doubles. */
static void one_row(const OracleCfg* c, const void* q, const void* kv, const int32_t* kv_lens,
                    const int32_t* page_indices, const int32_t* cu_q_lens, int32_t s, int64_t t,
                    int64_t qh, double* out, double* x) {
    const int64_t D = c->head_dim;
    const int64_t Dv = c->v_head_dim; /* width of V and of the output row */
    const int64_t G = c->num_q_heads / c->num_kv_heads;
    const int64_t h = qh / G;
    const int64_t q_len = (int64_t)cu_q_lens[s + 1] - cu_q_lens[s];
    const int64_t kv_len = kv_lens[s];
    const int64_t i = t - cu_q_lens[s];
    const int64_t p = kv_len - q_len + i;
    const double ks = c->has_k_scale ? c->k_scale : 1.0;
    const double vs = c->has_v_scale ? c->v_scale : 1.0;
    const int64_t qrow = (t * c->num_q_heads + qh) * D; /* element offset of the query row */

    for (int64_t d = 0; d < Dv; ++d) out[d] = 0.0;
    double xmax = -INFINITY;
    int any = 0;
    /* a sink logit starts the row maximum */
    if (c->has_sinks) xmax = c->sinks[qh];
    for (int64_t j = 0; j < kv_len; ++j) {
        if (!key_allowed(c, kv_len, p, j)) continue;
        int64_t page = page_indices[(int64_t)s * c->pages_per_seq + j / c->page_size];
        int64_t slot = j % c->page_size;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += q_elem(c, q, qrow + d) * (kv_elem(c, kv, page, slot, h, 0, d) * ks);
        double xj = c->sm_scale * dot;
        if (c->has_soft_cap) xj = c->soft_cap * tanh(xj / c->soft_cap);
        x[j] = xj;
        if (xj > xmax) xmax = xj;
        any = 1;
    }
    if (!any) return; /* no allowed key: row is 0 (with a sink too: its term carries no value) */
    double denom = 0.0;
    /* the sink's term joins the denominator and takes no value */
    if (c->has_sinks) denom += exp(c->sinks[qh] - xmax);
    for (int64_t j = 0; j < kv_len; ++j) {
        if (!key_allowed(c, kv_len, p, j)) continue;
        double w = exp(x[j] - xmax);
        denom += w;
        int64_t page = page_indices[(int64_t)s * c->pages_per_seq + j / c->page_size];
        int64_t slot = j % c->page_size;
        for (int64_t d = 0; d < Dv; ++d) out[d] += w * (kv_elem(c, kv, page, slot, h, 1, d) * vs);
    }
    for (int64_t d = 0; d < Dv; ++d) out[d] /= denom;
}

static int32_t seq_of_token(const int32_t* cu_q_lens, int32_t num_seqs, int64_t t) {
    /* Last s with cu_q_lens[s] <= t < cu_q_lens[s+1]; -1 if none. */
    for (int32_t s = 0; s < num_seqs; ++s)
        if (t >= cu_q_lens[s] && t < cu_q_lens[s + 1]) return s;
    return -1;
}

typedef struct {
    const OracleCfg* c;
    const void* q;
    const void* kv;
    const int32_t* kv_lens;
    const int32_t* page_indices;
    const int32_t* cu_q_lens;
    int32_t num_seqs;
    const int64_t* rows; /* (token, q head) pairs, or NULL for all rows */
    int64_t nrows;
    double* out;
    int64_t next;
    int64_t max_kv;
} Job;

static void* worker(void* arg) {
    Job* jb = (Job*)arg;
    const OracleCfg* c = jb->c;
    const int64_t D = c->v_head_dim; /* output row width */
    double* x = (double*)malloc(sizeof(double) * (size_t)(jb->max_kv > 0 ? jb->max_kv : 1));
    for (;;) {
        int64_t r = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (r >= jb->nrows) break;
        int64_t t, qh;
        if (jb->rows) {
            t = jb->rows[2 * r];
            qh = jb->rows[2 * r + 1];
        } else {
            t = r / c->num_q_heads;
            qh = r % c->num_q_heads;
        }
        double* o = jb->out + r * D;
        int32_t s = seq_of_token(jb->cu_q_lens, jb->num_seqs, t);
        if (s < 0) {
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        one_row(c, jb->q, jb->kv, jb->kv_lens, jb->page_indices, jb->cu_q_lens, s, t, qh, o, x);
    }
    free(x);
    return NULL;
}

static int run_job(Job* jb, int nthreads) {
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    jb->max_kv = 0;
    for (int32_t s = 0; s < jb->num_seqs; ++s)
        if (jb->kv_lens[s] > jb->max_kv) jb->max_kv = jb->kv_lens[s];
    pthread_t th[256];
    int started = 0;
    for (int k = 0; k < nthreads; ++k) {
        if (pthread_create(&th[k], NULL, worker, jb) != 0) break;
        ++started;
    }
    if (started == 0) worker(jb);
    for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
    return started > 0 ? started : 1;
}

/* All rows: out[num_q_tokens, num_q_heads, v_head_dim] in fp64.
 * Returns the number of threads used, or -code on invalid input. */
static int cfg_ok(const OracleCfg* c) {
    if (!c || c->num_kv_heads <= 0 || c->num_q_heads % c->num_kv_heads) return 0;
    if (c->v_head_dim < 1 || c->v_head_dim > c->head_dim || (!c->latent && c->v_head_dim != c->head_dim)) return 0;
    return 1;
}

int rpa_oracle_forward(const OracleCfg* c, const void* q, const void* kv_pages,
                       const int32_t* kv_lens, const int32_t* page_indices, const int32_t* cu_q_lens,
                       int32_t num_seqs, double* out, int nthreads) {
    if (!cfg_ok(c)) return -OR_INVALID_ARG;
    int v = rpa_oracle_validate(c, kv_lens, page_indices, cu_q_lens, num_seqs);
    if (v) return -v;
    Job jb = {c, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, NULL,
              c->num_q_tokens * c->num_q_heads, out, 0, 0};
    return run_job(&jb, nthreads);
}

/* Selected rows only: rows = nrows (token, q head) int64 pairs; out[nrows, v_head_dim]. */
int rpa_oracle_rows(const OracleCfg* c, const void* q, const void* kv_pages, const int32_t* kv_lens,
                    const int32_t* page_indices, const int32_t* cu_q_lens, int32_t num_seqs,
                    const int64_t* rows, int64_t nrows, double* out, int nthreads) {
    if (!cfg_ok(c)) return -OR_INVALID_ARG;
    int v = rpa_oracle_validate(c, kv_lens, page_indices, cu_q_lens, num_seqs);
    if (v) return -v;
    Job jb = {c, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, rows, nrows, out, 0, 0};
    return run_job(&jb, nthreads);
}
