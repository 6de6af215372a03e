/*
 * fp64 CPU oracle for paged grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg do.  It shares no code, header or constant
 * with the CUDA library.
 *
 * What it computes, and where the pages define it
 * ------------------------------------------------
 * The KV cache is one unified pool from which every request takes pages;
 * a page is the pool's allocation unit and its size is configurable
 * ("Mini-SGLang 实战指南", §6.2 "Page Size" and §6.5 "Radix Cache";
 * "不懂SGLang？从miniSGLang开始", §1.2 "调度引擎").  Attention reads
 * the pool's history plus the newly computed K/V, and finds each request's
 * data through the page table and the positions
 * ("不懂SGLang？从miniSGLang开始", §1.3 "前向运算", items 1 and 3).  A
 * prefill chunk attends to the request's cached prefix and to itself,
 * causally ("Mini-SGLang 实战指南", §6.1 "Chunked Prefill" and §6.5).
 *
 * The pages give no formula, so this is the plain definition of causal
 * softmax attention written out term by term, per query row and query head:
 *
 *   slot(j)  = page_table[b][j / page_size] * page_size + j % page_size
 *   g        = h / (Hq / Hkv)                    (consecutive q heads share)
 *   s_j      = scale * sum_d q[d] * K[slot(j)][g][d]        for j = 0..p
 *   m        = max_j s_j
 *   w_j      = exp(s_j - m),  Z = sum_j w_j
 *   o[d]     = sum_j w_j * V[slot(j)][g][d] / Z
 *   lse      = m + ln Z                           (natural log)
 *
 * where p is the row's absolute position; keys j > p are never gathered.
 * Every bf16 input is widened to fp64 exactly; all arithmetic is fp64.
 *
 * The store step is a byte copy: pool[out_loc[t]] = new[t].
 *
 * Compile-time switch ORACLE_MUTANT (default 0) plants one deliberate
 * mistake; the CPU tests build those variants to show that each planted
 * mistake fails at least one pin.  The default build never defines it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_OUT_OF_RANGE 4

/* bf16 bit pattern -> fp64, exact (a bf16 is the top half of an fp32). */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------- store */

int oracle_store_kv(uint16_t *k_pool, uint16_t *v_pool, int64_t num_slots,
                    int32_t num_kv_heads, int32_t head_dim,
                    const uint16_t *k_new, const uint16_t *v_new,
                    const int32_t *out_loc, int64_t n_tokens) {
    if (num_slots < 0 || num_kv_heads <= 0 || head_dim <= 0 || n_tokens < 0)
        return ORACLE_BAD_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t s = out_loc[t];
        if (s < 0 || s >= num_slots) return ORACLE_OUT_OF_RANGE;
        memcpy(k_pool + s * row, k_new + t * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_pool + s * row, v_new + t * row, (size_t)row * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------ attention */

/*
 * One work item = one (request b, query row r, query head h).  The row's
 * query vector is q[qrow][h][:], its absolute position is pos, and it
 * writes o[item][:] and lse[item].
 */
typedef struct {
    const uint16_t *q;
    int32_t hq, hkv, d;
    const uint16_t *k_pool, *v_pool;
    int64_t num_slots;
    int32_t page_size;
    const int32_t *page_table;
    int64_t pt_stride;
    int32_t pt_width; /* valid entries per page-table row */
    double scale;
    int64_t n_items;
    const int32_t *item_req, *item_qrow, *item_pos, *item_head;
    double *o, *lse;
    int status; /* first error seen (written under no lock; any nonzero wins) */
    int64_t next; /* work counter */
    pthread_mutex_t lock;
} attn_job;

static int64_t slot_of(const attn_job *J, int32_t b, int64_t j, int *err) {
    int64_t page_idx = j / J->page_size;
    if (page_idx >= J->pt_width) { *err = ORACLE_OUT_OF_RANGE; return 0; }
    int64_t page = J->page_table[(int64_t)b * J->pt_stride + page_idx];
#if ORACLE_MUTANT == 5
    int64_t slot = page + j % J->page_size;              /* page id used as a slot */
#else
    int64_t slot = page * J->page_size + j % J->page_size;
#endif
    if (page < 0 || slot < 0 || slot >= J->num_slots) { *err = ORACLE_OUT_OF_RANGE; return 0; }
    return slot;
}

static int attn_item(const attn_job *J, int64_t it, double *s_buf, double *q_buf) {
    const int32_t b = J->item_req[it], qrow = J->item_qrow[it];
    const int32_t h = J->item_head[it];
    const int64_t p = J->item_pos[it];
    const int32_t d = J->d;
    const int32_t group = J->hq / J->hkv;
#if ORACLE_MUTANT == 2
    const int32_t g = h % J->hkv;                         /* interleaved head map */
#else
    const int32_t g = h / group;
#endif
    double *o = J->o + it * d;
    if (p < 0) return ORACLE_BAD_ARG;
#if ORACLE_MUTANT == 1
    const int64_t n_keys = p;                             /* drops the diagonal key */
#else
    const int64_t n_keys = p + 1;                         /* keys 0..p inclusive */
#endif
    const uint16_t *qv = J->q + ((int64_t)qrow * J->hq + h) * d;
    for (int32_t x = 0; x < d; ++x) q_buf[x] = bf16_to_f64(qv[x]);

    /* 1. scores of the gathered keys */
    int err = 0;
    for (int64_t j = 0; j < n_keys; ++j) {
        int64_t slot = slot_of(J, b, j, &err);
        if (err) return err;
        const uint16_t *kv = J->k_pool + (slot * J->hkv + g) * d;
        double acc = 0.0;
        for (int32_t x = 0; x < d; ++x) acc += q_buf[x] * bf16_to_f64(kv[x]);
#if ORACLE_MUTANT == 3
        s_buf[j] = acc;                                   /* scale dropped */
#else
        s_buf[j] = J->scale * acc;
#endif
    }
    /* 2. softmax: max, weights, normaliser */
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) if (s_buf[j] > m) m = s_buf[j];
    double z = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) { s_buf[j] = exp(s_buf[j] - m); z += s_buf[j]; }
    /* 3. weighted sum of values */
    for (int32_t x = 0; x < d; ++x) o[x] = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        int64_t slot = slot_of(J, b, j, &err);
        if (err) return err;
#if ORACLE_MUTANT == 7
        const uint16_t *vv = J->k_pool + (slot * J->hkv + g) * d;  /* K used as V */
#else
        const uint16_t *vv = J->v_pool + (slot * J->hkv + g) * d;
#endif
        for (int32_t x = 0; x < d; ++x) o[x] += s_buf[j] * bf16_to_f64(vv[x]);
    }
#if ORACLE_MUTANT != 8
    for (int32_t x = 0; x < d; ++x) o[x] /= z;            /* (mutant 8: unnormalised) */
#endif
#if ORACLE_MUTANT == 4
    J->lse[it] = (m + log(z)) / log(2.0);                 /* log2 instead of ln */
#else
    J->lse[it] = m + log(z);
#endif
    return ORACLE_OK;
}

static void *attn_worker(void *arg) {
    attn_job *J = (attn_job *)arg;
    int64_t max_keys = 1;
    for (int64_t i = 0; i < J->n_items; ++i)
        if ((int64_t)J->item_pos[i] + 1 > max_keys) max_keys = (int64_t)J->item_pos[i] + 1;
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)max_keys);
    double *q_buf = (double *)malloc(sizeof(double) * (size_t)J->d);
    if (!s_buf || !q_buf) {
        pthread_mutex_lock(&J->lock);
        J->status = ORACLE_BAD_ARG;
        pthread_mutex_unlock(&J->lock);
        free(s_buf); free(q_buf);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t it = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (it >= J->n_items) break;
        int rc = attn_item(J, it, s_buf, q_buf);
        if (rc) {
            pthread_mutex_lock(&J->lock);
            if (!J->status) J->status = rc;
            pthread_mutex_unlock(&J->lock);
        }
    }
    free(s_buf); free(q_buf);
    return NULL;
}

/*
 * Attention for an explicit list of (request, query row, position, head)
 * items.  q: bf16 bits [*, hq, d]; pools: bf16 bits [num_slots, hkv, d];
 * page_table: int32 [num_reqs, pt_stride] (pt_width valid columns).
 * Outputs: o fp64 [n_items, d], lse fp64 [n_items].  Returns 0 on success.
 */
int oracle_attention_items(const uint16_t *q, int32_t hq, int32_t hkv, int32_t d,
                           const uint16_t *k_pool, const uint16_t *v_pool,
                           int64_t num_slots, int32_t page_size,
                           const int32_t *page_table, int64_t pt_stride, int32_t pt_width,
                           double scale, int64_t n_items,
                           const int32_t *item_req, const int32_t *item_qrow,
                           const int32_t *item_pos, const int32_t *item_head,
                           double *o, double *lse, int32_t n_threads) {
    if (hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0 || page_size <= 0 || n_items < 0)
        return ORACLE_BAD_ARG;
    attn_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.hq = hq; J.hkv = hkv; J.d = d;
    J.k_pool = k_pool; J.v_pool = v_pool; J.num_slots = num_slots;
    J.page_size = page_size; J.page_table = page_table;
    J.pt_stride = pt_stride; J.pt_width = pt_width; J.scale = scale;
    J.n_items = n_items; J.item_req = item_req; J.item_qrow = item_qrow;
    J.item_pos = item_pos; J.item_head = item_head; J.o = o; J.lse = lse;
    pthread_mutex_init(&J.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 0; i < n_threads; ++i)
        if (pthread_create(&th[i], NULL, attn_worker, &J) == 0) ++started;
    if (started == 0) attn_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&J.lock);
    return J.status;
}

/* Which planted mistake this build carries (0 = none). */
int oracle_mutant_id(void) { return ORACLE_MUTANT; }
