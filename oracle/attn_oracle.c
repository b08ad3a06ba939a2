/*
 * attn_oracle.c -- plain fp64 CPU oracle for scaled-dot-product attention
 * (forward with log-sum-exp stats, FlashAttention-2 style backward) and for
 * the NSA selected-attention backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA product path
 * shares no code with it and never calls it.
 *
 * Everything here is the textbook definition written out, with no tiling, no
 * online softmax and no blocking:
 *
 *   s_ij  = scale * q_i . k_j                    (multiplicative scale:
 *           cuDNN-frontend sample "51_scaled_dot_product_attention_backward",
 *           cell "Problem sizes", attn_scale = 1/sqrt(d))
 *   vis   = mask predicate (none / causal top-left / causal bottom-right)
 *   LSE_i = log sum_{j vis} exp(s_ij)            (the fp32 "stats" of shape
 *           (B,H,S,1) the same sample passes from forward to backward)
 *   P_ij  = exp(s_ij - LSE_i) if vis, else 0
 *   O_i   = sum_j P_ij v_j
 *   D_i   = dO_i . O_i                           (O as supplied by the caller)
 *   dP_ij = dO_i . v_j
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j  = scale sum_{i, heads of the group} dS_ij q_i
 *   dV_j  = sum_{i, heads of the group} P_ij dO_i
 *
 * The last three are the gradient formulas of the Ascend CANN page
 * "aclnnNsaSelectedAttentionGrad", section Function / Formula
 * (dV = P^T dY, dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d)), with the
 * 1/sqrt(d) taken as the caller's scale.  The sample notebook names the
 * FlashAttention-2 algorithm for the backward; D, P, dP and dS above are
 * that algorithm's standard intermediate quantities.
 *
 * NSA (same Ascend page, Function / Formula): per query token t and kv head
 * g the selected key set is the union over c < selectedBlockCount of the
 * blocks [topk[t,g,c] * bs, topk[t,g,c] * bs + bs) of the token's own
 * sequence.  The keys and values are gathered explicitly, the backward above
 * runs on the gathered rows, and the gathered dK / dV rows are added back to
 * the rows they came from.  The softmax stats are the page's softmaxMax and
 * softmaxSum: P = exp(s - max) / sum.  The page's attenMaskOptional (2-D,
 * BOOL / UINT8, in the signature and the parameter table, used by no formula)
 * is read as: entry (i, j) nonzero removes key j for query i, positions local
 * to the sequence, on top of the selection and the sparse mode.
 *
 * Layout of every tensor here (fp64): token-major "TND"
 *   q, o, dO, dq : [Tq][h][d]      k, v, dk, dv : [Tkv][h_kv][d]
 *   (NSA: v, dv, o and dO have the value head dim d_v, which the Ascend
 *   page's constraints let differ from the query / key head dim d)
 *   lse, max, sum: [Tq][h]         topk         : [Tq][h_kv][cnt] (int32)
 * Sequences are given by inclusive cumulative lengths (no leading zero), as
 * the Ascend page's actualSeqQLen / actualSeqKvLen are.  A fixed-length batch
 * is the special case cu = {S, 2S, ...}.
 * Query head hq belongs to kv head hq / (h / h_kv).
 * A row with no visible key has O = 0, LSE = +inf and P = 0.
 *
 * Parity unpinned (conventions the Ascend page leaves open; no value on any
 * page fixes them, so no test can pin them):
 *   - sparse_mode 2 is read as causal bottom-right on the sequence's key
 *     positions, sparse_mode 0 as no mask beyond the selection;
 *   - softmaxMax / softmaxSum hold one value per (token, head), replicated
 *     over their 8 lanes; lane 0 is read;
 *   - topk block ids are local to the token's sequence (block c covers keys
 *     [c*bs, c*bs + bs) of that sequence) and must be distinct.
 * Everything else is pinned by the tests: finite differences, softmax
 * invariants, closed forms and a second, masked-dense NSA path.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORA_OK 0
#define ORA_ERR 1

/* ------------------------------------------------------------------------ */
/* problem descriptions                                                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t nseq;          /* number of sequences                              */
    const int64_t *cu_q;   /* inclusive cumulative query lengths, nseq entries  */
    const int64_t *cu_kv;  /* inclusive cumulative key lengths, nseq entries    */
    int64_t h, h_kv, d;    /* query heads, key/value heads, head dimension      */
    double scale;          /* multiplies q.k                                    */
    int mask;              /* 0 none, 1 causal top-left, 2 causal bottom-right  */
} ora_dense_t;

typedef struct {
    int64_t nseq;
    const int64_t *cu_q, *cu_kv;
    int64_t n1, n2, d;     /* query heads, kv heads, head dimension             */
    double scale;
    int64_t block_size;    /* selectedBlockSize                                 */
    int64_t block_count;   /* selectedBlockCount                                */
    int sparse_mode;       /* 0: no mask beyond the selection; 2: causal
                              bottom-right on the sequence's key positions      */
    int64_t d_v;           /* head dim of value, attentionOut and dY (the page
                              allows it to differ from the query / key head
                              dim d); 0: equal to d                             */
    const uint8_t *atten_mask; /* attenMaskOptional: NULL, or [mask_rows][mask_cols]
                              with nonzero = key j removed for query i (local
                              positions), on top of the selection and the
                              sparse mode                                       */
    int64_t mask_rows, mask_cols;
} ora_nsa_t;

static int64_t value_dim(const ora_nsa_t *pb) { return pb->d_v > 0 ? pb->d_v : pb->d; }

static int64_t seq_start(const int64_t *cu, int64_t b) { return b == 0 ? 0 : cu[b - 1]; }
static int64_t seq_len(const int64_t *cu, int64_t b) { return cu[b] - seq_start(cu, b); }

/* Visibility of key j (local to its sequence) to query i (local).            */
static int visible(int mask, int64_t i, int64_t j, int64_t lq, int64_t lkv)
{
    if (mask == 1) return j <= i;
    if (mask == 2) return j <= i + (lkv - lq);
    return 1;
}

static double dot(const double *a, const double *b, int64_t n)
{
    double s = 0.0;
    for (int64_t x = 0; x < n; ++x) s += a[x] * b[x];
    return s;
}

/* ------------------------------------------------------------------------ */
/* a tiny work-sharing pool: units are claimed from an atomic counter        */
/* ------------------------------------------------------------------------ */

typedef void (*unit_fn)(void *ctx, int64_t unit);
typedef struct {
    unit_fn fn;
    void *ctx;
    int64_t nunits;
    atomic_llong next;
} pool_t;

static void *pool_worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    for (;;) {
        int64_t u = atomic_fetch_add(&p->next, 1);
        if (u >= p->nunits) break;
        p->fn(p->ctx, u);
    }
    return NULL;
}

static int ora_threads_default(void)
{
    const char *e = getenv("ORACLE_THREADS");
    if (e && atoi(e) > 0) return atoi(e);
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_units(unit_fn fn, void *ctx, int64_t nunits, int nthreads)
{
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.nunits = nunits;
    atomic_init(&p.next, 0);
    if (nthreads <= 0) nthreads = ora_threads_default();
    if (nthreads > nunits) nthreads = (int)(nunits > 0 ? nunits : 1);
    if (nthreads <= 1) {
        pool_worker(&p);
        return;
    }
    pthread_t *t = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&t[i], NULL, pool_worker, &p);
    for (int i = 0; i < nthreads; ++i) pthread_join(t[i], NULL);
    free(t);
}

int ora_thread_count(void) { return ora_threads_default(); }

/* ======================================================================== */
/* dense attention                                                          */
/* ======================================================================== */

typedef struct {
    const ora_dense_t *pb;
    const double *q, *k, *v, *o, *dout, *lse;
    double *o_out, *lse_out, *dq, *dk, *dv;
} dense_ctx;

/* Forward for one (sequence, kv head) unit: every query head of the group. */
static void dense_fwd_unit(void *vctx, int64_t unit)
{
    dense_ctx *c = (dense_ctx *)vctx;
    const ora_dense_t *pb = c->pb;
    const int64_t b = unit / pb->h_kv, g = unit % pb->h_kv;
    const int64_t G = pb->h / pb->h_kv, d = pb->d;
    const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
    const int64_t k0 = seq_start(pb->cu_kv, b), lkv = seq_len(pb->cu_kv, b);
    double *s = (double *)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1));
    for (int64_t hq = g * G; hq < (g + 1) * G; ++hq) {
        for (int64_t i = 0; i < lq; ++i) {
            const double *qi = c->q + ((q0 + i) * pb->h + hq) * d;
            double *oi = c->o_out + ((q0 + i) * pb->h + hq) * d;
            double mx = -INFINITY;
            for (int64_t j = 0; j < lkv; ++j) {
                if (!visible(pb->mask, i, j, lq, lkv)) continue;
                s[j] = pb->scale * dot(qi, c->k + ((k0 + j) * pb->h_kv + g) * d, d);
                if (s[j] > mx) mx = s[j];
            }
            for (int64_t x = 0; x < d; ++x) oi[x] = 0.0;
            if (mx == -INFINITY) { /* no visible key */
                c->lse_out[(q0 + i) * pb->h + hq] = INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int64_t j = 0; j < lkv; ++j)
                if (visible(pb->mask, i, j, lq, lkv)) sum += exp(s[j] - mx);
            const double lse = mx + log(sum);
            c->lse_out[(q0 + i) * pb->h + hq] = lse;
            for (int64_t j = 0; j < lkv; ++j) {
                if (!visible(pb->mask, i, j, lq, lkv)) continue;
                const double p = exp(s[j] - lse);
                const double *vj = c->v + ((k0 + j) * pb->h_kv + g) * d;
                for (int64_t x = 0; x < d; ++x) oi[x] += p * vj[x];
            }
        }
    }
    free(s);
}

/* Backward for one (sequence, kv head) unit.  The unit owns the dK / dV rows
 * of its kv head in its sequence and the dQ rows of its query heads.        */
static void dense_bwd_unit(void *vctx, int64_t unit)
{
    dense_ctx *c = (dense_ctx *)vctx;
    const ora_dense_t *pb = c->pb;
    const int64_t b = unit / pb->h_kv, g = unit % pb->h_kv;
    const int64_t G = pb->h / pb->h_kv, d = pb->d;
    const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
    const int64_t k0 = seq_start(pb->cu_kv, b), lkv = seq_len(pb->cu_kv, b);
    for (int64_t j = 0; j < lkv; ++j)
        for (int64_t x = 0; x < d; ++x) {
            c->dk[((k0 + j) * pb->h_kv + g) * d + x] = 0.0;
            c->dv[((k0 + j) * pb->h_kv + g) * d + x] = 0.0;
        }
    for (int64_t hq = g * G; hq < (g + 1) * G; ++hq) {
        for (int64_t i = 0; i < lq; ++i) {
            const int64_t row = (q0 + i) * pb->h + hq;
            const double *qi = c->q + row * d, *oi = c->o + row * d, *doi = c->dout + row * d;
            double *dqi = c->dq + row * d;
            const double lse = c->lse[row];
            const double Di = dot(doi, oi, d);
            for (int64_t x = 0; x < d; ++x) dqi[x] = 0.0;
            for (int64_t j = 0; j < lkv; ++j) {
                if (!visible(pb->mask, i, j, lq, lkv)) continue;
                const double *kj = c->k + ((k0 + j) * pb->h_kv + g) * d;
                const double *vj = c->v + ((k0 + j) * pb->h_kv + g) * d;
                double *dkj = c->dk + ((k0 + j) * pb->h_kv + g) * d;
                double *dvj = c->dv + ((k0 + j) * pb->h_kv + g) * d;
                const double p = (lse == INFINITY) ? 0.0 : exp(pb->scale * dot(qi, kj, d) - lse);
                const double dp = dot(doi, vj, d);
                const double ds = p * (dp - Di);
                for (int64_t x = 0; x < d; ++x) {
                    dqi[x] += pb->scale * ds * kj[x];
                    dkj[x] += pb->scale * ds * qi[x];
                    dvj[x] += p * doi[x];
                }
            }
        }
    }
}

int ora_dense_fwd(const ora_dense_t *pb, const double *q, const double *k, const double *v,
                  double *o, double *lse, int nthreads)
{
    if (!pb || !q || !k || !v || !o || !lse || pb->h_kv <= 0 || pb->h % pb->h_kv) return ORA_ERR;
    dense_ctx c;
    memset(&c, 0, sizeof c);
    c.pb = pb; c.q = q; c.k = k; c.v = v; c.o_out = o; c.lse_out = lse;
    run_units(dense_fwd_unit, &c, pb->nseq * pb->h_kv, nthreads);
    return ORA_OK;
}

int ora_dense_bwd(const ora_dense_t *pb, const double *q, const double *k, const double *v,
                  const double *o, const double *dout, const double *lse,
                  double *dq, double *dk, double *dv, int nthreads)
{
    if (!pb || !q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ORA_ERR;
    if (pb->h_kv <= 0 || pb->h % pb->h_kv) return ORA_ERR;
    dense_ctx c;
    memset(&c, 0, sizeof c);
    c.pb = pb; c.q = q; c.k = k; c.v = v; c.o = o; c.dout = dout; c.lse = lse;
    c.dq = dq; c.dk = dk; c.dv = dv;
    run_units(dense_bwd_unit, &c, pb->nseq * pb->h_kv, nthreads);
    return ORA_OK;
}

/* Sampled backward: the same formulas evaluated for chosen output rows only.
 * q_rows[r]  = token * h + head      -> dq_out[r][d]
 * kv_rows[r] = token * h_kv + head   -> dk_out[r][d], dv_out[r][d]
 * lse must be the full [Tq][h] array (each dK / dV row needs every query
 * row's stats).                                                             */
typedef struct {
    dense_ctx base;
    int64_t nq, nkv;
    const int64_t *q_rows, *kv_rows;
    double *dq_out, *dk_out, *dv_out;
} rows_ctx;

static int64_t seq_of(const int64_t *cu, int64_t nseq, int64_t t)
{
    for (int64_t b = 0; b < nseq; ++b)
        if (t < cu[b]) return b;
    return -1;
}

static void dense_rows_unit(void *vctx, int64_t r)
{
    rows_ctx *rc = (rows_ctx *)vctx;
    const dense_ctx *c = &rc->base;
    const ora_dense_t *pb = c->pb;
    const int64_t G = pb->h / pb->h_kv, d = pb->d;
    if (r < rc->nq) {
        const int64_t t = rc->q_rows[r] / pb->h, hq = rc->q_rows[r] % pb->h, g = hq / G;
        const int64_t b = seq_of(pb->cu_q, pb->nseq, t);
        const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
        const int64_t k0 = seq_start(pb->cu_kv, b), lkv = seq_len(pb->cu_kv, b);
        const int64_t i = t - q0, row = t * pb->h + hq;
        const double *qi = c->q + row * d, *oi = c->o + row * d, *doi = c->dout + row * d;
        const double lse = c->lse[row], Di = dot(doi, oi, d);
        double *out = rc->dq_out + r * d;
        for (int64_t x = 0; x < d; ++x) out[x] = 0.0;
        for (int64_t j = 0; j < lkv; ++j) {
            if (!visible(pb->mask, i, j, lq, lkv) || lse == INFINITY) continue;
            const double *kj = c->k + ((k0 + j) * pb->h_kv + g) * d;
            const double *vj = c->v + ((k0 + j) * pb->h_kv + g) * d;
            const double p = exp(pb->scale * dot(qi, kj, d) - lse);
            const double ds = p * (dot(doi, vj, d) - Di);
            for (int64_t x = 0; x < d; ++x) out[x] += pb->scale * ds * kj[x];
        }
        return;
    }
    r -= rc->nq;
    const int64_t tk = rc->kv_rows[r] / pb->h_kv, g = rc->kv_rows[r] % pb->h_kv;
    const int64_t b = seq_of(pb->cu_kv, pb->nseq, tk);
    const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
    const int64_t k0 = seq_start(pb->cu_kv, b), lkv = seq_len(pb->cu_kv, b);
    const int64_t j = tk - k0;
    const double *kj = c->k + (tk * pb->h_kv + g) * d, *vj = c->v + (tk * pb->h_kv + g) * d;
    double *dko = rc->dk_out + r * d, *dvo = rc->dv_out + r * d;
    for (int64_t x = 0; x < d; ++x) dko[x] = dvo[x] = 0.0;
    for (int64_t hq = g * G; hq < (g + 1) * G; ++hq)
        for (int64_t i = 0; i < lq; ++i) {
            const int64_t row = (q0 + i) * pb->h + hq;
            if (!visible(pb->mask, i, j, lq, lkv) || c->lse[row] == INFINITY) continue;
            const double *qi = c->q + row * d, *oi = c->o + row * d, *doi = c->dout + row * d;
            const double p = exp(pb->scale * dot(qi, kj, d) - c->lse[row]);
            const double ds = p * (dot(doi, vj, d) - dot(doi, oi, d));
            for (int64_t x = 0; x < d; ++x) {
                dko[x] += pb->scale * ds * qi[x];
                dvo[x] += p * doi[x];
            }
        }
}

int ora_dense_bwd_rows(const ora_dense_t *pb, const double *q, const double *k, const double *v,
                       const double *o, const double *dout, const double *lse,
                       int64_t nq, const int64_t *q_rows, double *dq_out,
                       int64_t nkv, const int64_t *kv_rows, double *dk_out, double *dv_out,
                       int nthreads)
{
    if (!pb || !q || !k || !v || !o || !dout || !lse) return ORA_ERR;
    if ((nq && (!q_rows || !dq_out)) || (nkv && (!kv_rows || !dk_out || !dv_out))) return ORA_ERR;
    rows_ctx rc;
    memset(&rc, 0, sizeof rc);
    rc.base.pb = pb; rc.base.q = q; rc.base.k = k; rc.base.v = v; rc.base.o = o;
    rc.base.dout = dout; rc.base.lse = lse;
    rc.nq = nq; rc.nkv = nkv; rc.q_rows = q_rows; rc.kv_rows = kv_rows;
    rc.dq_out = dq_out; rc.dk_out = dk_out; rc.dv_out = dv_out;
    run_units(dense_rows_unit, &rc, nq + nkv, nthreads);
    return ORA_OK;
}

/* ======================================================================== */
/* NSA selected attention                                                   */
/* ======================================================================== */

typedef struct {
    const ora_nsa_t *pb;
    const double *q, *k, *v, *o, *dout, *mx, *sm;
    const int32_t *topk;
    double *o_out, *mx_out, *sm_out, *dq, *dk, *dv;
    int status; /* set to ORA_ERR by any unit that meets a bad index */
} nsa_ctx;

/* Key rows (local to the sequence) of the selected blocks of (t, g), in the
 * order of topk; returns how many, or -1 on an index out of range or one
 * that repeats an earlier slot (the gather would count its keys twice).     */
static int64_t gather_rows(const ora_nsa_t *pb, const int32_t *topk_tg, int64_t lkv, int64_t *rows)
{
    int64_t n = 0;
    for (int64_t c = 0; c < pb->block_count; ++c) {
        const int64_t blk = topk_tg[c];
        if (blk < 0 || (blk + 1) * pb->block_size > lkv) return -1;
        for (int64_t e = 0; e < c; ++e)
            if (topk_tg[e] == blk) return -1;
        for (int64_t r = 0; r < pb->block_size; ++r) rows[n++] = blk * pb->block_size + r;
    }
    return n;
}

/* sparseMode 2 masks key j of query i when j > i + (lkv - lq).              */
static int nsa_mode_visible(const ora_nsa_t *pb, int64_t i, int64_t j, int64_t lq, int64_t lkv)
{
    return pb->sparse_mode == 2 ? visible(2, i, j, lq, lkv) : 1;
}

/* The sparse mode, then attenMaskOptional: a nonzero mask entry (i, j) removes
 * key j for query i.                                                          */
static int nsa_visible(const ora_nsa_t *pb, int64_t i, int64_t j, int64_t lq, int64_t lkv)
{
    if (!nsa_mode_visible(pb, i, j, lq, lkv)) return 0;
    return !(pb->atten_mask && pb->atten_mask[i * pb->mask_cols + j]);
}

static void nsa_fwd_unit(void *vctx, int64_t unit)
{
    nsa_ctx *c = (nsa_ctx *)vctx;
    const ora_nsa_t *pb = c->pb;
    const int64_t b = unit / pb->n2, g = unit % pb->n2, G = pb->n1 / pb->n2, d = pb->d, e = value_dim(pb);
    const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
    const int64_t k0 = seq_start(pb->cu_kv, b), lkv = seq_len(pb->cu_kv, b);
    const int64_t nsel = pb->block_count * pb->block_size;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)nsel);
    double *ksel = (double *)malloc(sizeof(double) * (size_t)(nsel * d));
    double *vsel = (double *)malloc(sizeof(double) * (size_t)(nsel * e));
    double *s = (double *)malloc(sizeof(double) * (size_t)nsel);
    for (int64_t i = 0; i < lq; ++i) {
        const int64_t t = q0 + i;
        if (gather_rows(pb, c->topk + (t * pb->n2 + g) * pb->block_count, lkv, rows) < 0) {
            c->status = ORA_ERR;
            continue;
        }
        /* selectedKey = Gather(key, topk), selectedValue = Gather(value, topk) */
        for (int64_t r = 0; r < nsel; ++r) {
            for (int64_t x = 0; x < d; ++x) ksel[r * d + x] = c->k[((k0 + rows[r]) * pb->n2 + g) * d + x];
            for (int64_t x = 0; x < e; ++x) vsel[r * e + x] = c->v[((k0 + rows[r]) * pb->n2 + g) * e + x];
        }
        for (int64_t hq = g * G; hq < (g + 1) * G; ++hq) {
            const int64_t row = t * pb->n1 + hq;
            const double *qi = c->q + row * d;
            double *oi = c->o_out + row * e;
            double mx = -INFINITY, sum = 0.0;
            for (int64_t r = 0; r < nsel; ++r) {
                if (!nsa_visible(pb, i, rows[r], lq, lkv)) continue;
                s[r] = pb->scale * dot(qi, ksel + r * d, d);
                if (s[r] > mx) mx = s[r];
            }
            for (int64_t x = 0; x < e; ++x) oi[x] = 0.0;
            if (mx != -INFINITY) {
                for (int64_t r = 0; r < nsel; ++r)
                    if (nsa_visible(pb, i, rows[r], lq, lkv)) sum += exp(s[r] - mx);
                for (int64_t r = 0; r < nsel; ++r) {
                    if (!nsa_visible(pb, i, rows[r], lq, lkv)) continue;
                    const double p = exp(s[r] - mx) / sum;
                    for (int64_t x = 0; x < e; ++x) oi[x] += p * vsel[r * e + x];
                }
            }
            c->mx_out[row] = mx;
            c->sm_out[row] = sum;
        }
    }
    free(rows); free(ksel); free(vsel); free(s);
}

/* Backward by explicit gather, dense backward on the gathered rows, then the
 * gathered gradients added back to the rows they came from.                 */
static void nsa_bwd_unit(void *vctx, int64_t unit)
{
    nsa_ctx *c = (nsa_ctx *)vctx;
    const ora_nsa_t *pb = c->pb;
    const int64_t b = unit / pb->n2, g = unit % pb->n2, G = pb->n1 / pb->n2, d = pb->d, e = value_dim(pb);
    const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
    const int64_t k0 = seq_start(pb->cu_kv, b), lkv = seq_len(pb->cu_kv, b);
    const int64_t nsel = pb->block_count * pb->block_size;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)nsel);
    double *ksel = (double *)malloc(sizeof(double) * (size_t)(nsel * d));
    double *vsel = (double *)malloc(sizeof(double) * (size_t)(nsel * e));
    double *dksel = (double *)malloc(sizeof(double) * (size_t)(nsel * d));
    double *dvsel = (double *)malloc(sizeof(double) * (size_t)(nsel * e));
    for (int64_t j = 0; j < lkv; ++j) {
        for (int64_t x = 0; x < d; ++x) c->dk[((k0 + j) * pb->n2 + g) * d + x] = 0.0;
        for (int64_t x = 0; x < e; ++x) c->dv[((k0 + j) * pb->n2 + g) * e + x] = 0.0;
    }
    for (int64_t i = 0; i < lq; ++i) {
        const int64_t t = q0 + i;
        if (gather_rows(pb, c->topk + (t * pb->n2 + g) * pb->block_count, lkv, rows) < 0) {
            c->status = ORA_ERR;
            continue;
        }
        for (int64_t r = 0; r < nsel; ++r) {
            for (int64_t x = 0; x < d; ++x) {
                ksel[r * d + x] = c->k[((k0 + rows[r]) * pb->n2 + g) * d + x];
                dksel[r * d + x] = 0.0;
            }
            for (int64_t x = 0; x < e; ++x) {
                vsel[r * e + x] = c->v[((k0 + rows[r]) * pb->n2 + g) * e + x];
                dvsel[r * e + x] = 0.0;
            }
        }
        for (int64_t hq = g * G; hq < (g + 1) * G; ++hq) {
            const int64_t row = t * pb->n1 + hq;
            const double *qi = c->q + row * d, *oi = c->o + row * e, *doi = c->dout + row * e;
            double *dqi = c->dq + row * d;
            const double mx = c->mx[row], sm = c->sm[row];
            const double Di = dot(doi, oi, e);
            for (int64_t x = 0; x < d; ++x) dqi[x] = 0.0;
            if (mx == -INFINITY || sm == 0.0) continue; /* no visible key */
            for (int64_t r = 0; r < nsel; ++r) {
                if (!nsa_visible(pb, i, rows[r], lq, lkv)) continue;
                const double p = exp(pb->scale * dot(qi, ksel + r * d, d) - mx) / sm;
                const double ds = p * (dot(doi, vsel + r * e, e) - Di);
                for (int64_t x = 0; x < d; ++x) {
                    dqi[x] += pb->scale * ds * ksel[r * d + x];
                    dksel[r * d + x] += pb->scale * ds * qi[x];
                }
                for (int64_t x = 0; x < e; ++x) dvsel[r * e + x] += p * doi[x];
            }
        }
        /* scatter the gathered gradients back through the indices */
        for (int64_t r = 0; r < nsel; ++r) {
            for (int64_t x = 0; x < d; ++x) c->dk[((k0 + rows[r]) * pb->n2 + g) * d + x] += dksel[r * d + x];
            for (int64_t x = 0; x < e; ++x) c->dv[((k0 + rows[r]) * pb->n2 + g) * e + x] += dvsel[r * e + x];
        }
    }
    free(rows); free(ksel); free(vsel); free(dksel); free(dvsel);
}

static int nsa_check(const ora_nsa_t *pb)
{
    if (!pb || pb->n2 <= 0 || pb->n1 % pb->n2 || pb->block_size <= 0 || pb->block_count <= 0) return ORA_ERR;
    if (pb->d <= 0 || pb->d_v < 0) return ORA_ERR;
    if (pb->sparse_mode != 0 && pb->sparse_mode != 2) return ORA_ERR;
    if (pb->atten_mask) {  /* the mask covers every sequence's local positions */
        for (int64_t b = 0; b < pb->nseq; ++b)
            if (seq_len(pb->cu_q, b) > pb->mask_rows || seq_len(pb->cu_kv, b) > pb->mask_cols) return ORA_ERR;
    }
    return ORA_OK;
}

int ora_nsa_fwd(const ora_nsa_t *pb, const double *q, const double *k, const double *v,
                const int32_t *topk, double *o, double *mx, double *sm, int nthreads)
{
    if (nsa_check(pb) || !q || !k || !v || !topk || !o || !mx || !sm) return ORA_ERR;
    nsa_ctx c;
    memset(&c, 0, sizeof c);
    c.pb = pb; c.q = q; c.k = k; c.v = v; c.topk = topk; c.o_out = o; c.mx_out = mx; c.sm_out = sm;
    run_units(nsa_fwd_unit, &c, pb->nseq * pb->n2, nthreads);
    return c.status;
}

int ora_nsa_bwd(const ora_nsa_t *pb, const double *q, const double *k, const double *v,
                const double *o, const double *dout, const double *mx, const double *sm,
                const int32_t *topk, double *dq, double *dk, double *dv, int nthreads)
{
    if (nsa_check(pb) || !q || !k || !v || !o || !dout || !mx || !sm || !topk) return ORA_ERR;
    if (!dq || !dk || !dv) return ORA_ERR;
    nsa_ctx c;
    memset(&c, 0, sizeof c);
    c.pb = pb; c.q = q; c.k = k; c.v = v; c.o = o; c.dout = dout; c.mx = mx; c.sm = sm;
    c.topk = topk; c.dq = dq; c.dk = dk; c.dv = dv;
    run_units(nsa_bwd_unit, &c, pb->nseq * pb->n2, nthreads);
    return c.status;
}

/* Second, independent NSA path: dense attention over the whole sequence
 * with the mask M_tj = [block of j is selected by (t, g)] and the sparse-mode
 * visibility; it computes its own softmax (max, sum), O and the gradients
 * (exact O, so this is the true gradient of the masked-dense attention).
 * Outputs o, dq [Tq][n1][d], dk, dv [Tkv][n2][d].                          */
static void nsa_dense_unit(void *vctx, int64_t unit)
{
    nsa_ctx *c = (nsa_ctx *)vctx;
    const ora_nsa_t *pb = c->pb;
    const int64_t b = unit / pb->n2, g = unit % pb->n2, G = pb->n1 / pb->n2, d = pb->d, e = value_dim(pb);
    const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
    const int64_t k0 = seq_start(pb->cu_kv, b), lkv = seq_len(pb->cu_kv, b);
    char *sel = (char *)malloc((size_t)(lkv > 0 ? lkv : 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1));
    for (int64_t j = 0; j < lkv; ++j) {
        for (int64_t x = 0; x < d; ++x) c->dk[((k0 + j) * pb->n2 + g) * d + x] = 0.0;
        for (int64_t x = 0; x < e; ++x) c->dv[((k0 + j) * pb->n2 + g) * e + x] = 0.0;
    }
    for (int64_t i = 0; i < lq; ++i) {
        const int64_t t = q0 + i;
        memset(sel, 0, (size_t)lkv);
        for (int64_t cc = 0; cc < pb->block_count; ++cc) {
            const int64_t blk = c->topk[(t * pb->n2 + g) * pb->block_count + cc];
            if (blk < 0 || (blk + 1) * pb->block_size > lkv) { c->status = ORA_ERR; continue; }
            if (sel[blk * pb->block_size]) { c->status = ORA_ERR; continue; } /* block already selected */
            for (int64_t r = 0; r < pb->block_size; ++r) sel[blk * pb->block_size + r] = 1;
        }
        for (int64_t j = 0; j < lkv; ++j) sel[j] = sel[j] && nsa_visible(pb, i, j, lq, lkv);
        for (int64_t hq = g * G; hq < (g + 1) * G; ++hq) {
            const int64_t row = t * pb->n1 + hq;
            const double *qi = c->q + row * d, *doi = c->dout + row * e;
            double *oi = c->o_out + row * e, *dqi = c->dq + row * d;
            double mx = -INFINITY, sum = 0.0;
            for (int64_t j = 0; j < lkv; ++j) {
                if (!sel[j]) continue;
                p[j] = pb->scale * dot(qi, c->k + ((k0 + j) * pb->n2 + g) * d, d);
                if (p[j] > mx) mx = p[j];
            }
            for (int64_t x = 0; x < e; ++x) oi[x] = 0.0;
            for (int64_t x = 0; x < d; ++x) dqi[x] = 0.0;
            if (mx == -INFINITY) continue;
            for (int64_t j = 0; j < lkv; ++j)
                if (sel[j]) sum += exp(p[j] - mx);
            for (int64_t j = 0; j < lkv; ++j) {
                if (!sel[j]) continue;
                p[j] = exp(p[j] - mx) / sum;
                const double *vj = c->v + ((k0 + j) * pb->n2 + g) * e;
                for (int64_t x = 0; x < e; ++x) oi[x] += p[j] * vj[x];
            }
            const double Di = dot(doi, oi, e);
            for (int64_t j = 0; j < lkv; ++j) {
                if (!sel[j]) continue;
                const double *kj = c->k + ((k0 + j) * pb->n2 + g) * d;
                const double *vj = c->v + ((k0 + j) * pb->n2 + g) * e;
                double *dkj = c->dk + ((k0 + j) * pb->n2 + g) * d;
                double *dvj = c->dv + ((k0 + j) * pb->n2 + g) * e;
                const double ds = p[j] * (dot(doi, vj, e) - Di);
                for (int64_t x = 0; x < d; ++x) {
                    dqi[x] += pb->scale * ds * kj[x];
                    dkj[x] += pb->scale * ds * qi[x];
                }
                for (int64_t x = 0; x < e; ++x) dvj[x] += p[j] * doi[x];
            }
        }
    }
    free(sel); free(p);
}

int ora_nsa_masked_dense(const ora_nsa_t *pb, const double *q, const double *k, const double *v,
                         const double *dout, const int32_t *topk,
                         double *o, double *dq, double *dk, double *dv, int nthreads)
{
    if (nsa_check(pb) || !q || !k || !v || !dout || !topk || !o || !dq || !dk || !dv) return ORA_ERR;
    nsa_ctx c;
    memset(&c, 0, sizeof c);
    c.pb = pb; c.q = q; c.k = k; c.v = v; c.dout = dout; c.topk = topk;
    c.o_out = o; c.dq = dq; c.dk = dk; c.dv = dv;
    run_units(nsa_dense_unit, &c, pb->nseq * pb->n2, nthreads);
    return c.status;
}

/* Tokens that selected each block, per (sequence, kv head, block): the
 * ascending list of local token positions t with k in topk[t, g, :], leaving
 * out pairs whose every key is masked by the sparse mode.  Output is a CSR:
 * offsets[(b * n2 + g) * nblk_max + k] .. +1 index into tokens (global token
 * ids), where nblk_max = max over sequences of lkv / block_size.  This is the
 * definition written as a brute-force double loop.                          */
int ora_nsa_block_lists(const ora_nsa_t *pb, const int32_t *topk, int64_t nblk_max,
                        int64_t *offsets, int32_t *tokens)
{
    if (nsa_check(pb) || !topk || !offsets || !tokens) return ORA_ERR;
    int64_t n = 0;
    offsets[0] = 0;
    for (int64_t b = 0; b < pb->nseq; ++b) {
        const int64_t q0 = seq_start(pb->cu_q, b), lq = seq_len(pb->cu_q, b);
        const int64_t lkv = seq_len(pb->cu_kv, b);
        for (int64_t g = 0; g < pb->n2; ++g)
            for (int64_t blk = 0; blk < nblk_max; ++blk) {
                for (int64_t i = 0; i < lq; ++i) {
                    int chosen = 0;
                    for (int64_t cc = 0; cc < pb->block_count; ++cc)
                        if (topk[((q0 + i) * pb->n2 + g) * pb->block_count + cc] == blk) chosen = 1;
                    /* the block's first key is its most visible one (the sparse mode
                       alone decides; attenMaskOptional applies per element later) */
                    if (chosen && nsa_mode_visible(pb, i, blk * pb->block_size, lq, lkv))
                        tokens[n++] = (int32_t)(q0 + i);
                }
                offsets[(b * pb->n2 + g) * nblk_max + blk + 1] = n;
            }
    }
    return ORA_OK;
}
