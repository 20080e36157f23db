/*
 * attn_oracle.c -- plain, slow, FP64 CPU reference for causal scaled-dot-product
 * attention (forward, backward, LSE merge) and for the "naive reduced-precision"
 * implementation whose error sets the accuracy floor.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file.  It shares no code, header,
 * table or helper with the CUDA library and includes no GPU header.
 *
 * Sources followed (TransformerEngine PR #3527, "cuDNN FROST attention backend
 * for head_dim in (256, 512]"):
 *   - the forward saves a natural-log log-sum-exp in FP32 (description, "the
 *     forward LSE is natural-log logsumexp in fp32");
 *   - the reference must be float64, not float32 (review notes on TF32);
 *   - the accuracy criterion err(kernel, fp64) <= 2 * err(naive_bf16, fp64);
 *   - the sliding-window keep rule: the window applies to any mask type, -1 is
 *     unbounded on that side, a causal mask pins the right bound to the
 *     diagonal; the left bound counts visible tokens including the diagonal;
 *   - causal top-left and bottom-right alignment coincide when Sq == Skv;
 *   - a context-parallel ring merges partial results by exponentiating LSE
 *     differences.
 * TransformerEngine PR #3699 ("cuDNN FROST D128/D256 backward dispatch"):
 *   - rows with no visible key produce exactly zero dQ.
 *
 * Layout (all arrays contiguous, row-major):
 *   q  [Tq][hq][dqk]   k [Tk][hkv][dqk]   v [Tk][hkv][dv]   dout/o [Tq][hq][dv]
 *   lse [hq][Tq]       sequences are [cu_q[b], cu_q[b+1]) and [cu_k[b], cu_k[b+1])
 * A dense [B][S][H][d] tensor is the same memory with cu = {0, S, 2S, ...}.
 *
 * Query head h reads key/value head h / (hq / hkv) (contiguous GQA groups).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int nseq;
    const int32_t *cu_q, *cu_k;
    int hq, hkv, dqk, dv;
    int causal, bottom_right, wl, wr;
    double scale;
} ocfg_t;

/* Key j is visible from query i of a sequence with Lq queries and Lk keys. */
static int visible(const ocfg_t *c, long i, long j, long Lq, long Lk)
{
    long off = c->bottom_right ? (Lk - Lq) : 0;
    if (c->causal && j > i + off) return 0;
    if (c->wl >= 0 && j < i + off - c->wl) return 0;
    if (c->wr >= 0 && j > i + off + c->wr) return 0;
    return 1;
}

/* ------------------------------------------------------------------------ */
/* thread pool: run fn(item, ctx) for item in [0, n)                         */
typedef struct {
    void (*fn)(long, void *);
    void *ctx;
    long n;
    long next;
    pthread_mutex_t mu;
} pool_t;

static void *pool_worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        long it = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (it >= p->n) break;
        p->fn(it, p->ctx);
    }
    return NULL;
}

static void run_pool(long n, int nthreads, void (*fn)(long, void *), void *ctx)
{
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.n = n; p.next = 0;
    pthread_mutex_init(&p.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[started], NULL, pool_worker, &p) == 0) ++started;
    pool_worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------------ */
/* Exact forward: for each query row, scores over visible keys, softmax with  */
/* its maximum subtracted, LSE = m + ln(sum), O = sum_j P_ij v_j.             */
/* A row with no visible key gets O = 0 and LSE = -inf.                        */

typedef struct {
    const ocfg_t *c;
    const double *q, *k, *v;
    double *o, *lse;
    const uint8_t *head_sel; /* [hq] or NULL */
} fwd_ctx_t;

static void fwd_row(const ocfg_t *c, const double *q, const double *k, const double *v,
                    long b, int h, long i, double *s /* scratch [Lk] */,
                    double *o_row, double *lse_out)
{
    long q0 = c->cu_q[b], k0 = c->cu_k[b];
    long Lq = c->cu_q[b + 1] - q0, Lk = c->cu_k[b + 1] - k0;
    int g = h / (c->hq / c->hkv);
    const double *qi = q + ((q0 + i) * c->hq + h) * (long)c->dqk;
    double m = -INFINITY;
    for (long j = 0; j < Lk; ++j) {
        if (!visible(c, i, j, Lq, Lk)) { s[j] = -INFINITY; continue; }
        const double *kj = k + ((k0 + j) * c->hkv + g) * (long)c->dqk;
        double acc = 0.0;
        for (int t = 0; t < c->dqk; ++t) acc += qi[t] * kj[t];
        s[j] = c->scale * acc;
        if (s[j] > m) m = s[j];
    }
    for (int t = 0; t < c->dv; ++t) o_row[t] = 0.0;
    if (m == -INFINITY) { *lse_out = -INFINITY; return; }
    double l = 0.0;
    for (long j = 0; j < Lk; ++j)
        if (s[j] != -INFINITY) l += exp(s[j] - m);
    double lse = m + log(l);
    *lse_out = lse;
    for (long j = 0; j < Lk; ++j) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - lse);
        const double *vj = v + ((k0 + j) * c->hkv + g) * (long)c->dv;
        for (int t = 0; t < c->dv; ++t) o_row[t] += p * vj[t];
    }
}

static long max_len(const int32_t *cu, int n)
{
    long m = 0;
    for (int b = 0; b < n; ++b) if (cu[b + 1] - cu[b] > m) m = cu[b + 1] - cu[b];
    return m;
}

static void fwd_item(long item, void *vctx)
{
    fwd_ctx_t *x = (fwd_ctx_t *)vctx;
    const ocfg_t *c = x->c;
    long b = item / c->hq;
    int h = (int)(item % c->hq);
    if (x->head_sel && !x->head_sel[h]) return;
    long q0 = c->cu_q[b], Lq = c->cu_q[b + 1] - q0;
    long Lk = c->cu_k[b + 1] - c->cu_k[b];
    long Tq = c->cu_q[c->nseq];
    double *s = (double *)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
    for (long i = 0; i < Lq; ++i) {
        double *o_row = x->o + ((q0 + i) * c->hq + h) * (long)c->dv;
        fwd_row(c, x->q, x->k, x->v, b, h, i, s, o_row, &x->lse[(long)h * Tq + q0 + i]);
    }
    free(s);
}

static int check_cfg(const ocfg_t *c)
{
    if (c->nseq < 0 || c->hq <= 0 || c->hkv <= 0 || c->hq % c->hkv) return -1;
    if (c->dqk <= 0 || c->dv <= 0) return -1;
    if (c->cu_q[0] != 0 || c->cu_k[0] != 0) return -2;
    for (int b = 0; b < c->nseq; ++b)
        if (c->cu_q[b + 1] < c->cu_q[b] || c->cu_k[b + 1] < c->cu_k[b]) return -2;
    return 0;
}

int oracle_fwd(int nseq, const int32_t *cu_q, const int32_t *cu_k, int hq, int hkv,
               int dqk, int dv, const double *q, const double *k, const double *v,
               int causal, int bottom_right, int wl, int wr, double scale,
               double *o, double *lse, const uint8_t *head_sel, int nthreads)
{
    ocfg_t c = {nseq, cu_q, cu_k, hq, hkv, dqk, dv, causal, bottom_right, wl, wr, scale};
    int rc = check_cfg(&c);
    if (rc) return rc;
    fwd_ctx_t x = {&c, q, k, v, o, lse, head_sel};
    run_pool((long)nseq * hq, nthreads, fwd_item, &x);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Exact backward (gradient of O with respect to Q, K, V for upstream dO).   */
/*   D_i = sum_c dO_ic O_ic,  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i) */
/*   dQ_i = scale sum_j dS_ij k_j                                             */
/*   dK_j = scale sum_{i, h in group} dS_ij q_i                               */
/*   dV_j = sum_{i, h in group} P_ij dO_i                                     */
/* O and LSE are this file's own FP64 forward results.  One work item is one  */
/* (sequence, key/value head): it owns dK/dV of that head and dQ of the query */
/* heads in its group, so no two items write the same element.               */

typedef struct {
    const ocfg_t *c;
    const double *q, *k, *v, *dout;
    double *dq, *dk, *dv;
    const uint8_t *group_sel; /* [hkv] or NULL */
} bwd_ctx_t;

static void bwd_item(long item, void *vctx)
{
    bwd_ctx_t *x = (bwd_ctx_t *)vctx;
    const ocfg_t *c = x->c;
    long b = item / c->hkv;
    int g = (int)(item % c->hkv);
    if (x->group_sel && !x->group_sel[g]) return;
    int grp = c->hq / c->hkv;
    long q0 = c->cu_q[b], k0 = c->cu_k[b];
    long Lq = c->cu_q[b + 1] - q0, Lk = c->cu_k[b + 1] - k0;
    double *s = (double *)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
    double *orow = (double *)malloc(sizeof(double) * c->dv);
    for (long j = 0; j < Lk; ++j) {
        memset(x->dk + ((k0 + j) * c->hkv + g) * (long)c->dqk, 0, sizeof(double) * c->dqk);
        memset(x->dv + ((k0 + j) * c->hkv + g) * (long)c->dv, 0, sizeof(double) * c->dv);
    }
    for (int hh = 0; hh < grp; ++hh) {
        int h = g * grp + hh;
        for (long i = 0; i < Lq; ++i) {
            double lse;
            fwd_row(c, x->q, x->k, x->v, b, h, i, s, orow, &lse);
            const double *qi = x->q + ((q0 + i) * c->hq + h) * (long)c->dqk;
            const double *doi = x->dout + ((q0 + i) * c->hq + h) * (long)c->dv;
            double *dqi = x->dq + ((q0 + i) * c->hq + h) * (long)c->dqk;
            for (int t = 0; t < c->dqk; ++t) dqi[t] = 0.0;
            if (lse == -INFINITY) continue; /* keyless row: contributes nothing */
            double D = 0.0;
            for (int t = 0; t < c->dv; ++t) D += doi[t] * orow[t];
            for (long j = 0; j < Lk; ++j) {
                if (s[j] == -INFINITY) continue;
                double p = exp(s[j] - lse);
                const double *kj = x->k + ((k0 + j) * c->hkv + g) * (long)c->dqk;
                const double *vj = x->v + ((k0 + j) * c->hkv + g) * (long)c->dv;
                double *dkj = x->dk + ((k0 + j) * c->hkv + g) * (long)c->dqk;
                double *dvj = x->dv + ((k0 + j) * c->hkv + g) * (long)c->dv;
                double dp = 0.0;
                for (int t = 0; t < c->dv; ++t) dp += doi[t] * vj[t];
                double ds = p * (dp - D);
                for (int t = 0; t < c->dqk; ++t) {
                    dqi[t] += c->scale * ds * kj[t];
                    dkj[t] += c->scale * ds * qi[t];
                }
                for (int t = 0; t < c->dv; ++t) dvj[t] += p * doi[t];
            }
        }
    }
    free(orow);
    free(s);
}

int oracle_bwd(int nseq, const int32_t *cu_q, const int32_t *cu_k, int hq, int hkv,
               int dqk, int dv, const double *q, const double *k, const double *v,
               const double *dout, int causal, int bottom_right, int wl, int wr,
               double scale, double *dq, double *dk, double *dv_out,
               const uint8_t *group_sel, int nthreads)
{
    ocfg_t c = {nseq, cu_q, cu_k, hq, hkv, dqk, dv, causal, bottom_right, wl, wr, scale};
    int rc = check_cfg(&c);
    if (rc) return rc;
    bwd_ctx_t x = {&c, q, k, v, dout, dq, dk, dv_out, group_sel};
    run_pool((long)nseq * hkv, nthreads, bwd_item, &x);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* LSE-weighted merge of n partial results over disjoint key sets:           */
/*   LSE = ln sum_p exp(LSE_p)  (maximum subtracted first)                     */
/*   O   = sum_p exp(LSE_p - LSE) O_p                                          */
/* A part with LSE_p = -inf has weight 0; if every part is -inf, O = 0 and     */
/* LSE = -inf.                                                                 */
/* o_parts [n][rows][heads][dv], lse_parts [n][heads][rows]                    */
int oracle_lse_merge(int n, long rows, int heads, int dv, const double *o_parts,
                     const double *lse_parts, double *o_out, double *lse_out)
{
    if (n <= 0 || rows < 0 || heads <= 0 || dv <= 0) return -1;
    for (long r = 0; r < rows; ++r) {
        for (int h = 0; h < heads; ++h) {
            double m = -INFINITY;
            for (int p = 0; p < n; ++p) {
                double l = lse_parts[((long)p * heads + h) * rows + r];
                if (l > m) m = l;
            }
            double *orow = o_out + (r * heads + h) * (long)dv;
            for (int t = 0; t < dv; ++t) orow[t] = 0.0;
            if (m == -INFINITY) { lse_out[(long)h * rows + r] = -INFINITY; continue; }
            double w = 0.0;
            for (int p = 0; p < n; ++p) {
                double l = lse_parts[((long)p * heads + h) * rows + r];
                if (l != -INFINITY) w += exp(l - m);
            }
            double lse = m + log(w);
            lse_out[(long)h * rows + r] = lse;
            for (int p = 0; p < n; ++p) {
                double l = lse_parts[((long)p * heads + h) * rows + r];
                if (l == -INFINITY) continue;
                double a = exp(l - lse);
                const double *op = o_parts + (((long)p * rows + r) * heads + h) * (long)dv;
                for (int t = 0; t < dv; ++t) orow[t] += a * op[t];
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Naive reduced-precision implementation (the accuracy floor).  It follows   */
/* an unfused framework implementation: every tensor operation accumulates in */
/* FP32 and rounds its result to the storage type T (round to nearest even):  */
/*   S = rnd(Q K^T); S' = rnd(scale S); P = rnd(softmax_fp32(S')); O = rnd(P V)*/
/*   dP = rnd(dO V^T); D = rnd(rowsum(dO o O)); dS = rnd(P o (dP - D))         */
/*   dQ = rnd(scale rnd(dS K)); dK_h = rnd(scale rnd(dS^T Q)); dV_h = rnd(P^T dO)*/
/* and with GQA the per-query-head dK_h / dV_h are summed in FP32 and rounded */
/* (the gradient of a repeated key/value tensor).                              */
/* dtype: 0 = bfloat16, 1 = float16, 2 = no rounding (float32 throughout).     */

static float rnd_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) {         /* inf / nan: truncate */
        if (u & 0x007fffffu) u |= 0x00400000u;       /* keep nan quiet */
        u &= 0xffff0000u;
    } else {
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7fffu + lsb;                          /* round to nearest even */
        u &= 0xffff0000u;
    }
    memcpy(&f, &u, 4);
    return f;
}

static float rnd_t(float f, int dtype)
{
    if (dtype == 0) return rnd_bf16(f);
    if (dtype == 1) return (float)(_Float16)f;       /* C conversion: nearest even */
    return f;
}

typedef struct {
    const ocfg_t *c;
    int dtype;
    const float *q, *k, *v, *dout; /* T-representable values held as float */
    float *o, *lse;                 /* naive forward results (o rounded to T) */
    float *dq;                      /* [Tq][hq][dqk] */
    float *dk_h, *dv_h;             /* per-query-head partials [Tk][hq][d] */
    int do_bwd;
} naive_ctx_t;

/* Forward of one query row of the naive implementation: rounded scores, an
 * FP32 softmax rounded to T (p[j] = 0 for masked keys), O = rnd(P V).  Writes
 * p[0..Lk), o_row[0..dv) and *lse_out (-inf for a row with no visible key). */
static void naive_fwd_row(const ocfg_t *c, int dt, const float *q, const float *k,
                          const float *v, long b, int h, long i, float *p, float *acc,
                          float *o_row, float *lse_out)
{
    int g = h / (c->hq / c->hkv);
    long q0 = c->cu_q[b], k0 = c->cu_k[b];
    long Lq = c->cu_q[b + 1] - q0, Lk = c->cu_k[b + 1] - k0;
    const float *qi = q + ((q0 + i) * c->hq + h) * (long)c->dqk;
    float m = -INFINITY;
    for (long j = 0; j < Lk; ++j) {
        if (!visible(c, i, j, Lq, Lk)) { p[j] = -INFINITY; continue; }
        const float *kj = k + ((k0 + j) * c->hkv + g) * (long)c->dqk;
        float a = 0.0f;
        for (int t = 0; t < c->dqk; ++t) a += qi[t] * kj[t];
        float sv = rnd_t(rnd_t(a, dt) * (float)c->scale, dt);
        p[j] = sv;
        if (sv > m) m = sv;
    }
    for (int t = 0; t < c->dv; ++t) o_row[t] = 0.0f;
    if (m == -INFINITY) {
        *lse_out = -INFINITY;
        for (long j = 0; j < Lk; ++j) p[j] = 0.0f;
        return;
    }
    float l = 0.0f;
    for (long j = 0; j < Lk; ++j) {
        float e = (p[j] == -INFINITY) ? 0.0f : expf(p[j] - m);
        p[j] = e;
        l += e;
    }
    *lse_out = m + logf(l);
    for (long j = 0; j < Lk; ++j) p[j] = rnd_t(p[j] / l, dt);
    for (int t = 0; t < c->dv; ++t) acc[t] = 0.0f;
    for (long j = 0; j < Lk; ++j) {
        if (p[j] == 0.0f) continue;
        const float *vj = v + ((k0 + j) * c->hkv + g) * (long)c->dv;
        for (int t = 0; t < c->dv; ++t) acc[t] += p[j] * vj[t];
    }
    for (int t = 0; t < c->dv; ++t) o_row[t] = rnd_t(acc[t], dt);
}

static void naive_item(long item, void *vctx)
{
    naive_ctx_t *x = (naive_ctx_t *)vctx;
    const ocfg_t *c = x->c;
    int dt = x->dtype;
    long b = item / c->hq;
    int h = (int)(item % c->hq);
    int g = h / (c->hq / c->hkv);
    long q0 = c->cu_q[b], k0 = c->cu_k[b];
    long Lq = c->cu_q[b + 1] - q0, Lk = c->cu_k[b + 1] - k0;
    long Tq = c->cu_q[c->nseq];
    float *p = (float *)malloc(sizeof(float) * (Lk > 0 ? Lk : 1));
    float *ds = (float *)malloc(sizeof(float) * (Lk > 0 ? Lk : 1));
    float *acc = (float *)malloc(sizeof(float) * (c->dqk > c->dv ? c->dqk : c->dv));
    for (long i = 0; i < Lq; ++i) {
        const float *qi = x->q + ((q0 + i) * c->hq + h) * (long)c->dqk;
        float *oi = x->o + ((q0 + i) * c->hq + h) * (long)c->dv;
        naive_fwd_row(c, dt, x->q, x->k, x->v, b, h, i, p, acc, oi,
                      &x->lse[(long)h * Tq + q0 + i]);
        if (!x->do_bwd) continue;
        const float *doi = x->dout + ((q0 + i) * c->hq + h) * (long)c->dv;
        float D = 0.0f;
        for (int t = 0; t < c->dv; ++t) D += doi[t] * oi[t];
        D = rnd_t(D, dt);
        for (long j = 0; j < Lk; ++j) {
            if (p[j] == 0.0f) { ds[j] = 0.0f; continue; }
            const float *vj = x->v + ((k0 + j) * c->hkv + g) * (long)c->dv;
            float a = 0.0f;
            for (int t = 0; t < c->dv; ++t) a += doi[t] * vj[t];
            float dpv = rnd_t(a, dt);
            ds[j] = rnd_t(p[j] * (dpv - D), dt);
        }
        float *dqi = x->dq + ((q0 + i) * c->hq + h) * (long)c->dqk;
        for (int t = 0; t < c->dqk; ++t) acc[t] = 0.0f;
        for (long j = 0; j < Lk; ++j) {
            if (ds[j] == 0.0f) continue;
            const float *kj = x->k + ((k0 + j) * c->hkv + g) * (long)c->dqk;
            for (int t = 0; t < c->dqk; ++t) acc[t] += ds[j] * kj[t];
        }
        for (int t = 0; t < c->dqk; ++t) dqi[t] = rnd_t(rnd_t(acc[t], dt) * (float)c->scale, dt);
        /* dK_h and dV_h accumulate in FP32 over query rows; rounded at the end */
        for (long j = 0; j < Lk; ++j) {
            float *dkj = x->dk_h + ((k0 + j) * c->hq + h) * (long)c->dqk;
            float *dvj = x->dv_h + ((k0 + j) * c->hq + h) * (long)c->dv;
            if (ds[j] != 0.0f)
                for (int t = 0; t < c->dqk; ++t) dkj[t] += ds[j] * qi[t];
            if (p[j] != 0.0f)
                for (int t = 0; t < c->dv; ++t) dvj[t] += p[j] * doi[t];
        }
    }
    free(acc);
    free(ds);
    free(p);
}

/* Inputs are float arrays whose values are already representable in T.
 * Outputs: o [Tq][hq][dv], lse [hq][Tq]; if dout != NULL also dq, dk, dv. */
int oracle_naive(int nseq, const int32_t *cu_q, const int32_t *cu_k, int hq, int hkv,
                 int dqk, int dv, const float *q, const float *k, const float *v,
                 const float *dout, int causal, int bottom_right, int wl, int wr,
                 double scale, int dtype, float *o, float *lse, float *dq, float *dk,
                 float *dv_out, int nthreads)
{
    ocfg_t c = {nseq, cu_q, cu_k, hq, hkv, dqk, dv, causal, bottom_right, wl, wr, scale};
    int rc = check_cfg(&c);
    if (rc) return rc;
    long Tk = cu_k[nseq];
    float *dk_h = NULL, *dv_h = NULL;
    if (dout) {
        dk_h = (float *)calloc((size_t)(Tk > 0 ? Tk : 1) * hq * dqk, sizeof(float));
        dv_h = (float *)calloc((size_t)(Tk > 0 ? Tk : 1) * hq * dv, sizeof(float));
        if (!dk_h || !dv_h) { free(dk_h); free(dv_h); return -3; }
    }
    naive_ctx_t x = {&c, dtype, q, k, v, dout, o, lse, dq, dk_h, dv_h, dout != NULL};
    run_pool((long)nseq * hq, nthreads, naive_item, &x);
    if (dout) {
        int grp = hq / hkv;
        for (long j = 0; j < Tk; ++j)
            for (int g = 0; g < hkv; ++g) {
                float *dkj = dk + (j * hkv + g) * (long)dqk;
                float *dvj = dv_out + (j * hkv + g) * (long)dv;
                for (int t = 0; t < dqk; ++t) {
                    float s = 0.0f;
                    for (int hh = 0; hh < grp; ++hh) {
                        float r = rnd_t(dk_h[(j * hq + g * grp + hh) * (long)dqk + t], dtype);
                        s += rnd_t(r * (float)scale, dtype);
                    }
                    dkj[t] = rnd_t(s, dtype);
                }
                for (int t = 0; t < dv; ++t) {
                    float s = 0.0f;
                    for (int hh = 0; hh < grp; ++hh)
                        s += rnd_t(dv_h[(j * hq + g * grp + hh) * (long)dv + t], dtype);
                    dvj[t] = rnd_t(s, dtype);
                }
            }
        free(dk_h);
        free(dv_h);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* dK / dV of selected key rows only, exact (FP64) and naive.  The same       */
/* definitions as oracle_bwd and oracle_naive above, evaluated only for the  */
/* keys j of sequence b with key_sel[cu_k[b] + j] != 0; the other rows of    */
/* dk / dv are left as they are.  Every query row that sees a selected key   */
/* still needs its own complete forward (LSE, O and so D), so the cost is    */
/* one forward per such row.  The rows are split into work items of          */
/* (sequence, key/value head, block of query rows); each item sums its rows  */
/* into its own partial and the partials are added in item order at the end, */
/* so the result does not depend on the number of threads.                   */

enum { KV_ROWS = 256 };  /* query rows per work item */

typedef struct {
    const ocfg_t *c;
    int naive, dtype;
    const double *q, *k, *v, *dout;     /* exact: FP64 inputs */
    const float *fq, *fk, *fv, *fdout;  /* naive: T-representable floats */
    const long *sel;      /* selected keys: global key rows, grouped by sequence */
    const long *sel_lo;   /* [nseq + 1]: sequence b's entries are [sel_lo[b], sel_lo[b+1]) */
    long n_sel;
    const long *it_b, *it_i0;
    const int *it_g;
    double *pdk, *pdv;    /* exact partials [item][n_sel][d]          */
    float *fdk, *fdv;     /* naive partials [item][grp][n_sel][d]     */
} kv_ctx_t;

static void kv_item(long item, void *vctx)
{
    kv_ctx_t *x = (kv_ctx_t *)vctx;
    const ocfg_t *c = x->c;
    long b = x->it_b[item], i0 = x->it_i0[item];
    int g = x->it_g[item];
    int grp = c->hq / c->hkv;
    long q0 = c->cu_q[b], k0 = c->cu_k[b];
    long Lq = c->cu_q[b + 1] - q0, Lk = c->cu_k[b + 1] - k0;
    long i1 = i0 + KV_ROWS < Lq ? i0 + KV_ROWS : Lq;
    long s0 = x->sel_lo[b], s1 = x->sel_lo[b + 1];
    long nd = c->dqk > c->dv ? c->dqk : c->dv;
    double *s = (double *)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
    double *orow = (double *)malloc(sizeof(double) * c->dv);
    float *p = (float *)malloc(sizeof(float) * (Lk > 0 ? Lk : 1));
    float *acc = (float *)malloc(sizeof(float) * nd);
    float *fo = (float *)malloc(sizeof(float) * c->dv);
    for (int hh = 0; hh < grp; ++hh) {
        int h = g * grp + hh;
        for (long i = i0; i < i1; ++i) {
            int any = 0;  /* does row i see a selected key? */
            for (long e = s0; e < s1 && !any; ++e)
                any = visible(c, i, x->sel[e] - k0, Lq, Lk);
            if (!any) continue;
            if (!x->naive) {
                double lse;
                fwd_row(c, x->q, x->k, x->v, b, h, i, s, orow, &lse);
                if (lse == -INFINITY) continue;
                const double *qi = x->q + ((q0 + i) * c->hq + h) * (long)c->dqk;
                const double *doi = x->dout + ((q0 + i) * c->hq + h) * (long)c->dv;
                double D = 0.0;
                for (int t = 0; t < c->dv; ++t) D += doi[t] * orow[t];
                for (long e = s0; e < s1; ++e) {
                    long j = x->sel[e] - k0;
                    if (s[j] == -INFINITY) continue;
                    double pj = exp(s[j] - lse);
                    const double *vj = x->v + ((k0 + j) * c->hkv + g) * (long)c->dv;
                    double dp = 0.0;
                    for (int t = 0; t < c->dv; ++t) dp += doi[t] * vj[t];
                    double ds = pj * (dp - D);
                    double *dkj = x->pdk + ((size_t)item * x->n_sel + e) * c->dqk;
                    double *dvj = x->pdv + ((size_t)item * x->n_sel + e) * c->dv;
                    for (int t = 0; t < c->dqk; ++t) dkj[t] += c->scale * ds * qi[t];
                    for (int t = 0; t < c->dv; ++t) dvj[t] += pj * doi[t];
                }
            } else {
                int dt = x->dtype;
                float lse;
                naive_fwd_row(c, dt, x->fq, x->fk, x->fv, b, h, i, p, acc, fo, &lse);
                const float *qi = x->fq + ((q0 + i) * c->hq + h) * (long)c->dqk;
                const float *doi = x->fdout + ((q0 + i) * c->hq + h) * (long)c->dv;
                float D = 0.0f;
                for (int t = 0; t < c->dv; ++t) D += doi[t] * fo[t];
                D = rnd_t(D, dt);
                for (long e = s0; e < s1; ++e) {
                    long j = x->sel[e] - k0;
                    if (p[j] == 0.0f) continue;
                    const float *vj = x->fv + ((k0 + j) * c->hkv + g) * (long)c->dv;
                    float a = 0.0f;
                    for (int t = 0; t < c->dv; ++t) a += doi[t] * vj[t];
                    float dpv = rnd_t(a, dt);
                    float ds = rnd_t(p[j] * (dpv - D), dt);
                    float *dkj = x->fdk + (((size_t)item * grp + hh) * x->n_sel + e) * c->dqk;
                    float *dvj = x->fdv + (((size_t)item * grp + hh) * x->n_sel + e) * c->dv;
                    if (ds != 0.0f)
                        for (int t = 0; t < c->dqk; ++t) dkj[t] += ds * qi[t];
                    for (int t = 0; t < c->dv; ++t) dvj[t] += p[j] * doi[t];
                }
            }
        }
    }
    free(fo);
    free(acc);
    free(p);
    free(orow);
    free(s);
}

static int kv_run(const ocfg_t *c, int naive, int dtype, const void *q, const void *k,
                  const void *v, const void *dout, const uint8_t *key_sel,
                  const uint8_t *group_sel, void *dk, void *dv_out, int nthreads)
{
    int rc = check_cfg(c);
    if (rc) return rc;
    long Tk = c->cu_k[c->nseq];
    int grp = c->hq / c->hkv;
    long *sel_lo = (long *)calloc((size_t)c->nseq + 1, sizeof(long));
    long n_sel = 0;
    for (long j = 0; j < Tk; ++j) n_sel += key_sel[j] != 0;
    long *sel = (long *)malloc(sizeof(long) * (n_sel > 0 ? n_sel : 1));
    long n_items = 0, e = 0;
    for (int b = 0; b < c->nseq; ++b) {
        sel_lo[b] = e;
        for (long j = c->cu_k[b]; j < c->cu_k[b + 1]; ++j)
            if (key_sel[j]) sel[e++] = j;
        long Lq = c->cu_q[b + 1] - c->cu_q[b];
        for (int g = 0; g < c->hkv; ++g)
            if (!group_sel || group_sel[g]) n_items += (Lq + KV_ROWS - 1) / KV_ROWS;
    }
    sel_lo[c->nseq] = e;
    long *it_b = (long *)malloc(sizeof(long) * (n_items > 0 ? n_items : 1));
    long *it_i0 = (long *)malloc(sizeof(long) * (n_items > 0 ? n_items : 1));
    int *it_g = (int *)malloc(sizeof(int) * (n_items > 0 ? n_items : 1));
    long it = 0;
    for (int b = 0; b < c->nseq; ++b) {
        long Lq = c->cu_q[b + 1] - c->cu_q[b];
        for (int g = 0; g < c->hkv; ++g) {
            if (group_sel && !group_sel[g]) continue;
            for (long i0 = 0; i0 < Lq; i0 += KV_ROWS) {
                it_b[it] = b;
                it_g[it] = g;
                it_i0[it] = i0;
                ++it;
            }
        }
    }
    size_t np = (size_t)(n_items > 0 ? n_items : 1) * (size_t)(n_sel > 0 ? n_sel : 1);
    kv_ctx_t x;
    memset(&x, 0, sizeof(x));
    x.c = c; x.naive = naive; x.dtype = dtype;
    x.sel = sel; x.sel_lo = sel_lo; x.n_sel = n_sel;
    x.it_b = it_b; x.it_i0 = it_i0; x.it_g = it_g;
    if (!naive) {
        x.q = (const double *)q; x.k = (const double *)k; x.v = (const double *)v;
        x.dout = (const double *)dout;
        x.pdk = (double *)calloc(np * c->dqk, sizeof(double));
        x.pdv = (double *)calloc(np * c->dv, sizeof(double));
        if (!x.pdk || !x.pdv) rc = -3;
    } else {
        x.fq = (const float *)q; x.fk = (const float *)k; x.fv = (const float *)v;
        x.fdout = (const float *)dout;
        x.fdk = (float *)calloc(np * grp * c->dqk, sizeof(float));
        x.fdv = (float *)calloc(np * grp * c->dv, sizeof(float));
        if (!x.fdk || !x.fdv) rc = -3;
    }
    if (!rc) run_pool(n_items, nthreads, kv_item, &x);
    /* add the partials of each (selected key, kv head) in item order */
    for (long e2 = 0; e2 < n_sel && !rc; ++e2) {
        long j = sel[e2];
        int b = 0;
        while (c->cu_k[b + 1] <= j) ++b;
        for (int g = 0; g < c->hkv; ++g) {
            if (group_sel && !group_sel[g]) continue;
            if (!naive) {
                double *dkj = (double *)dk + (j * c->hkv + g) * (long)c->dqk;
                double *dvj = (double *)dv_out + (j * c->hkv + g) * (long)c->dv;
                for (int t = 0; t < c->dqk; ++t) dkj[t] = 0.0;
                for (int t = 0; t < c->dv; ++t) dvj[t] = 0.0;
                for (long m = 0; m < n_items; ++m) {
                    if (it_b[m] != b || it_g[m] != g) continue;
                    const double *pk = x.pdk + ((size_t)m * n_sel + e2) * c->dqk;
                    const double *pv = x.pdv + ((size_t)m * n_sel + e2) * c->dv;
                    for (int t = 0; t < c->dqk; ++t) dkj[t] += pk[t];
                    for (int t = 0; t < c->dv; ++t) dvj[t] += pv[t];
                }
            } else {
                /* as oracle_naive: per query head FP32 sums rounded, then summed */
                float *dkj = (float *)dk + (j * c->hkv + g) * (long)c->dqk;
                float *dvj = (float *)dv_out + (j * c->hkv + g) * (long)c->dv;
                for (int t = 0; t < c->dqk; ++t) {
                    float sum = 0.0f;
                    for (int hh = 0; hh < grp; ++hh) {
                        float a = 0.0f;
                        for (long m = 0; m < n_items; ++m)
                            if (it_b[m] == b && it_g[m] == g)
                                a += x.fdk[(((size_t)m * grp + hh) * n_sel + e2) * c->dqk + t];
                        sum += rnd_t(rnd_t(a, dtype) * (float)c->scale, dtype);
                    }
                    dkj[t] = rnd_t(sum, dtype);
                }
                for (int t = 0; t < c->dv; ++t) {
                    float sum = 0.0f;
                    for (int hh = 0; hh < grp; ++hh) {
                        float a = 0.0f;
                        for (long m = 0; m < n_items; ++m)
                            if (it_b[m] == b && it_g[m] == g)
                                a += x.fdv[(((size_t)m * grp + hh) * n_sel + e2) * c->dv + t];
                        sum += rnd_t(a, dtype);
                    }
                    dvj[t] = rnd_t(sum, dtype);
                }
            }
        }
    }
    free(x.pdk); free(x.pdv); free(x.fdk); free(x.fdv);
    free(it_g); free(it_i0); free(it_b); free(sel); free(sel_lo);
    return rc;
}

/* Exact dK / dV (FP64) of the selected key rows; dk [Tk][hkv][dqk],
 * dv [Tk][hkv][dv], only the selected rows (and selected groups) written. */
int oracle_bwd_kv(int nseq, const int32_t *cu_q, const int32_t *cu_k, int hq, int hkv,
                  int dqk, int dv, const double *q, const double *k, const double *v,
                  const double *dout, int causal, int bottom_right, int wl, int wr,
                  double scale, const uint8_t *key_sel, const uint8_t *group_sel,
                  double *dk, double *dv_out, int nthreads)
{
    ocfg_t c = {nseq, cu_q, cu_k, hq, hkv, dqk, dv, causal, bottom_right, wl, wr, scale};
    return kv_run(&c, 0, 0, q, k, v, dout, key_sel, group_sel, dk, dv_out, nthreads);
}

/* The naive implementation's dK / dV of the selected key rows (FP32). */
int oracle_naive_kv(int nseq, const int32_t *cu_q, const int32_t *cu_k, int hq, int hkv,
                    int dqk, int dv, const float *q, const float *k, const float *v,
                    const float *dout, int causal, int bottom_right, int wl, int wr,
                    double scale, int dtype, const uint8_t *key_sel, const uint8_t *group_sel,
                    float *dk, float *dv_out, int nthreads)
{
    ocfg_t c = {nseq, cu_q, cu_k, hq, hkv, dqk, dv, causal, bottom_right, wl, wr, scale};
    return kv_run(&c, 1, dtype, q, k, v, dout, key_sel, group_sel, dk, dv_out, nthreads);
}

/* Round float values to T in place (used to make T-representable inputs). */
void oracle_round(float *x, long n, int dtype)
{
    for (long i = 0; i < n; ++i) x[i] = rnd_t(x[i], dtype);
}
