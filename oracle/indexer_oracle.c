/*
 * Plain fp64 CPU oracle for the lightning-indexer backward.
 *
 * TEST INFRASTRUCTURE ONLY (like selattn_oracle.c): the slow, obviously
 * correct statement of what the GPU library must compute; shares no code,
 * header, table or constant with the CUDA path.
 *
 * Source: "aclnnLightningIndexerGrad" page, formula section:
 *     S  = Relu(Matmul(Query, Gather(Key, Indices)))
 *     Y  = Dy * Weights
 *     dW = Reduce(S * dy)
 *     dQ = Matmul(ReluGrad(Y, S), Gather(Key, Indices))
 *     dK = ScatterAdd(Matmul(ReluGrad(Y, S), Q), Indices)
 * Readings (the page's parameter tables are lost):
 *   - query [T1, n1, d], key [T2, n2, d] with query head h using key head
 *     h / G (G = n1 / n2), weights [T1, n1], indices and dy [T1, n2, topk]:
 *     per (token, key head) the topk selected key positions, local to the
 *     token's batch, and the gradient of the index score at each of them;
 *   - S[t,h,j] = relu(<q[t,h], k[idx[t,j]]>) with no scale (none in the
 *     formula); Y[t,h,j] = dy[t,j] * w[t,h] (Dy broadcast over the heads);
 *     ReluGrad(Y, S) = Y where S > 0, else 0; Reduce sums over the selected
 *     positions j;
 *   - ScatterAdd adds the row of every selection into dK at its key row, so a
 *     position selected twice counts twice;
 *   - an index of -1 marks an empty slot (no contribution); any other id
 *     outside [0, S2_b) is an error;
 *   - layouts as in selattn_oracle.c: TND (batch b's rows cu[b]..cu[b+1]-1)
 *     or BSND (batch b padded to s1_max / s2_max rows from b * s_max).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { LIO_F64 = 0, LIO_BF16 = 1, LIO_F16 = 2, LIO_F32 = 3 };
enum { LIO_OK = 0, LIO_EARG = -1, LIO_EINDEX = -2 };

typedef struct {
    const void *data;
    int32_t dtype;
    int32_t pad_;
} lio_tensor;

typedef struct {
    int32_t batch, n1, n2, d, topk;
    int32_t layout, s1_max, s2_max;    /* layout 0: TND, 1: BSND */
    const int32_t *cu_q, *cu_kv;       /* B+1 prefix sums of the (valid) lengths */
    const int32_t *idx;                /* [T1, n2, topk] */
    lio_tensor q, k, w, dy;            /* [T1,n1,d], [T2,n2,d], [T1,n1], [T1,n2,topk] */
} lio_problem;

static double dec16(uint16_t h, int bf)
{
    if (bf) {
        union { uint32_t u; float f; } c;
        c.u = (uint32_t)h << 16;
        return (double)c.f;          /* every bf16 value is a float: exact */
    }
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);
    return s ? -v : v;
}

static double ldv(const lio_tensor *t, int64_t i)
{
    switch (t->dtype) {
    case LIO_F64: return ((const double *)t->data)[i];
    case LIO_BF16: return dec16(((const uint16_t *)t->data)[i], 1);
    case LIO_F16: return dec16(((const uint16_t *)t->data)[i], 0);
    default: return (double)((const float *)t->data)[i];
    }
}

static int64_t q0(const lio_problem *p, int b) { return p->layout ? (int64_t)b * p->s1_max : p->cu_q[b]; }
static int64_t k0(const lio_problem *p, int b) { return p->layout ? (int64_t)b * p->s2_max : p->cu_kv[b]; }
static int64_t rows_q(const lio_problem *p) { return p->layout ? (int64_t)p->batch * p->s1_max : p->cu_q[p->batch]; }
static int64_t rows_k(const lio_problem *p) { return p->layout ? (int64_t)p->batch * p->s2_max : p->cu_kv[p->batch]; }

static int check(const lio_problem *p)
{
    if (!p || p->batch < 1 || p->n1 < 1 || p->n2 < 1 || p->n1 % p->n2 || p->d < 1 || p->topk < 1) return LIO_EARG;
    if (!p->cu_q || !p->cu_kv || !p->idx || p->cu_q[0] || p->cu_kv[0]) return LIO_EARG;
    if (p->layout != 0 && p->layout != 1) return LIO_EARG;
    for (int b = 0; b < p->batch; ++b) {
        if (p->cu_q[b + 1] < p->cu_q[b] || p->cu_kv[b + 1] < p->cu_kv[b]) return LIO_EARG;
        if (p->layout && (p->cu_q[b + 1] - p->cu_q[b] > p->s1_max || p->cu_kv[b + 1] - p->cu_kv[b] > p->s2_max))
            return LIO_EARG;
    }
    return LIO_OK;
}

/*
 * The backward restricted to the query rows t in [t_lo, t_hi): their dq and
 * dw rows and their contributions to dk.  dq [T1, n1, d], dk [T2, n2, d],
 * dw [T1, n1] are overwritten (rows outside the range, padding rows and key
 * rows no query in the range selected stay zero).
 */
int lio_backward_range(const lio_problem *p, int64_t t_lo, int64_t t_hi, double *dq, double *dk, double *dw)
{
    int rc = check(p);
    if (rc) return rc;
    const int G = p->n1 / p->n2, d = p->d;
    memset(dq, 0, sizeof(double) * rows_q(p) * p->n1 * d);
    memset(dk, 0, sizeof(double) * rows_k(p) * p->n2 * d);
    memset(dw, 0, sizeof(double) * rows_q(p) * p->n1);
    for (int b = 0; b < p->batch; ++b) {
        const int64_t s2 = p->cu_kv[b + 1] - p->cu_kv[b];
        for (int64_t t = q0(p, b); t < q0(p, b) + (p->cu_q[b + 1] - p->cu_q[b]); ++t) {
            if (t < t_lo || t >= t_hi) continue;
            for (int n2 = 0; n2 < p->n2; ++n2)
                for (int j = 0; j < p->topk; ++j) {
                    const int64_t sel = ((int64_t)t * p->n2 + n2) * p->topk + j;
                    const int64_t id = p->idx[sel];
                    if (id == -1) continue;                       /* empty slot */
                    if (id < 0 || id >= s2) return LIO_EINDEX;
                    const int64_t krow = (k0(p, b) + id) * p->n2 + n2;   /* row of Gather(Key, Indices) */
                    const double dyv = ldv(&p->dy, sel);
                    for (int g = 0; g < G; ++g) {
                        const int h = n2 * G + g;
                        const int64_t qrow = (int64_t)t * p->n1 + h;
                        /* S = Relu(Query . Key_sel) */
                        double x = 0.0;
                        for (int e = 0; e < d; ++e) x += ldv(&p->q, qrow * d + e) * ldv(&p->k, krow * d + e);
                        const double s = x > 0.0 ? x : 0.0;
                        /* dW = Reduce(S * dy) */
                        dw[qrow] += s * dyv;
                        /* Y = Dy * Weights; ReluGrad(Y, S) */
                        const double yg = x > 0.0 ? dyv * ldv(&p->w, qrow) : 0.0;
                        if (yg == 0.0) continue;
                        for (int e = 0; e < d; ++e) {
                            dq[qrow * d + e] += yg * ldv(&p->k, krow * d + e);   /* dQ = ReluGrad . Key_sel */
                            dk[krow * d + e] += yg * ldv(&p->q, qrow * d + e);   /* dK = ScatterAdd(ReluGrad^T . Q) */
                        }
                    }
                }
        }
    }
    return LIO_OK;
}

/* The whole backward (every query row). */
int lio_backward(const lio_problem *p, double *dq, double *dk, double *dw)
{
    return lio_backward_range(p, 0, INT64_MAX, dq, dk, dw);
}

/*
 * Index scores of the selected positions (the forward whose gradient the
 * backward is): score[t, n2, j] = sum over the G heads h of key head n2 of
 * w[t,h] * relu(<q[t,h], k[idx[t,n2,j]]>); 0 for empty slots.  Used by the
 * finite-difference pin.
 */
int lio_scores(const lio_problem *p, double *score)
{
    int rc = check(p);
    if (rc) return rc;
    const int G = p->n1 / p->n2, d = p->d;
    memset(score, 0, sizeof(double) * rows_q(p) * p->n2 * p->topk);
    for (int b = 0; b < p->batch; ++b) {
        const int64_t s2 = p->cu_kv[b + 1] - p->cu_kv[b];
        for (int64_t t = q0(p, b); t < q0(p, b) + (p->cu_q[b + 1] - p->cu_q[b]); ++t)
            for (int n2 = 0; n2 < p->n2; ++n2)
                for (int j = 0; j < p->topk; ++j) {
                    const int64_t sel = ((int64_t)t * p->n2 + n2) * p->topk + j;
                    const int64_t id = p->idx[sel];
                    if (id == -1) continue;
                    if (id < 0 || id >= s2) return LIO_EINDEX;
                    const int64_t krow = (k0(p, b) + id) * p->n2 + n2;
                    double acc = 0.0;
                    for (int g = 0; g < G; ++g) {
                        const int64_t qrow = (int64_t)t * p->n1 + n2 * G + g;
                        double x = 0.0;
                        for (int e = 0; e < d; ++e) x += ldv(&p->q, qrow * d + e) * ldv(&p->k, krow * d + e);
                        acc += ldv(&p->w, qrow) * (x > 0.0 ? x : 0.0);
                    }
                    score[sel] = acc;
                }
    }
    return LIO_OK;
}

/* batch of a valid query row, -1 otherwise */
static int batch_of_q(const lio_problem *p, int64_t t)
{
    for (int b = 0; b < p->batch; ++b)
        if (t >= q0(p, b) && t < q0(p, b) + (p->cu_q[b + 1] - p->cu_q[b])) return b;
    return -1;
}

/* dQ [nrows, n1, d] and dW [nrows, n1] of the query rows tokens[0..nrows). */
int lio_q_rows(const lio_problem *p, int64_t nrows, const int64_t *tokens, double *dq, double *dw)
{
    int rc = check(p);
    if (rc) return rc;
    const int G = p->n1 / p->n2, d = p->d;
    memset(dq, 0, sizeof(double) * nrows * p->n1 * d);
    memset(dw, 0, sizeof(double) * nrows * p->n1);
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t t = tokens[i];
        const int b = batch_of_q(p, t);
        if (b < 0) return LIO_EARG;
        const int64_t s2 = p->cu_kv[b + 1] - p->cu_kv[b];
        for (int n2 = 0; n2 < p->n2; ++n2)
            for (int j = 0; j < p->topk; ++j) {
                const int64_t sel = (t * p->n2 + n2) * p->topk + j;
                const int64_t id = p->idx[sel];
                if (id == -1) continue;
                if (id < 0 || id >= s2) return LIO_EINDEX;
                const int64_t krow = (k0(p, b) + id) * p->n2 + n2;
                const double dyv = ldv(&p->dy, sel);
                for (int g = 0; g < G; ++g) {
                    const int h = n2 * G + g;
                    const int64_t qrow = t * p->n1 + h;
                    double x = 0.0;
                    for (int e = 0; e < d; ++e) x += ldv(&p->q, qrow * d + e) * ldv(&p->k, krow * d + e);
                    dw[i * p->n1 + h] += (x > 0.0 ? x : 0.0) * dyv;
                    const double yg = x > 0.0 ? dyv * ldv(&p->w, qrow) : 0.0;
                    for (int e = 0; e < d && yg != 0.0; ++e) dq[(i * p->n1 + h) * d + e] += yg * ldv(&p->k, krow * d + e);
                }
            }
    }
    return LIO_OK;
}

/* dK [nrows, d] of key rows (key axis row, key head) = (key_rows[i], heads[i]):
 * every selection of that key by any query row of its batch contributes. */
int lio_k_rows(const lio_problem *p, int64_t nrows, const int64_t *key_rows, const int32_t *heads, double *dk)
{
    int rc = check(p);
    if (rc) return rc;
    const int G = p->n1 / p->n2, d = p->d;
    memset(dk, 0, sizeof(double) * nrows * d);
    for (int64_t i = 0; i < nrows; ++i) {
        const int n2 = heads[i];
        int b = -1;
        for (int bb = 0; bb < p->batch; ++bb)
            if (key_rows[i] >= k0(p, bb) && key_rows[i] < k0(p, bb) + (p->cu_kv[bb + 1] - p->cu_kv[bb])) b = bb;
        if (b < 0 || n2 < 0 || n2 >= p->n2) return LIO_EARG;
        const int64_t id = key_rows[i] - k0(p, b);
        const int64_t krow = key_rows[i] * p->n2 + n2;
        for (int64_t t = q0(p, b); t < q0(p, b) + (p->cu_q[b + 1] - p->cu_q[b]); ++t)
            for (int j = 0; j < p->topk; ++j) {
                const int64_t sel = (t * p->n2 + n2) * p->topk + j;
                if (p->idx[sel] != id) continue;
                const double dyv = ldv(&p->dy, sel);
                for (int g = 0; g < G; ++g) {
                    const int64_t qrow = t * p->n1 + n2 * G + g;
                    double x = 0.0;
                    for (int e = 0; e < d; ++e) x += ldv(&p->q, qrow * d + e) * ldv(&p->k, krow * d + e);
                    const double yg = x > 0.0 ? dyv * ldv(&p->w, qrow) : 0.0;
                    for (int e = 0; e < d && yg != 0.0; ++e) dk[i * d + e] += yg * ldv(&p->q, qrow * d + e);
                }
            }
    }
    return LIO_OK;
}
