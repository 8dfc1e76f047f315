/*
 * Plain fp64 CPU oracle for NSA selected-attention backward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the GPU library must compute.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * Sources (operator documentation pages):
 *   [NSA]  "NsaSelectedAttentionGrad" README (ops-transformer):
 *          section "function description" (Gather formula for selectedKey /
 *          selectedValue; backward formulas for dV, dQ, dK),
 *          section "parameters" (query, key, value, attentionOut,
 *          attentionOutGrad, softmaxMax, softmaxSum, topkIndices, scaleValue),
 *          section "constraints" (TND layout, G = N1/N2, stat shape
 *          [T1,N1,8], topkIndices shape [T1,N2,selectedBlockCount]).
 *   [FA]   "aclnnFlashAttentionUnpaddingScoreGradV3": Formula section
 *          (forward S = QK^T/sqrt(d), P = Softmax(S), Y = PV; backward
 *          dV = P^T dY, dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d)).
 *
 * Readings taken where the pages are silent (all stated, nothing hidden):
 *   - the gathered key rows of (token t in batch b, KV head n2) are
 *     cu_kv[b] + idx*bs + r for each idx in topkIndices[t][n2][:] in list
 *     order and r in [0,bs): block ids are local to the batch;
 *   - query head h uses KV head h / G (consecutive heads share a KV head);
 *   - no mask: every gathered row is attended; duplicate ids count twice;
 *   - softmaxMax is the row max of scale*q.k over the gathered rows and
 *     softmaxSum the sum of exp(scale*q.k - max); all 8 lanes are equal and
 *     lane 0 is read;
 *   - the backward uses the GIVEN attentionOut and stats:
 *       P_j  = exp(s_j - max) / sum,       s_j = scale * <q, k_j>
 *       Delta = sum_d dY_d * O_d            (row-wise)
 *       dP_j = <dY, v_j>,  dS_j = P_j (dP_j - Delta)
 *       dQ   = scale * sum_j dS_j k_j
 *       dK_j += scale * dS_j q,   dV_j += P_j dY   (scatter-add to key rows)
 *     with scale = scaleValue (the reciprocal of sqrt(d) in the formula).
 *   - layouts (the lightning-indexer page allows TND or BSND; the README's
 *     calling section has a non-TND sample): in TND the rows of batch b are
 *     cu_q[b] .. cu_q[b+1]-1 (keys: cu_kv); in BSND every batch is padded to
 *     s1_max query / s2_max key rows, batch b starts at row b * s1_max
 *     (b * s2_max) and cu_q / cu_kv hold the prefix sums of the valid lengths.
 *     Padding rows take no part in the result; their gradients stay zero.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element types an input array may hold */
enum { SAO_F64 = 0, SAO_BF16 = 1, SAO_F16 = 2, SAO_F32 = 3 };

/* status codes */
enum { SAO_OK = 0, SAO_EARG = -1, SAO_EINDEX = -2, SAO_ENOMEM = -3 };

typedef struct {
    const void *data;
    int32_t dtype;  /* SAO_* */
    int32_t pad_;
} sao_tensor;

/* One selected-attention problem in TND layout (see [NSA] constraints). */
typedef struct {
    int32_t batch;            /* B */
    int32_t n1, n2;           /* query heads, key/value heads; n1 % n2 == 0 */
    int32_t d_qk, d_v;        /* head dims of q/k and of v/o/dy */
    int32_t block_size;       /* selectedBlockSize */
    int32_t block_count;      /* selectedBlockCount */
    int32_t stat_stride;      /* elements between rows of softmaxMax/Sum (8 in the op layout) */
    double scale;             /* scaleValue */
    const int32_t *cu_q;      /* B+1 prefix sums of query lengths (host) */
    const int32_t *cu_kv;     /* B+1 prefix sums of key lengths (host) */
    const int32_t *topk;      /* [T1, n2, block_count] block ids, batch local */
    sao_tensor q;             /* [T1, n1, d_qk] */
    sao_tensor k;             /* [T2, n2, d_qk] */
    sao_tensor v;             /* [T2, n2, d_v]  */
    sao_tensor o;             /* [T1, n1, d_v]  attentionOut (backward only) */
    sao_tensor dy;            /* [T1, n1, d_v]  attentionOutGrad (backward only) */
    sao_tensor smax;          /* [T1, n1, stat_stride] softmaxMax (backward only) */
    sao_tensor ssum;          /* [T1, n1, stat_stride] softmaxSum (backward only) */
    int32_t layout;           /* 0: TND; 1: BSND, every batch padded to s1_max / s2_max rows */
    int32_t s1_max, s2_max;   /* BSND only */
    int32_t pad_;
} sao_problem;

/* ---- element decoding (exact: every 16-bit and fp32 value is a double) ---- */

static double dec_bf16(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double dec_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);   /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double ld(const sao_tensor *t, int64_t i)
{
    switch (t->dtype) {
    case SAO_F64: return ((const double *)t->data)[i];
    case SAO_BF16: return dec_bf16(((const uint16_t *)t->data)[i]);
    case SAO_F16: return dec_f16(((const uint16_t *)t->data)[i]);
    default: return (double)((const float *)t->data)[i];
    }
}

/* ---- problem bookkeeping ---- */

/* first query / key row of batch b, and its valid query rows */
static int64_t q_row0(const sao_problem *p, int b) { return p->layout ? (int64_t)b * p->s1_max : p->cu_q[b]; }
static int64_t kv_row0(const sao_problem *p, int b) { return p->layout ? (int64_t)b * p->s2_max : p->cu_kv[b]; }
static int64_t q_len(const sao_problem *p, int b) { return p->cu_q[b + 1] - p->cu_q[b]; }

/* rows along the query / key axis of the tensors */
static int64_t total_q(const sao_problem *p) { return p->layout ? (int64_t)p->batch * p->s1_max : p->cu_q[p->batch]; }
static int64_t total_kv(const sao_problem *p)
{
    return p->layout ? (int64_t)p->batch * p->s2_max : p->cu_kv[p->batch];
}

/* batch of a valid query row, -1 for a padding row or one out of range */
static int batch_of_token(const sao_problem *p, int64_t t)
{
    for (int b = 0; b < p->batch; ++b)
        if (t >= q_row0(p, b) && t < q_row0(p, b) + q_len(p, b)) return b;
    return -1;
}

static int check_problem(const sao_problem *p)
{
    if (!p || p->batch < 1 || p->n1 < 1 || p->n2 < 1 || p->n1 % p->n2 != 0) return SAO_EARG;
    if (p->d_qk < 1 || p->d_v < 1 || p->block_size < 1 || p->block_count < 1) return SAO_EARG;
    if (!p->cu_q || !p->cu_kv || !p->topk) return SAO_EARG;
    if (p->cu_q[0] != 0 || p->cu_kv[0] != 0) return SAO_EARG;
    if (p->layout != 0 && p->layout != 1) return SAO_EARG;
    for (int b = 0; b < p->batch; ++b) {
        if (p->cu_q[b + 1] < p->cu_q[b] || p->cu_kv[b + 1] < p->cu_kv[b]) return SAO_EARG;
        if (p->layout && (q_len(p, b) > p->s1_max || p->cu_kv[b + 1] - p->cu_kv[b] > p->s2_max)) return SAO_EARG;
    }
    return SAO_OK;
}

/*
 * [NSA] function description, Gather:
 *   selectedKey = Gather(key, topkIndices[i]), 0 <= i < selectedBlockCount
 * Writes the L = block_count * block_size key-row ids (rows of the [T2] axis)
 * gathered for token t of batch b and KV head n2, in list order.
 */
static int gather_rows(const sao_problem *p, int b, int64_t t, int n2, int64_t *rows)
{
    const int32_t *ids = p->topk + ((int64_t)t * p->n2 + n2) * p->block_count;
    int64_t s2 = p->cu_kv[b + 1] - p->cu_kv[b];
    int64_t nblk = s2 / p->block_size;
    int64_t L = 0;
    for (int i = 0; i < p->block_count; ++i) {
        int64_t id = ids[i];
        if (id < 0 || id >= nblk) return SAO_EINDEX;
        for (int r = 0; r < p->block_size; ++r) rows[L++] = kv_row0(p, b) + id * p->block_size + r;
    }
    return SAO_OK;
}

/* Delta = sum_d dY[t,h,d] * O[t,h,d]  (softmax adjoint term of dS) */
static double row_delta(const sao_problem *p, int64_t t, int h)
{
    int64_t off = ((int64_t)t * p->n1 + h) * p->d_v;
    double acc = 0.0;
    for (int d = 0; d < p->d_v; ++d) acc += ld(&p->dy, off + d) * ld(&p->o, off + d);
    return acc;
}

/* dP_j = <dY[t,h], v[row_j, n2]> */
static double dp_of(const sao_problem *p, int64_t t, int h, int n2, int64_t row)
{
    int64_t yoff = ((int64_t)t * p->n1 + h) * p->d_v;
    int64_t voff = (row * p->n2 + n2) * p->d_v;
    double acc = 0.0;
    for (int d = 0; d < p->d_v; ++d) acc += ld(&p->dy, yoff + d) * ld(&p->v, voff + d);
    return acc;
}

/* s_j = scale * <q[t,h], k[row, n2]>  ([FA] forward: S = QK^T / sqrt(d)) */
static double score_of(const sao_problem *p, int64_t t, int h, int n2, int64_t row)
{
    int64_t qoff = ((int64_t)t * p->n1 + h) * p->d_qk;
    int64_t koff = (row * p->n2 + n2) * p->d_qk;
    double acc = 0.0;
    for (int d = 0; d < p->d_qk; ++d) acc += ld(&p->q, qoff + d) * ld(&p->k, koff + d);
    return p->scale * acc;
}

/*
 * Forward over the gathered rows ([FA] forward with no pse, mask or
 * dropout; [NSA] parameters: attentionOut, softmaxMax, softmaxSum are the
 * forward's outputs).  For every (t, h):
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  O = sum_j exp(s_j - m)/l * v_j
 * Outputs: o [T1, n1, d_v], m and l [T1, n1] (one value per row).
 */
/* forward of one row (t, h) of batch b into o_row[d_v], *m, *l */
static int row_forward(const sao_problem *p, int b, int64_t t, int h, int64_t *rows, double *s,
                       double *o_row, double *m_out, double *l_out)
{
    int G = p->n1 / p->n2;
    int n2 = h / G;
    int64_t L = (int64_t)p->block_count * p->block_size;
    int rc = gather_rows(p, b, t, n2, rows);
    if (rc) return rc;
    for (int64_t j = 0; j < L; ++j) s[j] = score_of(p, t, h, n2, rows[j]);
    double m = -INFINITY;
    for (int64_t j = 0; j < L; ++j) if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < L; ++j) l += exp(s[j] - m);
    for (int d = 0; d < p->d_v; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j < L; ++j) {
        double pj = exp(s[j] - m) / l;
        int64_t voff = (rows[j] * p->n2 + n2) * p->d_v;
        for (int d = 0; d < p->d_v; ++d) o_row[d] += pj * ld(&p->v, voff + d);
    }
    *m_out = m;
    *l_out = l;
    return SAO_OK;
}

int sao_forward(const sao_problem *p, double *o, double *m_out, double *l_out)
{
    int rc = check_problem(p);
    if (rc) return rc;
    int64_t L = (int64_t)p->block_count * p->block_size;
    int64_t *rows = malloc(sizeof(int64_t) * L);
    double *s = malloc(sizeof(double) * L);
    if (!rows || !s) { free(rows); free(s); return SAO_ENOMEM; }
    for (int b = 0; b < p->batch && rc == SAO_OK; ++b)
        for (int64_t t = q_row0(p, b); t < q_row0(p, b) + q_len(p, b) && rc == SAO_OK; ++t)
            for (int h = 0; h < p->n1 && rc == SAO_OK; ++h) {
                int64_t r = (int64_t)t * p->n1 + h;
                rc = row_forward(p, b, t, h, rows, s, o + r * p->d_v, m_out + r, l_out + r);
            }
    free(rows);
    free(s);
    return rc;
}

/* Forward of selected rows only: rows_th[i] = t * n1 + h; o is [nrows, d_v]. */
int sao_forward_rows(const sao_problem *p, int64_t nrows, const int64_t *rows_th, double *o,
                     double *m_out, double *l_out)
{
    int rc = check_problem(p);
    if (rc) return rc;
    int64_t L = (int64_t)p->block_count * p->block_size;
    int64_t *rows = malloc(sizeof(int64_t) * L);
    double *s = malloc(sizeof(double) * L);
    if (!rows || !s) { free(rows); free(s); return SAO_ENOMEM; }
    for (int64_t i = 0; i < nrows && rc == SAO_OK; ++i) {
        int64_t t = rows_th[i] / p->n1;
        int h = (int)(rows_th[i] % p->n1);
        int b = batch_of_token(p, t);
        if (b < 0) { rc = SAO_EARG; break; }
        rc = row_forward(p, b, t, h, rows, s, o + i * p->d_v, m_out + i, l_out + i);
    }
    free(rows);
    free(s);
    return rc;
}

/*
 * Backward of one query row (t, h) over its gathered rows.
 *   dq_row  (may be NULL): receives scale * sum_j dS_j k_j
 *   dk, dv  (may be NULL): dK_j += scale dS_j q and dV_j += P_j dY for every
 *           gathered row j.  With only_block < 0 they are the full
 *           [T2, n2, d] arrays; otherwise they are [block_size, d] arrays of
 *           block only_block and only rows of that block are visited.
 * [NSA] function description (dV = P^T dY, dQ = dS K/sqrt(d),
 * dK = dS^T Q/sqrt(d)); [FA] Formula (same, dense form).  P_j only needs s_j
 * and the given stats, so each j is independent of the others.
 */
static int row_backward(const sao_problem *p, int b, int64_t t, int h, int64_t *rows,
                        double *dq_row, double *dk, double *dv, int only_block)
{
    int G = p->n1 / p->n2;
    int n2 = h / G;
    int64_t L = (int64_t)p->block_count * p->block_size;
    int rc = gather_rows(p, b, t, n2, rows);
    if (rc) return rc;
    /* key row -> first element of its dK / dV row in the target arrays */
    int64_t blk_row0 = only_block < 0 ? 0 : kv_row0(p, b) + (int64_t)only_block * p->block_size;
    int64_t srow = ((int64_t)t * p->n1 + h) * p->stat_stride;
    double m = ld(&p->smax, srow);       /* lane 0 */
    double l = ld(&p->ssum, srow);
    double delta = row_delta(p, t, h);
    int64_t qoff = ((int64_t)t * p->n1 + h) * p->d_qk;
    int64_t yoff = ((int64_t)t * p->n1 + h) * p->d_v;
    if (dq_row)
        for (int d = 0; d < p->d_qk; ++d) dq_row[d] = 0.0;
    const int32_t *ids = p->topk + ((int64_t)t * p->n2 + n2) * p->block_count;
    for (int64_t j = 0; j < L; ++j) {
        int blk = ids[j / p->block_size];
        int want_dq = dq_row != NULL;
        int want_kv = (dk || dv) && (only_block < 0 || blk == only_block);
        if (!want_dq && !want_kv) continue;
        double sj = score_of(p, t, h, n2, rows[j]);
        double pj = exp(sj - m) / l;
        double dsj = pj * (dp_of(p, t, h, n2, rows[j]) - delta);
        int64_t koff = (rows[j] * p->n2 + n2) * p->d_qk;
        int64_t tk = only_block < 0 ? koff : (rows[j] - blk_row0) * p->d_qk;
        int64_t tv = only_block < 0 ? (rows[j] * p->n2 + n2) * p->d_v : (rows[j] - blk_row0) * p->d_v;
        if (want_dq)
            for (int d = 0; d < p->d_qk; ++d) dq_row[d] += p->scale * dsj * ld(&p->k, koff + d);
        if (want_kv && dk)
            for (int d = 0; d < p->d_qk; ++d) dk[tk + d] += p->scale * dsj * ld(&p->q, qoff + d);
        if (want_kv && dv)
            for (int d = 0; d < p->d_v; ++d) dv[tv + d] += pj * ld(&p->dy, yoff + d);
    }
    return SAO_OK;
}

/* Full backward: dq [T1,n1,d_qk], dk [T2,n2,d_qk], dv [T2,n2,d_v]; key rows
 * nobody selected keep dK = dV = 0. */
int sao_backward(const sao_problem *p, double *dq, double *dk, double *dv)
{
    int rc = check_problem(p);
    if (rc) return rc;
    int64_t T2 = total_kv(p);
    memset(dk, 0, sizeof(double) * T2 * p->n2 * p->d_qk);
    memset(dv, 0, sizeof(double) * T2 * p->n2 * p->d_v);
    int64_t L = (int64_t)p->block_count * p->block_size;
    int64_t *rows = malloc(sizeof(int64_t) * L);
    if (!rows) return SAO_ENOMEM;
    for (int b = 0; b < p->batch && rc == SAO_OK; ++b)
        for (int64_t t = q_row0(p, b); t < q_row0(p, b) + q_len(p, b) && rc == SAO_OK; ++t)
            for (int h = 0; h < p->n1 && rc == SAO_OK; ++h)
                rc = row_backward(p, b, t, h, rows, dq + ((int64_t)t * p->n1 + h) * p->d_qk, dk, dv, -1);
    free(rows);
    return rc;
}

/* dQ of selected rows only: rows_th[i] = t * n1 + h; dq is [nrows, d_qk]. */
int sao_dq_rows(const sao_problem *p, int64_t nrows, const int64_t *rows_th, double *dq)
{
    int rc = check_problem(p);
    if (rc) return rc;
    int64_t L = (int64_t)p->block_count * p->block_size;
    int64_t *rows = malloc(sizeof(int64_t) * L);
    if (!rows) return SAO_ENOMEM;
    for (int64_t i = 0; i < nrows && rc == SAO_OK; ++i) {
        int64_t t = rows_th[i] / p->n1;
        int h = (int)(rows_th[i] % p->n1);
        int b = batch_of_token(p, t);
        if (b < 0 || t >= total_q(p)) { rc = SAO_EARG; break; }
        rc = row_backward(p, b, t, h, rows, dq + i * p->d_qk, NULL, NULL, -1);
    }
    free(rows);
    return rc;
}

/*
 * dK and dV of one key block (batch b, KV head n2, block id kb) from the query
 * tokens t in [t_lo, t_hi) of batch b: every such row whose list for n2 names
 * kb contributes (once per naming).  dk_blk is [block_size, d_qk], dv_blk is
 * [block_size, d_v]; both are overwritten.
 */
int sao_dkdv_block_range(const sao_problem *p, int b, int n2, int kb, int64_t t_lo, int64_t t_hi,
                         double *dk_blk, double *dv_blk)
{
    int rc = check_problem(p);
    if (rc) return rc;
    if (b < 0 || b >= p->batch || n2 < 0 || n2 >= p->n2 || kb < 0) return SAO_EARG;
    if (t_lo < q_row0(p, b)) t_lo = q_row0(p, b);
    if (t_hi > q_row0(p, b) + q_len(p, b)) t_hi = q_row0(p, b) + q_len(p, b);
    int G = p->n1 / p->n2;
    int64_t L = (int64_t)p->block_count * p->block_size;
    memset(dk_blk, 0, sizeof(double) * p->block_size * p->d_qk);
    memset(dv_blk, 0, sizeof(double) * p->block_size * p->d_v);
    int64_t *rows = malloc(sizeof(int64_t) * L);
    if (!rows) return SAO_ENOMEM;
    for (int64_t t = t_lo; t < t_hi && rc == SAO_OK; ++t) {
        const int32_t *ids = p->topk + ((int64_t)t * p->n2 + n2) * p->block_count;
        int hit = 0;
        for (int i = 0; i < p->block_count; ++i) hit |= ids[i] == kb;
        if (!hit) continue;
        for (int g = 0; g < G && rc == SAO_OK; ++g)
            rc = row_backward(p, b, t, n2 * G + g, rows, NULL, dk_blk, dv_blk, kb);
    }
    free(rows);
    return rc;
}

/* dK and dV of one key block from all query tokens of its batch. */
int sao_dkdv_block(const sao_problem *p, int b, int n2, int kb, double *dk_blk, double *dv_blk)
{
    if (!p || b < 0 || b >= p->batch) return SAO_EARG;
    return sao_dkdv_block_range(p, b, n2, kb, q_row0(p, b), q_row0(p, b) + q_len(p, b), dk_blk, dv_blk);
}
