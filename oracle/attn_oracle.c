/*
 * attn_oracle.c -- fp64 CPU oracle for the masked / modified attention forward
 * and its backward (gradients of Q, K, V).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may call this code.  The CUDA library never
 * links, loads or calls it, and it shares no code with the CUDA library.
 *
 * What it computes is the plain definition of softmax attention, evaluated
 * literally for each requested query row: materialise every score of the row,
 * apply the score modification and the mask, take the softmax in double
 * precision, and form the output row and its log-sum-exp.  There is no tiling,
 * no online softmax, no block skipping and no approximate exponential.
 *
 * Sources for the definition:
 *  - "FlashAttention-4 explained" (theneuron.ai), section "What Is Attention,
 *    and Why Is It Expensive?": every query is compared against every key;
 *    section "Enter Tri Dao and FlashAttention": tiling changes only where
 *    the data lives, with no approximation, so the exact definition is the
 *    oracle.
 *  - same page, section "PyTorch Gets the Upgrade Too": the mod variants
 *    sliding window, ALiBi and soft-capping.
 *  - "PyTorch 2.5 Introduces FlexAttention and TorchDynamo C++ Runtime",
 *    section "What Happened?": sliding window, document packing, prefix
 *    masking; body text: a score modification is a function of the query
 *    position q_idx and key position k_idx.
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes):
 *  - the scale multiplies Q.K first, then ALiBi is added, then the soft cap
 *    cap*tanh(s/cap) is applied;
 *  - ALiBi adds -m_h*(qpos - kpos) with m_h = 2^(-8(h+1)/H) for 0-based query
 *    head h unless slopes are given;
 *  - enabled masks combine with AND; causal: kpos <= qpos; window W:
 *    qpos - W < kpos <= qpos; document: doc[i] == doc[j]; prefix-LM:
 *    kpos <= qpos OR kpos < prefix_len[b]; qpos = i + q_offset, kpos = j;
 *  - GQA: query head h reads KV head h / (H / H_kv);
 *  - a relative-position bias table adds rel_bias[h][clamp(kpos - qpos,
 *    -R, R) + R] after ALiBi and before the soft cap; a block map hides
 *    every (query, key) pair whose 128 x 128 tile it marks 0 (both are the
 *    "further descriptor mods" of the design: a generic relative-position
 *    bias and a user block mask);
 *  - LSE is the natural-log log-sum-exp of the modified scores over visible
 *    keys; a row with no visible key has O = 0 and LSE = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    OR_MASK_CAUSAL = 1,
    OR_MASK_WINDOW = 2,
    OR_MASK_DOCUMENT = 4,
    OR_MASK_PREFIX_LM = 8,
    OR_MASK_BLOCKS = 16,
};
enum {
    OR_SCORE_ALIBI = 1,
    OR_SCORE_SOFTCAP = 2,
    OR_SCORE_RELBIAS = 4,
};
enum { OR_BLOCK = 128 };  /* edge of a block-map tile, in rows and keys */

/* The score and mask modifications of one call. */
typedef struct or_mods {
    uint32_t mask_flags, score_flags;
    int window, q_offset;
    const int32_t *doc_ids;     /* [B][S_k] */
    const int32_t *prefix_len;  /* [B] */
    const double *alibi_slopes; /* [H] or NULL for 2^(-8(h+1)/H) */
    double softcap;
    const uint8_t *blocks;      /* [B or 1][ceil(S_q/128)][ceil(S_k/128)] */
    int blocks_batched;         /* 1: one map per batch entry */
    const double *rel_bias;     /* [H][2 * rel_max + 1] */
    int rel_max;
} or_mods;

/* A bfloat16 value is the upper 16 bits of an IEEE binary32 value, so the
 * conversion to double is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Is key j visible to query row i of batch b?  Each enabled mask is
 * evaluated as written and the results are combined with AND. */
static int visible(int64_t i, int64_t j, int b, int S_q, int S_k, const or_mods *m)
{
    int64_t qpos = i + (int64_t)m->q_offset;
    int64_t kpos = j;
    int vis = 1;
    if (m->mask_flags & OR_MASK_CAUSAL)
        vis = vis && (kpos <= qpos);
    if (m->mask_flags & OR_MASK_WINDOW)
        vis = vis && (qpos - (int64_t)m->window < kpos) && (kpos <= qpos);
    if (m->mask_flags & OR_MASK_DOCUMENT)
        vis = vis && (m->doc_ids[(int64_t)b * S_k + i] == m->doc_ids[(int64_t)b * S_k + j]);
    if (m->mask_flags & OR_MASK_PREFIX_LM)
        vis = vis && ((kpos <= qpos) || (kpos < (int64_t)m->prefix_len[b]));
    if (m->mask_flags & OR_MASK_BLOCKS) {
        const int64_t nq = (S_q + OR_BLOCK - 1) / OR_BLOCK, nk = (S_k + OR_BLOCK - 1) / OR_BLOCK;
        const int64_t mb = m->blocks_batched ? b : 0;
        vis = vis && m->blocks[(mb * nq + i / OR_BLOCK) * nk + j / OR_BLOCK] != 0;
    }
    return vis;
}

/* The modified score of (row i of head h, key j) from the scaled dot
 * product x: ALiBi, then the relative-position bias, then the soft cap. */
static double modified_score(double x, int64_t i, int64_t j, int h, int H, const or_mods *m)
{
    const double qpos = (double)(i + m->q_offset);
    double s = x;
    if (m->score_flags & OR_SCORE_ALIBI) {
        const double slope = m->alibi_slopes ? m->alibi_slopes[h]
                                             : pow(2.0, -8.0 * (double)(h + 1) / (double)H);
        s += -slope * (qpos - (double)j);
    }
    if (m->score_flags & OR_SCORE_RELBIAS) {
        int64_t r = j - (i + (int64_t)m->q_offset);
        if (r < -(int64_t)m->rel_max)
            r = -(int64_t)m->rel_max;
        if (r > (int64_t)m->rel_max)
            r = (int64_t)m->rel_max;
        s += m->rel_bias[(int64_t)h * (2 * (int64_t)m->rel_max + 1) + r + m->rel_max];
    }
    if (m->score_flags & OR_SCORE_SOFTCAP)
        s = m->softcap * tanh(s / m->softcap);
    return s;
}

static int check_dims(int B, int H, int H_kv, int S_q, int S_k, int D, const or_mods *m)
{
    if (B <= 0 || H <= 0 || H_kv <= 0 || S_q <= 0 || S_k <= 0 || D <= 0)
        return -1;
    if (H % H_kv != 0)
        return -1;
    if ((m->mask_flags & OR_MASK_DOCUMENT) && (m->doc_ids == NULL || S_q != S_k))
        return -1;
    if ((m->mask_flags & OR_MASK_PREFIX_LM) && m->prefix_len == NULL)
        return -1;
    if ((m->mask_flags & OR_MASK_BLOCKS) && m->blocks == NULL)
        return -1;
    if ((m->score_flags & OR_SCORE_SOFTCAP) && !(m->softcap > 0.0))
        return -1;
    if ((m->score_flags & OR_SCORE_RELBIAS) && (m->rel_bias == NULL || m->rel_max < 0))
        return -1;
    return 0;
}

/*
 * oracle_attn_rows: attention forward for a list of query rows.
 *
 *  q      bf16 bits, [B][H][S_q][D]
 *  k, v   bf16 bits, [B][H_kv][S_k][D]
 *  scale  the softmax scale as the caller's float value
 *  rows   flattened row ids r = (b*H + h)*S_q + i, n_rows of them
 *  out    [n_rows][D] doubles, O rows (unrounded)
 *  lse    [n_rows] doubles, natural-log LSE (-inf for rows with no key)
 *  probs  optional [n_rows][S_k] doubles: the softmax probability of every
 *         key (0 for hidden keys); NULL to skip
 *  alibi_slopes  optional [H] doubles; NULL means 2^(-8(h+1)/H)
 *  doc_ids [B][S_k] int32 (needed with the document mask, S_q == S_k)
 *  prefix_len [B] int32 (needed with the prefix-LM mask)
 *
 * Returns 0 on success, -1 on an argument error.
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int B, int H, int H_kv, int S_q, int S_k, int D,
                     double scale, const or_mods *m, const int64_t *rows, int64_t n_rows,
                     double *out, double *lse, double *probs)
{
    if (check_dims(B, H, H_kv, S_q, S_k, D, m))
        return -1;
    const int group = H / H_kv;
    int bad = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S_k);
        unsigned char *vis = (unsigned char *)malloc((size_t)S_k);
        double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
        if (s == NULL || vis == NULL || qrow == NULL) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                int64_t row = rows[r];
                if (row < 0 || row >= (int64_t)B * H * S_q) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                int64_t i = row % S_q;
                int h = (int)((row / S_q) % H);
                int b = (int)(row / ((int64_t)S_q * H));
                int hk = h / group;
                const uint16_t *qp = q + (((int64_t)b * H + h) * S_q + i) * D;
                const uint16_t *kb = k + ((int64_t)b * H_kv + hk) * (int64_t)S_k * D;
                const uint16_t *vb = v + ((int64_t)b * H_kv + hk) * (int64_t)S_k * D;
                for (int d = 0; d < D; ++d)
                    qrow[d] = bf16_to_double(qp[d]);

                /* scores of every key, then the mods, then the mask */
                double M = -INFINITY;
                for (int64_t j = 0; j < S_k; ++j) {
                    const uint16_t *kp = kb + j * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += qrow[d] * bf16_to_double(kp[d]);
                    const double sj = modified_score(scale * dot, i, j, h, H, m);
                    s[j] = sj;
                    vis[j] = (unsigned char)visible(i, j, b, S_q, S_k, m);
                    if (vis[j] && sj > M)
                        M = sj;
                }

                double *o = out + r * D;
                for (int d = 0; d < D; ++d)
                    o[d] = 0.0;
                if (M == -INFINITY) {
                    /* no visible key: O = 0, LSE = -inf */
                    lse[r] = -INFINITY;
                    if (probs)
                        memset(probs + r * S_k, 0, sizeof(double) * (size_t)S_k);
                    continue;
                }
                double Z = 0.0;
                for (int64_t j = 0; j < S_k; ++j)
                    if (vis[j])
                        Z += exp(s[j] - M);
                for (int64_t j = 0; j < S_k; ++j) {
                    double p = vis[j] ? exp(s[j] - M) / Z : 0.0;
                    if (probs)
                        probs[r * S_k + j] = p;
                    if (p != 0.0) {
                        const uint16_t *vp = vb + j * D;
                        for (int d = 0; d < D; ++d)
                            o[d] += p * bf16_to_double(vp[d]);
                    }
                }
                lse[r] = M + log(Z);
            }
        }
        free(s);
        free(vis);
        free(qrow);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------
 * Backward: gradients of the attention forward with respect to Q, K and V,
 * given the gradient dO of the output, from the same plain definition.
 *
 * Source: the forward's definition above and calculus.  The pages name the
 * backward pass as the step after the forward ("FlashAttention-4
 * explained", section "FlashAttention-4: Built for Blackwell") but print no
 * formula, so the gradient is written out from the chain rule:
 *
 *   x_ij  = scale * q_i . k_j                      (scaled score)
 *   s_ij  = mod(x_ij)  (+ ALiBi bias, then cap * tanh(./cap))
 *   p_ij  = exp(s_ij - LSE_i) on visible keys, 0 elsewhere
 *   O_i   = sum_j p_ij v_j
 *   dV_j  = sum_i p_ij dO_i                        (over every query head of
 *   dP_ij = dO_i . v_j                              the K/V head's group)
 *   dS_ij = p_ij (dP_ij - sum_j' p_ij' dP_ij')      (softmax Jacobian)
 *         = p_ij (dP_ij - dO_i . O_i)
 *   dX_ij = dS_ij * ds/dx,  ds/dx = 1, or 1 - (s_ij/cap)^2 with the soft cap
 *   dQ_i  = scale * sum_j dX_ij k_j
 *   dK_j  = scale * sum_i dX_ij q_i                (summed over the group)
 *
 * Rows with no visible key contribute nothing (p = 0 everywhere).
 * ------------------------------------------------------------------------ */

/* The forward of one query row: scores after the mods s[], visibility vis[],
 * probabilities p[], the output row o[] and the natural-log LSE (-inf and
 * all-zero p/o when no key is visible).  Returns 0, or -1 when no key is
 * visible. */
static int row_forward(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       int b, int h, int64_t i, int H, int H_kv, int S_q, int S_k,
                       int D, double scale, const or_mods *m, double *qrow,
                       double *s, unsigned char *vis, double *p, double *o,
                       double *lse)
{
    const int hk = h / (H / H_kv);
    const uint16_t *qp = q + (((int64_t)b * H + h) * S_q + i) * D;
    const uint16_t *kb = k + ((int64_t)b * H_kv + hk) * (int64_t)S_k * D;
    const uint16_t *vb = v + ((int64_t)b * H_kv + hk) * (int64_t)S_k * D;
    for (int d = 0; d < D; ++d)
        qrow[d] = bf16_to_double(qp[d]);
    double M = -INFINITY;
    for (int64_t j = 0; j < S_k; ++j) {
        const uint16_t *kp = kb + j * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qrow[d] * bf16_to_double(kp[d]);
        const double sj = modified_score(scale * dot, i, j, h, H, m);
        s[j] = sj;
        vis[j] = (unsigned char)visible(i, j, b, S_q, S_k, m);
        if (vis[j] && sj > M)
            M = sj;
    }
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (M == -INFINITY) {
        memset(p, 0, sizeof(double) * (size_t)S_k);
        *lse = -INFINITY;
        return -1;
    }
    double Z = 0.0;
    for (int64_t j = 0; j < S_k; ++j)
        if (vis[j])
            Z += exp(s[j] - M);
    for (int64_t j = 0; j < S_k; ++j) {
        p[j] = vis[j] ? exp(s[j] - M) / Z : 0.0;
        if (p[j] != 0.0) {
            const uint16_t *vp = vb + j * D;
            for (int d = 0; d < D; ++d)
                o[d] += p[j] * bf16_to_double(vp[d]);
        }
    }
    *lse = M + log(Z);
    return 0;
}

/* d s / d x of the score modification at modified score s. */
static double mod_slope(double s, const or_mods *m)
{
    if (m->score_flags & OR_SCORE_SOFTCAP) {
        double t = s / m->softcap;
        return 1.0 - t * t;
    }
    return 1.0;
}

/*
 * oracle_attn_bwd_rows: dQ of a list of query rows.
 *
 *  q, k, v, arguments as oracle_attn_rows; dout bf16 bits [B][H][S_q][D]
 *  rows   flattened (b*H + h)*S_q + i
 *  dq     [n_rows][D] doubles
 */
int oracle_attn_bwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *dout, int B, int H, int H_kv, int S_q, int S_k,
                         int D, double scale, const or_mods *m, const int64_t *rows,
                         int64_t n_rows, double *dq)
{
    if (check_dims(B, H, H_kv, S_q, S_k, D, m))
        return -1;
    const int group = H / H_kv;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S_k);
        double *p = (double *)malloc(sizeof(double) * (size_t)S_k);
        unsigned char *vis = (unsigned char *)malloc((size_t)S_k);
        double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
        double *g = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !p || !vis || !qrow || !o || !g) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                const int64_t row = rows[r];
                if (row < 0 || row >= (int64_t)B * H * S_q) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                const int64_t i = row % S_q;
                const int h = (int)((row / S_q) % H);
                const int b = (int)(row / ((int64_t)S_q * H));
                const int hk = h / group;
                double *dqr = dq + r * D;
                for (int d = 0; d < D; ++d)
                    dqr[d] = 0.0;
                double lse;
                if (row_forward(q, k, v, b, h, i, H, H_kv, S_q, S_k, D, scale, m, qrow, s, vis,
                                p, o, &lse) != 0)
                    continue;
                const uint16_t *dop = dout + (((int64_t)b * H + h) * S_q + i) * D;
                const uint16_t *kb = k + ((int64_t)b * H_kv + hk) * (int64_t)S_k * D;
                const uint16_t *vb = v + ((int64_t)b * H_kv + hk) * (int64_t)S_k * D;
                double delta = 0.0;
                for (int d = 0; d < D; ++d) {
                    g[d] = bf16_to_double(dop[d]);
                    delta += g[d] * o[d];
                }
                for (int64_t j = 0; j < S_k; ++j) {
                    if (p[j] == 0.0)
                        continue;
                    const uint16_t *vp = vb + j * D;
                    double dp = 0.0;
                    for (int d = 0; d < D; ++d)
                        dp += g[d] * bf16_to_double(vp[d]);
                    const double dx = p[j] * (dp - delta) * mod_slope(s[j], m);
                    const uint16_t *kp = kb + j * D;
                    for (int d = 0; d < D; ++d)
                        dqr[d] += scale * dx * bf16_to_double(kp[d]);
                }
            }
        }
        free(s);
        free(p);
        free(vis);
        free(qrow);
        free(o);
        free(g);
    }
    return bad ? -1 : 0;
}

/*
 * oracle_attn_bwd_keys: dK and dV of a list of key positions.
 *
 *  keys   flattened (b*H_kv + hk)*S_k + j
 *  dk, dv [n_keys][D] doubles, summed over the H/H_kv query heads of the
 *         K/V head
 *
 * Needs every query row of the K/V head's group: their LSE and
 * dO_i . O_i are computed once per (b, hk) that appears in keys.
 */
int oracle_attn_bwd_keys(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *dout, int B, int H, int H_kv, int S_q, int S_k,
                         int D, double scale, const or_mods *m, const int64_t *keys,
                         int64_t n_keys, double *dk, double *dv)
{
    if (check_dims(B, H, H_kv, S_q, S_k, D, m))
        return -1;
    const int group = H / H_kv;
    for (int64_t r = 0; r < n_keys; ++r)
        if (keys[r] < 0 || keys[r] >= (int64_t)B * H_kv * S_k)
            return -1;
    const int64_t n_rows = (int64_t)group * S_q;  /* query rows of one K/V head */
    double *lse = (double *)malloc(sizeof(double) * (size_t)n_rows);
    double *delta = (double *)malloc(sizeof(double) * (size_t)n_rows);
    if (!lse || !delta) {
        free(lse);
        free(delta);
        return -1;
    }
    int bad = 0;
    for (int64_t bh = 0; bh < (int64_t)B * H_kv; ++bh) {
        int any = 0;
        for (int64_t r = 0; r < n_keys; ++r)
            if (keys[r] / S_k == bh)
                any = 1;
        if (!any)
            continue;
        const int b = (int)(bh / H_kv), hk = (int)(bh % H_kv);
        /* every query row of the group: LSE and dO . O */
#pragma omp parallel
        {
            double *s = (double *)malloc(sizeof(double) * (size_t)S_k);
            double *p = (double *)malloc(sizeof(double) * (size_t)S_k);
            unsigned char *vis = (unsigned char *)malloc((size_t)S_k);
            double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
            double *o = (double *)malloc(sizeof(double) * (size_t)D);
            if (!s || !p || !vis || !qrow || !o) {
#pragma omp atomic write
                bad = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (int64_t rr = 0; rr < n_rows; ++rr) {
                    const int h = hk * group + (int)(rr / S_q);
                    const int64_t i = rr % S_q;
                    double l;
                    row_forward(q, k, v, b, h, i, H, H_kv, S_q, S_k, D, scale, m, qrow, s, vis, p,
                                o, &l);
                    const uint16_t *dop = dout + (((int64_t)b * H + h) * S_q + i) * D;
                    double dd = 0.0;
                    for (int d = 0; d < D; ++d)
                        dd += bf16_to_double(dop[d]) * o[d];
                    lse[rr] = l;
                    delta[rr] = dd;
                }
            }
            free(s);
            free(p);
            free(vis);
            free(qrow);
            free(o);
        }
        /* each requested key of this head: sum over the group's rows */
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_keys; ++r) {
            if (keys[r] / S_k != bh)
                continue;
            const int64_t j = keys[r] % S_k;
            const uint16_t *kp = k + ((int64_t)bh * S_k + j) * D;
            const uint16_t *vp = v + ((int64_t)bh * S_k + j) * D;
            double *dkr = dk + r * D, *dvr = dv + r * D;
            for (int d = 0; d < D; ++d)
                dkr[d] = dvr[d] = 0.0;
            for (int64_t rr = 0; rr < n_rows; ++rr) {
                if (lse[rr] == -INFINITY)
                    continue;
                const int h = hk * group + (int)(rr / S_q);
                const int64_t i = rr % S_q;
                if (!visible(i, j, b, S_q, S_k, m))
                    continue;
                const uint16_t *qp = q + (((int64_t)b * H + h) * S_q + i) * D;
                const uint16_t *dop = dout + (((int64_t)b * H + h) * S_q + i) * D;
                double dot = 0.0, dp = 0.0;
                for (int d = 0; d < D; ++d) {
                    dot += bf16_to_double(qp[d]) * bf16_to_double(kp[d]);
                    dp += bf16_to_double(dop[d]) * bf16_to_double(vp[d]);
                }
                const double sj = modified_score(scale * dot, i, j, h, H, m);
                const double pj = exp(sj - lse[rr]);
                const double dx = pj * (dp - delta[rr]) * mod_slope(sj, m);
                for (int d = 0; d < D; ++d) {
                    dvr[d] += pj * bf16_to_double(dop[d]);
                    dkr[d] += scale * dx * bf16_to_double(qp[d]);
                }
            }
        }
    }
    free(lse);
    free(delta);
    return bad ? -1 : 0;
}
