/*
 * attn_oracle.c -- fp64 CPU oracle for the masked / modified attention forward.
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
};
enum {
    OR_SCORE_ALIBI = 1,
    OR_SCORE_SOFTCAP = 2,
};

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
static int visible(int64_t i, int64_t j, int b, int S_k, uint32_t mask_flags,
                   int window, int q_offset, const int32_t *doc_ids,
                   const int32_t *prefix_len)
{
    int64_t qpos = i + (int64_t)q_offset;
    int64_t kpos = j;
    int vis = 1;
    if (mask_flags & OR_MASK_CAUSAL)
        vis = vis && (kpos <= qpos);
    if (mask_flags & OR_MASK_WINDOW)
        vis = vis && (qpos - (int64_t)window < kpos) && (kpos <= qpos);
    if (mask_flags & OR_MASK_DOCUMENT)
        vis = vis && (doc_ids[(int64_t)b * S_k + i] == doc_ids[(int64_t)b * S_k + j]);
    if (mask_flags & OR_MASK_PREFIX_LM)
        vis = vis && ((kpos <= qpos) || (kpos < (int64_t)prefix_len[b]));
    return vis;
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
                     double scale, uint32_t mask_flags, uint32_t score_flags,
                     int window, int q_offset, const int32_t *doc_ids,
                     const int32_t *prefix_len, const double *alibi_slopes,
                     double softcap, const int64_t *rows, int64_t n_rows,
                     double *out, double *lse, double *probs)
{
    if (B <= 0 || H <= 0 || H_kv <= 0 || S_q <= 0 || S_k <= 0 || D <= 0)
        return -1;
    if (H % H_kv != 0)
        return -1;
    if ((mask_flags & OR_MASK_DOCUMENT) && (doc_ids == NULL || S_q != S_k))
        return -1;
    if ((mask_flags & OR_MASK_PREFIX_LM) && prefix_len == NULL)
        return -1;
    if ((score_flags & OR_SCORE_SOFTCAP) && !(softcap > 0.0))
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
                double slope = 0.0;
                if (score_flags & OR_SCORE_ALIBI)
                    slope = alibi_slopes ? alibi_slopes[h]
                                         : pow(2.0, -8.0 * (double)(h + 1) / (double)H);
                double qpos = (double)(i + q_offset);

                /* scores of every key, then the mods, then the mask */
                double M = -INFINITY;
                for (int64_t j = 0; j < S_k; ++j) {
                    const uint16_t *kp = kb + j * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += qrow[d] * bf16_to_double(kp[d]);
                    double sj = scale * dot;
                    if (score_flags & OR_SCORE_ALIBI)
                        sj += -slope * (qpos - (double)j);
                    if (score_flags & OR_SCORE_SOFTCAP)
                        sj = softcap * tanh(sj / softcap);
                    s[j] = sj;
                    vis[j] = (unsigned char)visible(i, j, b, S_k, mask_flags, window,
                                                    q_offset, doc_ids, prefix_len);
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
