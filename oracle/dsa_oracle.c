/*
 * dsa_oracle.c -- plain float64 CPU oracle for the DSA indexer -> top-k ->
 * sparse absorbed-MLA attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call
 * this file; only the test suite, the package entry point's smoke check and
 * the benchmark's CPU-baseline leg use it.  It shares no code, header, table
 * or helper with the CUDA library.
 *
 * Every function is the definition written out: no blocking, no fusion, no
 * reordering beyond what the definition states.  Each call handles a range of
 * rows [row_begin, row_end) so a caller may spread rows over threads; the code
 * for one row is single-threaded and deterministic.
 *
 * Inputs are the raw bf16 bit patterns (uint16) the GPU path reads; each is
 * widened exactly to double.  Sources followed:
 *   - exo PR #2539 (GLM-5.2/5.3 glm_moe_dsa attention), section "Prefill",
 *     bullet "Indexer scores in float32, in one kernel": score = sum over the
 *     32 indexer heads of relu(q_h . k) times the head weight, mask applied.
 *   - same page, section "Prefill", bullets "The first 2048 queries attend
 *     causally" and "Sparse attention from 8192 keys": each query keeps its
 *     2048 best keys; a query before position 2048 keeps every earlier key.
 *   - SlimServe "GLM52_PIPELINE_TRACE.md", section 6 "Attention core
 *     (absorbed MLA)": Q = [q_nope.wk_b (512) | q_pe (64)], K = [kv_cmpr |
 *     k_pe], V = kv_cmpr; kq = K.Q, softmax with kq_scale, kqv = V.softmax.
 *   - same page, Config line: qk_nope 192 + qk_rope 64 give the softmax scale
 *     1/sqrt(256) (passed in as `scale`).
 * Readings where the pages are silent (tie rule, masked value, output order,
 * empty selections) are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Indexer scores.
 *   S[r, j] = sum_{h < Hi} w[r, h] * max(0, sum_{d < Di} qI[r, h, d] * kI[b, j, d])
 * for keys j <= min(p_r, kv_len[b] - 1), where row r = b * L + i sits at
 * position p_r = q_pos0[b] + i.  Every other key j < Nmax is masked and holds
 * -inf (reading: "with the mask applied" -- a masked key is never selectable).
 * No extra scale is applied: any 1/sqrt constant is taken as folded into w.
 *   qI [B, L, Hi, Di], kI [B, Nmax, Di], w [B, L, Hi] (indexed by absolute row);
 *   S [row_end - row_begin, Nmax]: S[0] is the output of row row_begin.
 */
void oracle_indexer(const uint16_t *qI, const uint16_t *kI, const float *w,
                    const int32_t *q_pos0, const int32_t *kv_len,
                    int B, int L, int Nmax, int Hi, int Di,
                    int row_begin, int row_end, double *S)
{
    (void)B;
    for (int r = row_begin; r < row_end; ++r) {
        int b = r / L, i = r % L;
        long p = (long)q_pos0[b] + i;
        long last = p < (long)kv_len[b] - 1 ? p : (long)kv_len[b] - 1;
        const uint16_t *q = qI + (size_t)r * Hi * Di;
        const float *wr = w + (size_t)r * Hi;
        double *srow = S + (size_t)(r - row_begin) * Nmax;
        for (int j = 0; j < Nmax; ++j) {
            if ((long)j > last) {
                srow[j] = -INFINITY;
                continue;
            }
            const uint16_t *k = kI + ((size_t)b * Nmax + j) * Di;
            double acc = 0.0;
            for (int h = 0; h < Hi; ++h) {
                double dot = 0.0;
                for (int d = 0; d < Di; ++d)
                    dot += bf16_to_double(q[(size_t)h * Di + d]) * bf16_to_double(k[d]);
                double relu = dot > 0.0 ? dot : 0.0;
                acc += (double)wr[h] * relu;
            }
            srow[j] = acc;
        }
    }
}

/* ordering for selection: larger score first, then lower key index */
typedef struct {
    float s;
    int32_t j;
} cand_t;

static int cmp_score_desc_index_asc(const void *a, const void *b)
{
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;          /* -0.0 and +0.0 compare equal here */
    return (x->j > y->j) - (x->j < y->j);
}

static int cmp_int_asc(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * Top-k selection on float32 scores (the pages fix float32 for the indexer sum,
 * so the selection is decided on float32 values).
 *   n = number of causal keys = min(p_r + 1, kv_len[b]).
 *   n <= K : idx = 0, 1, ..., n-1 followed by K - n entries of -1
 *            (a query before position K keeps every earlier key).
 *   n >  K : the K keys j < n with the largest S[r, j]; equal scores are
 *            ordered by the lower key index (tie rule: lower index wins);
 *            -0.0 equals +0.0.  The chosen indices are written ascending.
 * S is [row_end - row_begin, ld] and idx is [row_end - row_begin, K]: their
 * first row belongs to query row row_begin.
 */
void oracle_topk(const float *S, int64_t ld, const int32_t *q_pos0, const int32_t *kv_len,
                 int B, int L, int K, int row_begin, int row_end, int32_t *idx)
{
    (void)B;
    for (int r = row_begin; r < row_end; ++r) {
        int b = r / L, i = r % L;
        long p = (long)q_pos0[b] + i;
        long n = p + 1 < (long)kv_len[b] ? p + 1 : (long)kv_len[b];
        if (n < 0) n = 0;
        int32_t *out = idx + (size_t)(r - row_begin) * K;
        if (n <= K) {
            for (long t = 0; t < K; ++t) out[t] = t < n ? (int32_t)t : -1;
            continue;
        }
        cand_t *c = (cand_t *)malloc((size_t)n * sizeof *c);
        for (long j = 0; j < n; ++j) {
            c[j].s = S[(size_t)(r - row_begin) * ld + j];
            c[j].j = (int32_t)j;
        }
        qsort(c, (size_t)n, sizeof *c, cmp_score_desc_index_asc);
        for (int t = 0; t < K; ++t) out[t] = c[t].j;
        qsort(out, (size_t)K, sizeof *out, cmp_int_asc);
        free(c);
    }
}

/*
 * Sparse absorbed-MLA attention for one query row over its selected keys.
 *   For every head h and selected key t (entries idx[r, t] >= 0):
 *     s_t     = scale * sum_{d < D} q[r, h, d] * kv[b, idx_t, d]
 *     m       = max_t s_t,   e_t = exp(s_t - m)
 *     out[r,h,:] = sum_t e_t * kv[b, idx_t, 0:Dv] / sum_t e_t
 *     lse[r,h]   = m + log(sum_t e_t)          (natural log)
 * There is no softmax bias or sink.  A row that selects nothing gets a zero
 * output and lse = -inf.  row_batch[r] names the batch of each row, so one
 * routine serves prefill rows (all in batch 0) and decode rows (one per batch).
 *   q [R, H, D] and row_batch [R] are indexed by absolute row; kv [B, Nmax, D];
 *   idx [row_end - row_begin, K], out [.., H, Dv] and lse [.., H] start at row
 *   row_begin.
 */
void oracle_attn(const uint16_t *q, const uint16_t *kv, const int32_t *idx,
                 const int32_t *row_batch, int Nmax, int K, int H, int D, int Dv,
                 double scale, int row_begin, int row_end, double *out, double *lse)
{
    double *s = (double *)malloc((size_t)K * sizeof *s);
    for (int r = row_begin; r < row_end; ++r) {
        int b = row_batch[r];
        const int32_t *ir = idx + (size_t)(r - row_begin) * K;
        for (int h = 0; h < H; ++h) {
            const uint16_t *qh = q + ((size_t)r * H + h) * D;
            double *o = out + ((size_t)(r - row_begin) * H + h) * Dv;
            for (int v = 0; v < Dv; ++v) o[v] = 0.0;
            int any = 0;
            double m = -INFINITY;
            for (int t = 0; t < K; ++t) {
                if (ir[t] < 0) continue;
                const uint16_t *kr = kv + ((size_t)b * Nmax + ir[t]) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_to_double(qh[d]) * bf16_to_double(kr[d]);
                s[t] = scale * dot;
                if (!any || s[t] > m) m = s[t];
                any = 1;
            }
            if (!any) {
                lse[(size_t)(r - row_begin) * H + h] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int t = 0; t < K; ++t) {
                if (ir[t] < 0) continue;
                const uint16_t *kr = kv + ((size_t)b * Nmax + ir[t]) * D;
                double e = exp(s[t] - m);
                sum += e;
                for (int v = 0; v < Dv; ++v) o[v] += e * bf16_to_double(kr[v]);
            }
            for (int v = 0; v < Dv; ++v) o[v] /= sum;
            lse[(size_t)(r - row_begin) * H + h] = m + log(sum);
        }
    }
    free(s);
}

/*
 * Value up-projection (wv_b) of the attention output, per head.
 *   v[r, h, e] = sum_{d < Dv} o[r, h, d] * wv[h, e, d]      for e < E
 * SlimServe "GLM52_PIPELINE_TRACE.md", section 6 "Attention core (absorbed
 * MLA)": the product with wv_b decompresses each head's latent output (width
 * kv_lora_rank 512 = Dv) into its value (v_head_dim 256 = E, Config line).
 * The weight layout (one Dv-wide row per value feature, per head) is the
 * library's reading; the pages fix only the shapes.
 *   o [R, H, Dv] is indexed by absolute row; wv [H, E, Dv];
 *   v [row_end - row_begin, H, E] starts at row row_begin.
 */
void oracle_value_up_proj(const uint16_t *o, const uint16_t *wv, int H, int Dv, int E,
                          int row_begin, int row_end, double *v)
{
    for (int r = row_begin; r < row_end; ++r) {
        for (int h = 0; h < H; ++h) {
            const uint16_t *orow = o + ((size_t)r * H + h) * Dv;
            double *vr = v + ((size_t)(r - row_begin) * H + h) * E;
            for (int e = 0; e < E; ++e) {
                const uint16_t *wr = wv + ((size_t)h * E + e) * Dv;
                double acc = 0.0;
                for (int d = 0; d < Dv; ++d)
                    acc += bf16_to_double(orow[d]) * bf16_to_double(wr[d]);
                vr[e] = acc;
            }
        }
    }
}
