/*
 * carat_oracle.c -- plain fp64 CPU oracle for sliding-window ring attention
 * and grouped global speculative-verify attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or table with the CUDA path.
 *
 * What it computes, and where that is stated:
 *
 *  - Ring slot of a token: its absolute position modulo the window size
 *    ("Announcing Carat: An inference engine designed for Gemma 4",
 *    section "Replacing page lookups with a ring buffer").  A new token
 *    reuses the slot of the token one window older (same section), and the
 *    K and V rings are written in lockstep so they share one cyclic offset
 *    ("Improving Decode Throughput on Intel Gaudi 3", section "Our approach").
 *
 *  - Sliding-window attention: each query attends to the most recent 1024
 *    positions, its own included ("Improving Decode Throughput on Intel
 *    Gaudi 3", section "Patching sliding window KV allocation": a sliding
 *    layer needs KV only for a 1024-token window).  The oracle never touches a
 *    ring: it reads an explicitly materialised LINEAR history, which is what
 *    the ring must be equivalent to because attention does not depend on a
 *    common reordering of K and V (Gaudi page, "Our approach").
 *
 *  - Global verify attention: key_count = context_length + proposal_count,
 *    QK^T, a causal softmax in which no query looks at a key later than
 *    itself, then PV ("Announcing Carat ...", section "More FLOPs can be
 *    faster", the qk_matmul / causal_softmax / pv_matmul sequence).  Query j
 *    of a request sits at position context_length + j.
 *
 *  - Grouped-query attention: the query heads that share one KV head
 *    ("Announcing Carat ...", section "Doing it all in one kernel can be
 *    slower"); query head h reads KV head h / (Hq / Hkv).
 *
 * Arithmetic: every bf16 input is widened exactly to double; dot products,
 * the maximum, exp and the weighted sum are all double, in the plain order
 * of the definition (no blocking, no online rescaling).  Softmax is written
 * with the maximum subtracted first, which is the same value as the textbook
 * definition exp(s_t) / sum exp(s_u), only without overflow.
 *
 * Storage conventions (all row-major, bf16 as raw uint16 bit patterns):
 *   q        [proposal_count][q_heads][head_dim]
 *   history  [hist_len][kv_heads][head_dim], row i holds position hist_base+i
 *   out      [proposal_count][q_heads][head_dim], double
 *
 * Return codes: 0 = success, -1 = a needed position is not in the supplied
 * history, -2 = bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
static double bf16_value(uint16_t bits)
{
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* Slot that holds absolute position `position` in a ring of `window` slots. */
int64_t oracle_ring_slot(int64_t position, int64_t window)
{
    return position % window;
}

/* key_count = context_length + proposal_count (Carat, "More FLOPs can be faster"). */
int64_t oracle_key_count(int64_t context_length, int64_t proposal_count)
{
    return context_length + proposal_count;
}

/* First position a query at `position` may attend to.
 * window <= 0 means global attention (every earlier position). */
int64_t oracle_window_first(int64_t position, int64_t window)
{
    if (window <= 0)
        return 0;
    int64_t first = position - window + 1;
    return first > 0 ? first : 0;
}

/*
 * One output row: softmax over keys t in [first, position] of
 * scale * <q, K[t]>, applied to V[t].  K and V are read for KV head `kv_head`.
 */
int oracle_attention_row(double *out_row, const uint16_t *q_row,
                         const uint16_t *k_hist, const uint16_t *v_hist,
                         int64_t hist_base, int64_t hist_len,
                         int kv_heads, int head_dim, int kv_head,
                         int64_t position, int64_t window, double scale)
{
    if (head_dim <= 0 || kv_heads <= 0 || kv_head < 0 || kv_head >= kv_heads || position < 0)
        return -2;
    int64_t first = oracle_window_first(position, window);
    int64_t last = position;
    if (first < hist_base || last >= hist_base + hist_len)
        return -1;

    int64_t n = last - first + 1;
    double *score = (double *)malloc((size_t)n * sizeof(double));
    if (!score)
        return -2;

    /* scores s_t = scale * sum_d q[d] * K[t][d] */
    for (int64_t t = first; t <= last; ++t) {
        const uint16_t *k_row = k_hist + ((t - hist_base) * kv_heads + kv_head) * (int64_t)head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_value(q_row[d]) * bf16_value(k_row[d]);
        score[t - first] = scale * dot;
    }

    /* softmax weights w_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u) */
    double max_score = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (score[i] > max_score)
            max_score = score[i];

    double denom = 0.0;
    for (int d = 0; d < head_dim; ++d)
        out_row[d] = 0.0;
    for (int64_t t = first; t <= last; ++t) {
        double w = exp(score[t - first] - max_score);
        denom += w;
        const uint16_t *v_row = v_hist + ((t - hist_base) * kv_heads + kv_head) * (int64_t)head_dim;
        for (int d = 0; d < head_dim; ++d)
            out_row[d] += w * bf16_value(v_row[d]);
    }
    for (int d = 0; d < head_dim; ++d)
        out_row[d] /= denom;

    free(score);
    return 0;
}

/*
 * All rows of one request: proposal_count query positions x q_heads heads.
 * Query j sits at position context_length + j; query head h reads KV head
 * h / (q_heads / kv_heads).  window <= 0: global attention.
 */
int oracle_attention_request(double *out, const uint16_t *q,
                             const uint16_t *k_hist, const uint16_t *v_hist,
                             int64_t hist_base, int64_t hist_len,
                             int64_t context_length, int proposal_count,
                             int q_heads, int kv_heads, int head_dim,
                             int64_t window, double scale)
{
    if (proposal_count <= 0 || q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads != 0 ||
        context_length < 0)
        return -2;
    int group = q_heads / kv_heads;
    for (int j = 0; j < proposal_count; ++j) {
        int64_t position = context_length + j;
        for (int h = 0; h < q_heads; ++h) {
            int64_t row = (int64_t)j * q_heads + h;
            int rc = oracle_attention_row(out + row * head_dim, q + row * head_dim,
                                          k_hist, v_hist, hist_base, hist_len,
                                          kv_heads, head_dim, h / group,
                                          position, window, scale);
            if (rc != 0)
                return rc;
        }
    }
    return 0;
}

/*
 * Expected ring contents after the tokens at positions [0, key_count) have
 * been appended in order: the slot of each position is overwritten by every
 * later position with the same slot, so slot s ends up holding the LAST
 * position t < key_count with t mod window == s.  Written for every t in
 * [max(0, key_count - window), key_count); slot_valid[s] = 1 for those slots
 * and is left untouched for the others (a ring that has not wrapped yet).
 * ring: [window][kv_heads][head_dim] bf16 bits.
 */
int oracle_ring_expected(uint16_t *ring, uint8_t *slot_valid,
                         const uint16_t *hist, int64_t hist_base, int64_t hist_len,
                         int64_t key_count, int64_t window, int kv_heads, int head_dim)
{
    if (window <= 0 || key_count < 0)
        return -2;
    int64_t row_elems = (int64_t)kv_heads * head_dim;
    int64_t first = key_count - window > 0 ? key_count - window : 0;
    if (key_count > 0 && (first < hist_base || key_count - 1 >= hist_base + hist_len))
        return -1;
    for (int64_t t = first; t < key_count; ++t) {
        int64_t s = oracle_ring_slot(t, window);
        memcpy(ring + s * row_elems, hist + (t - hist_base) * row_elems,
               (size_t)row_elems * sizeof(uint16_t));
        slot_valid[s] = 1;
    }
    return 0;
}

/*
 * Rows that appending proposal_count tokens at positions
 * [context_length, context_length + proposal_count) overwrites in a ring of
 * `window` slots while a query of the same step still attends to them.
 * Query 0 sees [context_length - window + 1, context_length]; new token j
 * (j >= 1) lands on the slot of position context_length + j - window, which
 * lies inside that range.  Entry i (i = 0 .. proposal_count-2) is position
 * context_length - window + 1 + i; entries whose position is negative never
 * held a token and are flagged 0 in `row_valid`.
 * displaced: [proposal_count-1][2][kv_heads][head_dim] (K then V).
 */
int oracle_displaced_expected(uint16_t *displaced, uint8_t *row_valid,
                              const uint16_t *k_hist, const uint16_t *v_hist,
                              int64_t hist_base, int64_t hist_len,
                              int64_t context_length, int proposal_count,
                              int64_t window, int kv_heads, int head_dim)
{
    if (proposal_count < 1 || window <= 0)
        return -2;
    int64_t row_elems = (int64_t)kv_heads * head_dim;
    for (int i = 0; i < proposal_count - 1; ++i) {
        int64_t t = context_length - window + 1 + i;
        uint16_t *dst = displaced + (int64_t)i * 2 * row_elems;
        if (t < 0) {
            row_valid[i] = 0;
            continue;
        }
        if (t < hist_base || t >= hist_base + hist_len)
            return -1;
        memcpy(dst, k_hist + (t - hist_base) * row_elems, (size_t)row_elems * sizeof(uint16_t));
        memcpy(dst + row_elems, v_hist + (t - hist_base) * row_elems,
               (size_t)row_elems * sizeof(uint16_t));
        row_valid[i] = 1;
    }
    return 0;
}
