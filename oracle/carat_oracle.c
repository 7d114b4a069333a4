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
 *  - FP8 KV cache: the cache holds e4m3 codes ("gemma-cuda-hybrid",
 *    "Features" / "Server": FP8 e4m3 KV; "Limitations": lossy), here with one dequantisation
 *    scale per tensor; the attention of such a cache is the attention of its
 *    dequantised values (oracle_attention_request_f64).
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

/* Element i of a K or V history: bf16 bits (kind 0) or float64 (kind 1). */
static double hist_value(const void *hist, int64_t i, int kind)
{
    if (kind == 0)
        return bf16_value(((const uint16_t *)hist)[i]);
    return ((const double *)hist)[i];
}

/*
 * One output row: softmax over keys t in [first, position] of
 * scale * <q, K[t]>, applied to V[t].  K and V are read for KV head `kv_head`.
 */
static int attention_row(double *out_row, const uint16_t *q_row,
                         const void *k_hist, const void *v_hist, int kind,
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
        int64_t k_row = ((t - hist_base) * kv_heads + kv_head) * (int64_t)head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_value(q_row[d]) * hist_value(k_hist, k_row + d, kind);
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
        int64_t v_row = ((t - hist_base) * kv_heads + kv_head) * (int64_t)head_dim;
        for (int d = 0; d < head_dim; ++d)
            out_row[d] += w * hist_value(v_hist, v_row + d, kind);
    }
    for (int d = 0; d < head_dim; ++d)
        out_row[d] /= denom;

    free(score);
    return 0;
}

int oracle_attention_row(double *out_row, const uint16_t *q_row,
                         const uint16_t *k_hist, const uint16_t *v_hist,
                         int64_t hist_base, int64_t hist_len,
                         int kv_heads, int head_dim, int kv_head,
                         int64_t position, int64_t window, double scale)
{
    return attention_row(out_row, q_row, k_hist, v_hist, 0, hist_base, hist_len, kv_heads,
                         head_dim, kv_head, position, window, scale);
}

/*
 * All rows of one request: proposal_count query positions x q_heads heads.
 * Query j sits at position context_length + j; query head h reads KV head
 * h / (q_heads / kv_heads).  window <= 0: global attention.
 */
static int attention_request(double *out, const uint16_t *q,
                             const void *k_hist, const void *v_hist, int kind,
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
            int rc = attention_row(out + row * head_dim, q + row * head_dim,
                                   k_hist, v_hist, kind, hist_base, hist_len,
                                   kv_heads, head_dim, h / group,
                                   position, window, scale);
            if (rc != 0)
                return rc;
        }
    }
    return 0;
}

int oracle_attention_request(double *out, const uint16_t *q,
                             const uint16_t *k_hist, const uint16_t *v_hist,
                             int64_t hist_base, int64_t hist_len,
                             int64_t context_length, int proposal_count,
                             int q_heads, int kv_heads, int head_dim,
                             int64_t window, double scale)
{
    return attention_request(out, q, k_hist, v_hist, 0, hist_base, hist_len, context_length,
                             proposal_count, q_heads, kv_heads, head_dim, window, scale);
}

/* The same with K and V histories given as float64 values (a dequantised
 * FP8 cache: every element is its e4m3 value times the tensor's scale). */
int oracle_attention_request_f64(double *out, const uint16_t *q,
                                 const double *k_hist, const double *v_hist,
                                 int64_t hist_base, int64_t hist_len,
                                 int64_t context_length, int proposal_count,
                                 int q_heads, int kv_heads, int head_dim,
                                 int64_t window, double scale)
{
    return attention_request(out, q, k_hist, v_hist, 1, hist_base, hist_len, context_length,
                             proposal_count, q_heads, kv_heads, head_dim, window, scale);
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

/*
 * FP8 e4m3 (the KV-cache format of "gemma-cuda-hybrid", "Features" /
 * "Server": the cache is stored in e4m3; "Limitations": it is lossy).  The format: 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; there is no
 * infinity; S.1111.111 is NaN, so the largest finite value is
 * S.1111.110 = 1.75 * 2^8 = 448.
 */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xf;
    int m = code & 0x7;
    if (e == 0xf && m == 0x7)
        return NAN;
    double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/*
 * Nearest e4m3 value to x, ties to the even code (mantissa LSB 0), and
 * magnitudes beyond 448 clamped to 448 (saturating conversion).  Written as
 * a search over the 127 non-negative finite codes, which are increasing in
 * value, so the rounding rule can be checked by eye.
 */
uint8_t oracle_e4m3_encode(double x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7e;
    /* largest code whose value is <= a */
    int lo = 0;
    for (int c = 0; c <= 0x7e; ++c)
        if (oracle_e4m3_decode((uint8_t)c) <= a)
            lo = c;
    if (oracle_e4m3_decode((uint8_t)lo) == a)
        return sign | (uint8_t)lo;
    int hi = lo + 1;
    double dlo = a - oracle_e4m3_decode((uint8_t)lo);
    double dhi = oracle_e4m3_decode((uint8_t)hi) - a;
    int c;
    if (dlo < dhi)
        c = lo;
    else if (dhi < dlo)
        c = hi;
    else
        c = (lo & 1) == 0 ? lo : hi;
    return sign | (uint8_t)c;
}

/*
 * Quantise n bf16 values for an FP8 cache with dequantisation scale `scale`
 * (value = e4m3 * scale).  Reading taken where the pages are silent: one
 * scale per tensor (K, V), and each element is mapped as
 * e4m3_rn(fp32(x * fp32(1 / scale))) -- the reciprocal and the product each
 * rounded once to binary32, then one rounding to e4m3 with saturation.
 */
void oracle_quantize_bf16(uint8_t *dst, const uint16_t *src, int64_t n, float scale)
{
    float inv = 1.0f / scale;
    for (int64_t i = 0; i < n; ++i) {
        float prod = (float)(bf16_value(src[i]) * (double)inv); /* exact, then one rounding */
        dst[i] = oracle_e4m3_encode((double)prod);
    }
}

/* oracle_ring_expected for rows of `row_bytes` bytes (an FP8 ring). */
int oracle_ring_expected_bytes(uint8_t *ring, uint8_t *slot_valid, const uint8_t *hist,
                               int64_t hist_base, int64_t hist_len, int64_t key_count,
                               int64_t window, int64_t row_bytes)
{
    if (window <= 0 || key_count < 0 || row_bytes <= 0)
        return -2;
    int64_t first = key_count - window > 0 ? key_count - window : 0;
    if (key_count > 0 && (first < hist_base || key_count - 1 >= hist_base + hist_len))
        return -1;
    for (int64_t t = first; t < key_count; ++t) {
        int64_t s = oracle_ring_slot(t, window);
        memcpy(ring + s * row_bytes, hist + (t - hist_base) * row_bytes, (size_t)row_bytes);
        slot_valid[s] = 1;
    }
    return 0;
}

/* oracle_displaced_expected for rows of `row_bytes` bytes (an FP8 ring). */
int oracle_displaced_expected_bytes(uint8_t *displaced, uint8_t *row_valid,
                                    const uint8_t *k_hist, const uint8_t *v_hist,
                                    int64_t hist_base, int64_t hist_len, int64_t context_length,
                                    int proposal_count, int64_t window, int64_t row_bytes)
{
    if (proposal_count < 1 || window <= 0 || row_bytes <= 0)
        return -2;
    for (int i = 0; i < proposal_count - 1; ++i) {
        int64_t t = context_length - window + 1 + i;
        uint8_t *dst = displaced + (int64_t)i * 2 * row_bytes;
        if (t < 0) {
            row_valid[i] = 0;
            continue;
        }
        if (t < hist_base || t >= hist_base + hist_len)
            return -1;
        memcpy(dst, k_hist + (t - hist_base) * row_bytes, (size_t)row_bytes);
        memcpy(dst + row_bytes, v_hist + (t - hist_base) * row_bytes, (size_t)row_bytes);
        row_valid[i] = 1;
    }
    return 0;
}
