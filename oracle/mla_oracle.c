/*
 * mla_oracle.c -- fp64 CPU oracle for absorbed-MLA decode over a paged fp8 pool.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file: it exists so that tests, the smoke check and the
 * benchmark's CPU-baseline leg can compare the CUDA kernels against a plain,
 * slow, obviously correct definition.  It shares no code, header, table or
 * constant with the CUDA sources.
 *
 * What it computes (plain definition; the split kernels reach the same result
 * by a different route):
 *
 *   moonmath-ai/amd-kernels README, "MLA absorbed decode" and "Use / MLA decode":
 *   one fused fp8 row per token is both K (all d_v + d_rope columns) and V (the
 *   first d_v columns); a single per-tensor kv_scale dequantizes both parts; the
 *   queries are split into a latent part q_lat [.., H, d_v] and a RoPE part
 *   q_pe [.., H, d_rope]; the pool is paged with page_size 1, so kv_indices is a
 *   flat per-token slot list (any permutation or subset is legal); for q_len > 1
 *   draft position t attends KV [0, S - q_len + t] (read inclusive).
 *
 *   For one query row and head:
 *     k_j[c] = e4m3fn(pool[slot_j][c]) * kv_scale                (fp64)
 *     s_j    = scale * (sum_{c<d_v} q_lat[c] k_j[c] + sum_{c<d_rope} q_pe[c] k_j[d_v+c])
 *     M      = max_j s_j
 *     o[c]   = sum_j exp(s_j - M) k_j[c] / sum_j exp(s_j - M)     (c < d_v)
 *     lse2   = (M + ln sum_j exp(s_j - M)) / ln 2                  (base-2 LSE,
 *              README "MLA absorbed decode": the op returns a base-2 LSE)
 *   A row that sees no key has o = 0 and lse2 = -inf.
 *
 *   Split-K merge of per-split partials (o_s normalized, lse2_s base 2), as in
 *   hip_mha_decoding_num_partitions (split-K target merged by the reducer):
 *     M = max_s lse2_s;  w_s = 2^(lse2_s - M);
 *     o = out_scale * sum_s w_s o_s / sum_s w_s;  lse2 = M + log2 sum_s w_s.
 *
 *   Decode context parallelism (README, "MLA absorbed decode" and "Use / MLA
 *   decode", DCP): rank cp_rank of cp_world holds the positions p of every
 *   request with p % cp_world == cp_rank, in increasing order, so its local key
 *   i is the global position i * cp_world + cp_rank; seq_lens counts the rank's
 *   keys and glen gives the global lengths.  Draft row t of request b sees the
 *   global positions p <= glen[b] - q_len + t.  The rank returns o and the
 *   base-2 LSE of its share; the ranks' results combine by the split-K merge
 *   above with out_scale 1, the ranks playing the part of the splits.
 *
 *   Sparse variant ("[Perf] pa_decode_sparse ..." issue, "Measurements"): the
 *   same per-row definition with 448 NoPE + 64 RoPE columns, the key list being
 *   the token's row of the top-k index table; a negative index is an invalid
 *   entry and is skipped (has_invalid).
 *
 * Decoding follows the OCP 8-bit floating point specification for E4M3:
 * 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 encodes
 * the subnormals m * 2^-9; S.1111.111 is NaN; there are no infinities.
 * bf16 is the top half of an IEEE binary32.
 *
 * Return codes: 0 ok, -1 bad argument, -2 slot out of range, -3 NaN input.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_SLOT (-2)
#define ORACLE_NAN (-3)

/* ---- number formats ------------------------------------------------------ */

double oracle_e4m3fn_to_double(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int expo = (b >> 3) & 0xF;
    int mant = b & 0x7;
    double v;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    if (expo == 0)
        v = ldexp((double)mant, -9);                 /* 0.mmm * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -v : v;
}

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* 256-entry decode table, filled from oracle_e4m3fn_to_double on first use. */
static double g_e4m3[256];
static int g_e4m3_ready = 0;

static void e4m3_table_init(void)
{
    if (g_e4m3_ready)
        return;
    for (int i = 0; i < 256; ++i)
        g_e4m3[i] = oracle_e4m3fn_to_double((uint8_t)i);
    g_e4m3_ready = 1;
}

/* ---- one query row against a list of slots ------------------------------- */

/*
 * q_lat: bf16 [d_v], q_pe: bf16 [d_rope]; pool rows are d_v + d_rope bytes.
 * Slots < 0 are skipped.  o: [d_v] (fp64), lse2: base-2 LSE.
 */
static int attend_row(const uint16_t* q_lat, const uint16_t* q_pe, int d_v, int d_rope,
                      const uint8_t* pool, int64_t pool_rows,
                      const int32_t* slots, int64_t n, double scale, double kv_scale,
                      double* o, double* lse2)
{
    const int64_t width = (int64_t)d_v + d_rope;
    double* q = (double*)malloc(sizeof(double) * (size_t)width);
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    int rc = ORACLE_OK;
    if (!q || !s) {
        free(q);
        free(s);
        return ORACLE_BAD_ARG;
    }
    for (int c = 0; c < d_v; ++c)
        q[c] = oracle_bf16_to_double(q_lat[c]);
    for (int c = 0; c < d_rope; ++c)
        q[d_v + c] = oracle_bf16_to_double(q_pe[c]);
    for (int64_t c = 0; c < width; ++c)
        if (isnan(q[c])) rc = ORACLE_NAN;

    /* logits */
    double m = -INFINITY;
    int64_t valid = 0;
    for (int64_t j = 0; j < n && rc == ORACLE_OK; ++j) {
        int32_t slot = slots[j];
        if (slot < 0)
            continue;
        if ((int64_t)slot >= pool_rows) {
            rc = ORACLE_BAD_SLOT;
            break;
        }
        const uint8_t* row = pool + (int64_t)slot * width;
        double dot = 0.0;
        for (int64_t c = 0; c < width; ++c) {
            double k = g_e4m3[row[c]] * kv_scale;
            if (isnan(k)) {
                rc = ORACLE_NAN;
                break;
            }
            dot += q[c] * k;
        }
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
        ++valid;
    }

    for (int c = 0; c < d_v; ++c)
        o[c] = 0.0;
    if (rc != ORACLE_OK || valid == 0) {
        *lse2 = -INFINITY;
        free(q);
        free(s);
        return rc;
    }

    /* softmax-weighted sum of the V rows (first d_v columns of each row) */
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        int32_t slot = slots[j];
        if (slot < 0)
            continue;
        const uint8_t* row = pool + (int64_t)slot * width;
        double w = exp(s[j] - m);
        z += w;
        for (int c = 0; c < d_v; ++c)
            o[c] += w * (g_e4m3[row[c]] * kv_scale);
    }
    for (int c = 0; c < d_v; ++c)
        o[c] /= z;
    *lse2 = (m + log(z)) / log(2.0);
    free(q);
    free(s);
    return ORACLE_OK;
}

/* ---- exported entry points ----------------------------------------------- */

/* One row: the definition above on an explicit slot list. */
int oracle_attend(const uint16_t* q_lat, const uint16_t* q_pe, int d_v, int d_rope,
                  const uint8_t* pool, int64_t pool_rows,
                  const int32_t* slots, int64_t n, double scale, double kv_scale,
                  double* o, double* lse2)
{
    if (!q_lat || !pool || !o || !lse2 || d_v <= 0 || d_rope < 0 || n < 0)
        return ORACLE_BAD_ARG;
    if (d_rope > 0 && !q_pe)
        return ORACLE_BAD_ARG;
    e4m3_table_init();
    return attend_row(q_lat, q_pe, d_v, d_rope, pool, pool_rows, slots, n,
                      scale, kv_scale, o, lse2);
}

/* Split-K merge of ns partials (o_parts [ns, d_v], lse2_parts [ns]). */
int oracle_merge(const double* o_parts, const double* lse2_parts, int ns, int d_v,
                 double out_scale, double* o, double* lse2)
{
    if (!o_parts || !lse2_parts || !o || !lse2 || ns <= 0 || d_v <= 0)
        return ORACLE_BAD_ARG;
    double m = -INFINITY;
    for (int s = 0; s < ns; ++s)
        if (lse2_parts[s] > m)
            m = lse2_parts[s];
    for (int c = 0; c < d_v; ++c)
        o[c] = 0.0;
    if (m == -INFINITY) {
        *lse2 = -INFINITY;
        return ORACLE_OK;
    }
    double wsum = 0.0;
    for (int s = 0; s < ns; ++s) {
        if (lse2_parts[s] == -INFINITY)
            continue;
        double w = exp2(lse2_parts[s] - m);
        wsum += w;
        for (int c = 0; c < d_v; ++c)
            o[c] += w * o_parts[(int64_t)s * d_v + c];
    }
    for (int c = 0; c < d_v; ++c)
        o[c] = out_scale * o[c] / wsum;
    *lse2 = m + log2(wsum);
    return ORACLE_OK;
}

/*
 * Dense decode.  Rows r = b*q_len + t; the item index is r*H + h.  If sel is
 * non-NULL only the n_sel listed items are computed and o/lse2 are packed
 * [n_sel, d_v] / [n_sel]; otherwise every item is computed, o [R*H, d_v].
 * Request b's keys are kv_indices[kv_indptr[b] + j] for
 * j < seq_lens[b] - q_len + t + 1.
 */
int oracle_dense_decode(int32_t batch, int32_t q_len, int32_t num_heads,
                        int32_t d_v, int32_t d_rope,
                        const uint16_t* q_lat, const uint16_t* q_pe,
                        const uint8_t* pool, int64_t pool_rows,
                        const int32_t* seq_lens, const int32_t* kv_indices,
                        const int32_t* kv_indptr, double scale, double kv_scale,
                        const int64_t* sel, int64_t n_sel, double* o, double* lse2)
{
    if (batch < 0 || q_len <= 0 || num_heads <= 0 || d_v <= 0 || d_rope < 0)
        return ORACLE_BAD_ARG;
    if (!q_lat || (d_rope > 0 && !q_pe) || !pool || !seq_lens || !kv_indices ||
        !kv_indptr || !o || !lse2)
        return ORACLE_BAD_ARG;
    for (int32_t b = 0; b < batch; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > kv_indptr[b + 1] - kv_indptr[b])
            return ORACLE_BAD_ARG;
    e4m3_table_init();
    const int64_t items = sel ? n_sel : (int64_t)batch * q_len * num_heads;
    int rc = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < items; ++i) {
        int64_t item = sel ? sel[i] : i;
        int64_t r = item / num_heads;
        int64_t h = item % num_heads;
        int64_t b = r / q_len;
        int64_t t = r % q_len;
        int local;
        if (item < 0 || b >= batch) {
            local = ORACLE_BAD_ARG;
        } else {
            int64_t n = (int64_t)seq_lens[b] - q_len + t + 1;
            if (n < 0)
                n = 0;
            local = attend_row(q_lat + (r * num_heads + h) * d_v,
                               q_pe + (r * num_heads + h) * d_rope, d_v, d_rope,
                               pool, pool_rows, kv_indices + kv_indptr[b], n,
                               scale, kv_scale, o + i * d_v, lse2 + i);
        }
        if (local != ORACLE_OK) {
#pragma omp critical
            rc = local;
        }
    }
    return rc;
}

/*
 * One DCP rank's dense decode (same layouts as oracle_dense_decode; glen
 * [batch] global lengths).  Row t of request b attends its local keys
 * j < seq_lens[b] whose global position j*cp_world + cp_rank is at most
 * glen[b] - q_len + t; positions grow with j, so these are a prefix.
 */
int oracle_dcp_decode(int32_t batch, int32_t q_len, int32_t num_heads,
                      int32_t d_v, int32_t d_rope,
                      const uint16_t* q_lat, const uint16_t* q_pe,
                      const uint8_t* pool, int64_t pool_rows,
                      const int32_t* seq_lens, const int32_t* kv_indices,
                      const int32_t* kv_indptr, const int32_t* glen,
                      int32_t cp_rank, int32_t cp_world, double scale, double kv_scale,
                      double* o, double* lse2)
{
    if (batch < 0 || q_len <= 0 || num_heads <= 0 || d_v <= 0 || d_rope < 0 ||
        cp_world < 1 || cp_rank < 0 || cp_rank >= cp_world)
        return ORACLE_BAD_ARG;
    if (!q_lat || (d_rope > 0 && !q_pe) || !pool || !seq_lens || !kv_indices ||
        !kv_indptr || !glen || !o || !lse2)
        return ORACLE_BAD_ARG;
    for (int32_t b = 0; b < batch; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > kv_indptr[b + 1] - kv_indptr[b])
            return ORACLE_BAD_ARG;
    e4m3_table_init();
    const int64_t items = (int64_t)batch * q_len * num_heads;
    int rc = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < items; ++i) {
        int64_t r = i / num_heads;
        int64_t b = r / q_len;
        int64_t t = r % q_len;
        int64_t last = (int64_t)glen[b] - q_len + t;   /* last visible global position */
        int64_t n = 0;
        while (n < seq_lens[b] && n * cp_world + cp_rank <= last)
            ++n;
        /* item i is row r = i / num_heads, head h = i % num_heads */
        int local = attend_row(q_lat + i * d_v, q_pe + i * d_rope, d_v, d_rope,
                               pool, pool_rows, kv_indices + kv_indptr[b], n,
                               scale, kv_scale, o + i * d_v, lse2 + i);
        if (local != ORACLE_OK) {
#pragma omp critical
            rc = local;
        }
    }
    return rc;
}

/*
 * Sparse top-k decode: token t, head h (item t*H + h) attends the slots
 * indices[t*topk .. t*topk + topk), skipping negative entries.
 */
int oracle_sparse_decode(int32_t num_tokens, int32_t num_heads, int32_t topk,
                         int32_t d_v, int32_t d_rope,
                         const uint16_t* q_nope, const uint16_t* q_pe,
                         const uint8_t* pool, int64_t pool_rows, const int32_t* indices,
                         double scale, double kv_scale,
                         const int64_t* sel, int64_t n_sel, double* o, double* lse2)
{
    if (num_tokens < 0 || num_heads <= 0 || topk < 0 || d_v <= 0 || d_rope < 0)
        return ORACLE_BAD_ARG;
    if (!q_nope || (d_rope > 0 && !q_pe) || !pool || !indices || !o || !lse2)
        return ORACLE_BAD_ARG;
    e4m3_table_init();
    const int64_t items = sel ? n_sel : (int64_t)num_tokens * num_heads;
    int rc = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < items; ++i) {
        int64_t item = sel ? sel[i] : i;
        int64_t t = item / num_heads;
        int local;
        if (item < 0 || t >= num_tokens) {
            local = ORACLE_BAD_ARG;
        } else {
            local = attend_row(q_nope + item * d_v, q_pe + item * d_rope, d_v, d_rope,
                               pool, pool_rows, indices + t * topk, topk,
                               scale, kv_scale, o + i * d_v, lse2 + i);
        }
        if (local != ORACLE_OK) {
#pragma omp critical
            rc = local;
        }
    }
    return rc;
}
