/*
 * gqa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement, in float64, of what the
 * GQA attention library computes.  It exists so that the CUDA path can be
 * checked against something written independently of it.  Only the tests,
 * the smoke entry point and the benchmark's CPU-baseline leg may load it;
 * the product never does.  It shares no code, header or table with the CUDA
 * sources.
 *
 * Sources restated here (page title, then the item on that page):
 *   [FA]  mlx-native 0.18.0, src/ops/flash_attn_prefill_tensor.rs --
 *         module doc (layouts, GQA grouping, additive mask shared by every
 *         head, host contract), FlashAttnPrefillTensorParams (strides in
 *         elements, pre-softmax scale).
 *   [PA]  ferrum-kernels 0.8.3, src/backend/metal/vnext_ops/causal_attention.rs
 *         -- paged_state_regions (logical KV stream cut into fixed pages in
 *         logical order), validate_signature (per-token state [2, kv_heads,
 *         head_dim]), the shape test with 4096 B per token.
 *   [DF]  mlx-native 0.21.1, src/ops/dflash2_attention_pack.rs --
 *         DFlash2AttentionPackParams, the pack / mask / commit dispatchers
 *         and the worked example in gpu_pack_mask_and_commit_match_ring_semantics.
 *
 * Every float is widened exactly to double; products and sums are double.
 * Nothing is blocked, fused or reordered beyond the definitions below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ------------------------------------------------------------------ */
/* Exact widening of 16-bit floats (IEEE 754 binary16 and bfloat16).   */
/* ------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double widen_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);             /* zero or subnormal */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25); /* (1 + f/1024) 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the top half of a binary32 pattern. */
static double widen_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

double orc_widen16(uint16_t bits, int dtype)
{
    return dtype == ORC_BF16 ? widen_bf16(bits) : widen_f16(bits);
}

/* Round a binary32 value to the nearest bfloat16, ties to even.  NaN maps
 * to a quiet NaN with the same sign.  The cast rule is the usual IEEE
 * round-to-nearest-even: the dropped 16 low bits are compared with half an
 * ulp; the carry into the exponent field produces infinity on overflow. */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
    uint32_t keep = u >> 16;
    uint32_t drop = u & 0xffffu;
    if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u)))
        keep += 1;
    return (uint16_t)keep;
}

/* float32 -> IEEE 754 binary16, round to nearest, ties to even, from the
 * format's definition: 1 sign, 5 exponent (bias 15), 10 fraction bits;
 * subnormals below 2^-14, overflow to infinity, NaN kept quiet. */
uint16_t orc_f32_to_f16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t mag = u & 0x7fffffffu;
    if (mag > 0x7f800000u)
        return (uint16_t)(sign | 0x7e00u);
    if (mag == 0x7f800000u)
        return (uint16_t)(sign | 0x7c00u);
    const int e = (int)(mag >> 23) - 127;           /* unbiased exponent */
    uint32_t m = (mag & 0x7fffffu) | (mag ? 0x800000u : 0u);  /* 24-bit significand */
    if (mag == 0)
        return (uint16_t)sign;
    /* value = m * 2^(e - 23); the f16 unit in the last place is 2^(max(e, -14) - 10) */
    const int shift = (e < -14 ? -14 : e) - 10 - (e - 23);     /* bits dropped from m */
    uint32_t q;
    if (shift >= 32) {
        q = 0;
    } else {
        q = m >> shift;
        const uint32_t rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u)))
            q += 1;
    }
    /* q counts units of 2^(max(e,-14) - 10); rebuild the bit pattern */
    int be = (e < -14 ? -14 : e);
    if (q >= 0x800u) {          /* rounding carried into the next binade */
        q >>= 1;
        be += 1;
    }
    if (q < 0x400u)             /* subnormal (be == -14) */
        return (uint16_t)(sign | q);
    if (be > 15)
        return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | ((uint32_t)(be + 15) << 10) | (q & 0x3ffu));
}

static double load_q(const void *q, int q_dtype, int64_t idx)
{
    if (q_dtype == ORC_F32)
        return (double)((const float *)q)[idx];
    return orc_widen16(((const uint16_t *)q)[idx], q_dtype);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* One query row of masked attention, straight from the definition:    */
/*   s_j = scale * <q, k_j> + mask_j                                   */
/*   o   = sum_j exp(s_j - max s) v_j / sum_j exp(s_j - max s)         */
/* A row whose every score is -inf has no visible key; its output is   */
/* defined as zero.                                                    */
/* ------------------------------------------------------------------ */
static void attention_row(const double *q, int d,
                          const uint16_t *const *krow, const uint16_t *const *vrow,
                          int kv_dtype, int n_keys,
                          const double *mask, double scale,
                          double *s, double *out)
{
    double m = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int e = 0; e < d; ++e)
            dot += q[e] * orc_widen16(krow[j][e], kv_dtype);
        s[j] = scale * dot + (mask ? mask[j] : 0.0);
        if (s[j] > m)
            m = s[j];
    }
    for (int e = 0; e < d; ++e)
        out[e] = 0.0;
    if (m == -INFINITY)
        return;
    double denom = 0.0;
    for (int j = 0; j < n_keys; ++j) {
        double p = exp(s[j] - m);
        if (p == 0.0)
            continue;
        denom += p;
        for (int e = 0; e < d; ++e)
            out[e] += p * orc_widen16(vrow[j][e], kv_dtype);
    }
    for (int e = 0; e < d; ++e)
        out[e] /= denom;
}

/*
 * Masked grouped-query attention [FA, module doc]:
 *   Q  rows x n_heads x head_dim, element (i, h, e) at q[i*q_row_stride + h*q_head_stride + e]
 *   K,V n_keys x n_kv_heads x head_dim with their own row/head strides
 *   mask (optional) element (h, i, j) at mask[h*mask_head_stride + i*mask_row_stride + j];
 *        mask_head_stride == 0 means one mask shared by every head.
 * Query head h reads KV head h / (n_heads / n_kv_heads): each KV head serves a
 * contiguous group of query heads.
 * pairs: optional list of (row, head) to evaluate; out is then
 * [n_pairs][head_dim]; with pairs == NULL every (row, head) is evaluated and
 * out is [rows][n_heads][head_dim].
 */
int orc_attention(const void *q, int q_dtype, int64_t q_row_stride, int64_t q_head_stride,
                  const uint16_t *k, int64_t k_row_stride, int64_t k_head_stride,
                  const uint16_t *v, int64_t v_row_stride, int64_t v_head_stride,
                  int kv_dtype,
                  const uint16_t *mask, int mask_dtype, int64_t mask_row_stride,
                  int64_t mask_head_stride,
                  int rows, int n_heads, int n_kv_heads, int head_dim, int n_keys,
                  double scale, const int32_t *pairs, int64_t n_pairs, double *out)
{
    if (rows <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || n_keys < 0 ||
        n_heads % n_kv_heads != 0)
        return 1;
    const int group = n_heads / n_kv_heads;
    const int64_t total = pairs ? n_pairs : (int64_t)rows * n_heads;
    int bad = 0;

#pragma omp parallel
    {
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        double *mrow = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
        const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(n_keys > 0 ? n_keys : 1));
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(n_keys > 0 ? n_keys : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < total; ++t) {
            int i = pairs ? pairs[2 * t] : (int)(t / n_heads);
            int h = pairs ? pairs[2 * t + 1] : (int)(t % n_heads);
            if (i < 0 || i >= rows || h < 0 || h >= n_heads) {
                bad = 1;
                continue;
            }
            int kh = h / group;
            for (int e = 0; e < head_dim; ++e)
                qrow[e] = load_q(q, q_dtype, i * q_row_stride + h * q_head_stride + e);
            for (int j = 0; j < n_keys; ++j) {
                kr[j] = k + j * k_row_stride + kh * k_head_stride;
                vr[j] = v + j * v_row_stride + kh * v_head_stride;
                if (mask)
                    mrow[j] = orc_widen16(mask[h * mask_head_stride + i * mask_row_stride + j],
                                          mask_dtype);
            }
            attention_row(qrow, head_dim, kr, vr, kv_dtype, n_keys, mask ? mrow : NULL, scale,
                          s, out + t * head_dim);
        }
        free(qrow);
        free(mrow);
        free(s);
        free(kr);
        free(vr);
    }
    return bad ? 1 : 0;
}

/*
 * Paged decode [PA, paged_state_regions; validate_signature]:
 * sequence s has context_lens[s] tokens; token t lives in physical page
 * page_table[s][t / page_size] at slot t % page_size.  Inside a page the K
 * (and separately the V) element (slot, kv_head, e) sits at
 * page*page_stride + slot*token_stride + kv_head*head_stride + e.
 * The single query of sequence s attends to all of its context tokens; no
 * mask.  seq_list (optional) picks which sequences to evaluate; out is
 * [n_list][n_heads][head_dim] (or [num_seqs][...] when seq_list == NULL).
 * Returns 1 when a page id falls outside [0, num_pages).
 */
int orc_paged_decode(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                     int kv_dtype, int64_t page_stride, int64_t token_stride,
                     int64_t head_stride, const int32_t *page_table,
                     int64_t max_pages_per_seq, const int32_t *context_lens, int num_seqs,
                     int n_heads, int n_kv_heads, int head_dim, int page_size,
                     int64_t num_pages, double scale, const int32_t *seq_list, int n_list,
                     double *out)
{
    if (num_seqs <= 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 ||
        head_dim <= 0 || page_size <= 0)
        return 1;
    const int group = n_heads / n_kv_heads;
    const int count = seq_list ? n_list : num_seqs;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int idx = 0; idx < count; ++idx) {
        for (int h = 0; h < n_heads; ++h) {
            int sq = seq_list ? seq_list[idx] : idx;
            if (sq < 0 || sq >= num_seqs) {
                bad = 1;
                continue;
            }
            int ctx = context_lens[sq];
            if (ctx < 0 ||
                (int64_t)(ctx + page_size - 1) / page_size > max_pages_per_seq) {
                bad = 1;
                continue;
            }
            int kh = h / group;
            const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(ctx + 1));
            const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(ctx + 1));
            double *s = (double *)malloc(sizeof(double) * (size_t)(ctx + 1));
            double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
            int ok = 1;
            for (int t = 0; t < ctx; ++t) {
                int32_t page = page_table[(int64_t)sq * max_pages_per_seq + t / page_size];
                if (page < 0 || page >= num_pages) {
                    ok = 0;
                    break;
                }
                int64_t off = page * page_stride + (int64_t)(t % page_size) * token_stride +
                              kh * head_stride;
                kr[t] = k_pool + off;
                vr[t] = v_pool + off;
            }
            if (!ok) {
                bad = 1;
            } else {
                for (int e = 0; e < head_dim; ++e)
                    qrow[e] = (double)q[((int64_t)sq * n_heads + h) * head_dim + e];
                attention_row(qrow, head_dim, kr, vr, kv_dtype, ctx, NULL, scale, s,
                              out + ((int64_t)idx * n_heads + h) * head_dim);
            }
            free(kr);
            free(vr);
            free(s);
            free(qrow);
        }
    }
    return bad ? 1 : 0;
}

/* ------------------------------------------------------------------ */
/* DFlash2 ring KV [DF].  geom = {lanes, q_heads, kv_heads, head_dim,  */
/* rows, window, packed_len, max_commit}.                              */
/* ------------------------------------------------------------------ */

/* DFlash2AttentionPackParams::validate, restated. */
int orc_ring_geometry_valid(const uint32_t *g)
{
    uint32_t lanes = g[0], qh = g[1], kvh = g[2], d = g[3], rows = g[4], w = g[5], k = g[6],
             mc = g[7];
    if (lanes == 0 || lanes > 4 || qh == 0 || kvh == 0 || qh % kvh != 0)
        return 0;
    if (!(d == 128 || d == 256))
        return 0;
    if (rows < 2 || rows > 16 || w <= rows || k != w - 1 + rows)
        return 0;
    if (mc == 0 || mc > rows)
        return 0;
    return 1;
}

/*
 * Pack: packed_q[b][qh][r] = bf16(cur_q[b][r][qh]);
 * packed column c < rows holds the current row c (bf16 of cur_k / cur_v);
 * column c = rows + j holds the j-th most recent history entry, which is
 * ring slot (write_position - 1 - j) mod window, copied bit for bit, when
 * j < cache_length, and zeros otherwise.  write_position is the next ring
 * slot to be written (commit writes there), so slot wp-1 is the newest.
 * Device counters are clamped: cache_length to the window, write_position
 * taken mod window.
 */
int orc_pack_attention(const uint16_t *ring_k, const uint16_t *ring_v, const float *cur_q,
                       const float *cur_k, const float *cur_v, const uint32_t *cache_lengths,
                       const uint32_t *write_positions, uint16_t *packed_q, uint16_t *packed_k,
                       uint16_t *packed_v, const uint32_t *g)
{
    if (!orc_ring_geometry_valid(g))
        return 1;
    const int64_t B = g[0], H = g[1], HK = g[2], D = g[3], R = g[4], W = g[5], K = g[6];
    for (int64_t b = 0; b < B; ++b)
        for (int64_t qh = 0; qh < H; ++qh)
            for (int64_t r = 0; r < R; ++r)
                for (int64_t e = 0; e < D; ++e)
                    packed_q[((b * H + qh) * R + r) * D + e] =
                        orc_f32_to_bf16(cur_q[((b * R + r) * H + qh) * D + e]);
    for (int64_t b = 0; b < B; ++b) {
        int64_t len = cache_lengths[b] < W ? cache_lengths[b] : W;
        int64_t wp = write_positions[b] % W;
        for (int64_t kh = 0; kh < HK; ++kh)
            for (int64_t c = 0; c < K; ++c) {
                uint16_t *dk = packed_k + ((b * HK + kh) * K + c) * D;
                uint16_t *dv = packed_v + ((b * HK + kh) * K + c) * D;
                if (c < R) {
                    for (int64_t e = 0; e < D; ++e) {
                        dk[e] = orc_f32_to_bf16(cur_k[((b * R + c) * HK + kh) * D + e]);
                        dv[e] = orc_f32_to_bf16(cur_v[((b * R + c) * HK + kh) * D + e]);
                    }
                } else {
                    int64_t j = c - R;
                    if (j < len) {
                        int64_t slot = ((wp - 1 - j) % W + W) % W;
                        const uint16_t *sk = ring_k + ((b * HK + kh) * W + slot) * D;
                        const uint16_t *sv = ring_v + ((b * HK + kh) * W + slot) * D;
                        for (int64_t e = 0; e < D; ++e) {
                            dk[e] = sk[e];
                            dv[e] = sv[e];
                        }
                    } else {
                        for (int64_t e = 0; e < D; ++e) {
                            dk[e] = 0;
                            dv[e] = 0;
                        }
                    }
                }
            }
    }
    return 0;
}

/*
 * Mask: additive bf16, identical for every query head.  Query row r sits at
 * position L + r (L = cache length); history entry j at position L - 1 - j.
 * Current rows are mutually visible.  History entry j is visible to row r
 * when it exists (j < L) and lies inside the window of `window` positions
 * ending at the query (r + j + 1 < window).  Visible -> +0, else -inf.
 */
int orc_fill_mask(const uint32_t *cache_lengths, uint16_t *mask, const uint32_t *g)
{
    if (!orc_ring_geometry_valid(g))
        return 1;
    const int64_t B = g[0], H = g[1], R = g[4], W = g[5], K = g[6];
    const uint16_t zero = 0x0000, neg_inf = 0xff80;
    for (int64_t b = 0; b < B; ++b) {
        int64_t len = cache_lengths[b] < W ? cache_lengths[b] : W;
        for (int64_t qh = 0; qh < H; ++qh)
            for (int64_t r = 0; r < R; ++r)
                for (int64_t c = 0; c < K; ++c) {
                    int visible;
                    if (c < R) {
                        visible = 1;
                    } else {
                        int64_t j = c - R;
                        visible = (j < len) && (r + j + 1 < W);
                    }
                    mask[((b * H + qh) * R + r) * K + c] = visible ? zero : neg_inf;
                }
    }
    return 0;
}

/*
 * Commit: the first n = min(commit_counts[b], max_commit) accepted rows of
 * lane b go, as bf16, to ring slots (write_position + i) mod window.  Other
 * slots are untouched; the counters themselves are read-only.
 */
int orc_commit_kv(const float *new_k, const float *new_v, const uint32_t *commit_counts,
                  const uint32_t *write_positions, uint16_t *ring_k, uint16_t *ring_v,
                  const uint32_t *g)
{
    if (!orc_ring_geometry_valid(g))
        return 1;
    const int64_t B = g[0], HK = g[2], D = g[3], W = g[5], MC = g[7];
    for (int64_t b = 0; b < B; ++b) {
        int64_t n = commit_counts[b] < MC ? commit_counts[b] : MC;
        int64_t wp = write_positions[b] % W;
        for (int64_t i = 0; i < n; ++i) {
            int64_t slot = (wp + i) % W;
            for (int64_t kh = 0; kh < HK; ++kh)
                for (int64_t e = 0; e < D; ++e) {
                    ring_k[((b * HK + kh) * W + slot) * D + e] =
                        orc_f32_to_bf16(new_k[((b * MC + i) * HK + kh) * D + e]);
                    ring_v[((b * HK + kh) * W + slot) * D + e] =
                        orc_f32_to_bf16(new_v[((b * MC + i) * HK + kh) * D + e]);
                }
        }
    }
    return 0;
}

/*
 * Page append [PA, paged_state_regions and validate_signature; the prepare
 * step writes each new token's K and V into its page before attention]: token
 * i of the batch belongs to the sequence s with token_offsets[s] <= i <
 * token_offsets[s+1] and sits at position p = position_start[s] + (i -
 * token_offsets[s]); its K row (kv head g, element e) is rounded to nearest
 * even into the pool type and stored at
 *     pool[page*page_stride + (p % page_size)*token_stride + g*head_stride + e],
 * page = page_table[s*max_pages_per_seq + p / page_size].  A token whose page
 * entry lies outside the table or the pool is not written; the count of such
 * tokens is returned in *skipped.
 */
int orc_paged_append(const float *k_new, const float *v_new, const int32_t *token_offsets,
                     const int32_t *position_start, const int32_t *page_table,
                     int64_t max_pages_per_seq, uint16_t *k_pool, uint16_t *v_pool, int kv_dtype,
                     int64_t page_stride, int64_t token_stride, int64_t head_stride, int num_seqs,
                     int n_kv_heads, int head_dim, int page_size, int64_t num_pages,
                     int64_t *skipped)
{
    if (num_seqs <= 0 || n_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
        !(kv_dtype == ORC_F16 || kv_dtype == ORC_BF16))
        return 1;
    int64_t skip = 0;
    for (int s = 0; s < num_seqs; ++s)
        for (int64_t i = token_offsets[s]; i < token_offsets[s + 1]; ++i) {
            const int64_t p = (int64_t)position_start[s] + (i - token_offsets[s]);
            const int64_t slot_page = p / page_size;
            if (p < 0 || slot_page >= max_pages_per_seq) {
                ++skip;
                continue;
            }
            const int32_t page = page_table[(int64_t)s * max_pages_per_seq + slot_page];
            if (page < 0 || page >= num_pages) {
                ++skip;
                continue;
            }
            for (int g = 0; g < n_kv_heads; ++g)
                for (int e = 0; e < head_dim; ++e) {
                    const int64_t dst = page * page_stride + (p % page_size) * token_stride +
                                        g * head_stride + e;
                    const int64_t src = (i * n_kv_heads + g) * head_dim + e;
                    k_pool[dst] = kv_dtype == ORC_F16 ? orc_f32_to_f16(k_new[src])
                                                      : orc_f32_to_bf16(k_new[src]);
                    v_pool[dst] = kv_dtype == ORC_F16 ? orc_f32_to_f16(v_new[src])
                                                      : orc_f32_to_bf16(v_new[src]);
                }
        }
    *skipped = skip;
    return 0;
}

/*
 * Paged multi-token (chunked) prefill [PA, the causal attention of `tokens`
 * new queries at position_start over the paged state]: query token i of
 * sequence s (position p as for the append above) and query head h attend to
 * the keys at positions 0..p of their sequence, gathered from the pages as in
 * paged decode: out[i][h] = sum_t softmax_t(scale q.k_t) v_t.  q f32
 * [tokens][n_heads][head_dim] (widened exactly); out double, same layout.
 */
int orc_paged_prefill(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                      int kv_dtype, int64_t page_stride, int64_t token_stride,
                      int64_t head_stride, const int32_t *page_table, int64_t max_pages_per_seq,
                      const int32_t *token_offsets, const int32_t *position_start, int num_seqs,
                      int n_heads, int n_kv_heads, int head_dim, int page_size,
                      int64_t num_pages, double scale, double *out)
{
    if (num_seqs <= 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 ||
        head_dim <= 0 || page_size <= 0)
        return 1;
    const int group = n_heads / n_kv_heads;
    const int64_t total = token_offsets[num_seqs];
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t i = 0; i < total; ++i)
        for (int h = 0; h < n_heads; ++h) {
            int s = 0;
            while (s + 1 < num_seqs && token_offsets[s + 1] <= i)
                ++s;
            const int64_t p = (int64_t)position_start[s] + (i - token_offsets[s]);
            const int64_t n = p + 1;
            if (p < 0 || (n + page_size - 1) / page_size > max_pages_per_seq) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int kh = h / group;
            const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
            const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
            double *sc = (double *)malloc(sizeof(double) * (size_t)n);
            double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
            int ok = kr && vr && sc && qrow;
            for (int64_t t = 0; ok && t < n; ++t) {
                const int32_t page = page_table[(int64_t)s * max_pages_per_seq + t / page_size];
                if (page < 0 || page >= num_pages) {
                    ok = 0;
                    break;
                }
                const int64_t off = page * page_stride + (t % page_size) * token_stride + kh * head_stride;
                kr[t] = k_pool + off;
                vr[t] = v_pool + off;
            }
            if (!ok) {
#pragma omp atomic write
                bad = 1;
            } else {
                for (int e = 0; e < head_dim; ++e)
                    qrow[e] = (double)q[(i * n_heads + h) * head_dim + e];
                attention_row(qrow, head_dim, kr, vr, kv_dtype, (int)n, NULL, scale, sc,
                              out + (i * n_heads + h) * head_dim);
            }
            free(kr);
            free(vr);
            free(sc);
            free(qrow);
        }
    return bad ? 2 : 0;
}

/*
 * Verify attention read straight from the ring [DF, the pack and mask
 * dispatchers taken together]: for lane b, query head qh (KV head
 * qh / (q_heads / kv_heads)) and draft row r, the keys are
 *   - the rows current rows c, bf16(cur_k[b][c][kh]) / bf16(cur_v[b][c][kh]),
 *     all visible, and
 *   - every ring slot s whose history index j = (write_position - 1 - s) mod w
 *     satisfies j < min(cache_length, w) and r + j + 1 < w,
 * and the query is bf16(cur_q[b][r][qh]).  This is the same set of (key,
 * value, visibility) the packed layout holds, visited in ring order instead
 * of newest first.  out: double [b][r][h][d].
 */
int orc_verify_ring_attention(const uint16_t *ring_k, const uint16_t *ring_v, const float *cur_q,
                              const float *cur_k, const float *cur_v,
                              const uint32_t *cache_lengths, const uint32_t *write_positions,
                              const uint32_t *g, double scale, double *out)
{
    if (!orc_ring_geometry_valid(g))
        return 1;
    const int64_t B = g[0], H = g[1], HK = g[2], D = g[3], R = g[4], W = g[5];
    const int64_t group = H / HK, nk = R + W;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t qh = 0; qh < H; ++qh) {
            const int64_t kh = qh / group;
            const int64_t len = cache_lengths[b] < W ? cache_lengths[b] : W;
            const int64_t wp = write_positions[b] % W;
            uint16_t *cur = (uint16_t *)malloc(sizeof(uint16_t) * 2 * R * D);
            const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * nk);
            const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * nk);
            double *s = (double *)malloc(sizeof(double) * nk);
            double *q = (double *)malloc(sizeof(double) * D);
            if (!cur || !krow || !vrow || !s || !q) {
#pragma omp atomic write
                bad = 1;
            } else {
                for (int64_t c = 0; c < R; ++c)
                    for (int64_t e = 0; e < D; ++e) {
                        cur[c * D + e] = orc_f32_to_bf16(cur_k[((b * R + c) * HK + kh) * D + e]);
                        cur[(R + c) * D + e] = orc_f32_to_bf16(cur_v[((b * R + c) * HK + kh) * D + e]);
                    }
                for (int64_t r = 0; r < R; ++r) {
                    int n = 0;
                    for (int64_t c = 0; c < R; ++c) {
                        krow[n] = cur + c * D;
                        vrow[n] = cur + (R + c) * D;
                        ++n;
                    }
                    for (int64_t slot = 0; slot < W; ++slot) {
                        const int64_t j = ((wp - 1 - slot) % W + W) % W;
                        if (j < len && r + j + 1 < W) {
                            krow[n] = ring_k + ((b * HK + kh) * W + slot) * D;
                            vrow[n] = ring_v + ((b * HK + kh) * W + slot) * D;
                            ++n;
                        }
                    }
                    for (int64_t e = 0; e < D; ++e)
                        q[e] = widen_bf16(orc_f32_to_bf16(cur_q[((b * R + r) * H + qh) * D + e]));
                    attention_row(q, (int)D, krow, vrow, ORC_BF16, n, NULL, scale, s,
                                  out + ((b * R + r) * H + qh) * D);
                }
            }
            free(cur);
            free(krow);
            free(vrow);
            free(s);
            free(q);
        }
    return bad ? 2 : 0;
}

/*
 * Draft mask rows [DF, dispatch_dflash2_mask_rows_f32 and its test
 * gpu_mask_rows_preserve_anchors]: hidden is [lanes*rows][width] f32; in each
 * lane, row 0 (the anchor) is kept and rows 1..rows-1 become the widened bf16
 * mask embedding.
 */
int orc_set_mask_rows(const uint16_t *embedding, float *hidden, uint32_t lanes, uint32_t rows,
                      uint32_t width)
{
    if (lanes == 0 || lanes > 4 || rows < 2 || rows > 16 || width == 0)
        return 1;
    for (int64_t l = 0; l < lanes; ++l)
        for (int64_t r = 1; r < rows; ++r)
            for (int64_t e = 0; e < width; ++e)
                hidden[(l * rows + r) * width + e] = (float)widen_bf16(embedding[e]);
    return 0;
}
