/*
 * pkv_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the paged
 * KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The product path never
 * calls it, and it shares no code, header or helper with the CUDA library.
 *
 * What it follows (AstrAI, "docs/guides/inference.md"):
 *   - section "KV Cache": decode output o_n = sum_j softmax(q_n k_j / sqrt(d_k)) v_j,
 *     with RoPE applied before the cache write;
 *   - section "KVCache System": k_buffer / v_buffer laid out as
 *     [n_layers, size, n_kv_heads, head_dim], req_to_token [num_reqs, max_ctx_len]
 *     mapping a request's logical position to a physical token slot, the
 *     KVCache fields req_pool_indices, seq_lens, out_cache_loc, kv_indptr,
 *     qo_indptr, and the write `k_buffer[layer_id, out_cache_loc] = k`;
 *   - section "Attention Backend": decode writes K/V first and then reads the
 *     cache through req_to_token (page_size = 1: one slot per "page"); prefill
 *     writes K/V and then attends over a ragged batch addressed by
 *     qo_indptr / kv_indptr;
 *   - section "Rotary Embedding Backend": the cos/sin table freqs_cis
 *     [max_len, dim/2, 2] (f32 pairs) and a complex multiply per pair.
 * Causal alignment with a cached prefix follows astrai/model/transformer.py
 * `process_attention_mask` (mask length start_pos + seq_len): query row i of a
 * request whose cached prefix has P tokens sees logical positions j <= P + i.
 *
 * Readings taken where the pages are silent:
 *   - grouped-query mapping: query head h reads kv head h / (n_heads / n_kv_heads);
 *   - a context of length 0 yields an all-zero output row;
 *   - scale is passed in (the formula uses 1 / sqrt(head_dim));
 *   - the rotation pairs element 2i with 2i+1 (view_as_complex on the last dim).
 *
 * Every score, weight and sum is computed in double from the exact stored
 * values (bf16 widens exactly).  There is no blocking, splitting or online
 * rescaling: each output is the plain definition written out.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_OK = 0, ORACLE_ERR_ARG = -1, ORACLE_ERR_INDEX = -4, ORACLE_ERR_NOMEM = -6 };

/* Exact widening of one stored element to double. */
static double elem(const void *base, int dtype, int64_t index)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[index];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[index] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int elem_bytes(int dtype)
{
    return dtype == ORACLE_F32 ? 4 : 2;
}

/*
 * K/V cache write: k_buffer[layer_id, out_cache_loc[i]] = k[i] and the same
 * for v, for i in [0, n_new).  k and v are [n_new, n_kv_heads, head_dim].  The
 * copy is byte-for-byte, so the result is exact.  Later rows win on duplicate
 * locations (the pages leave duplicates unspecified).
 */
int oracle_kv_write(void *k_buffer, void *v_buffer, int dtype, int n_layers, int64_t size,
                    int n_kv_heads, int head_dim, int layer_id, const void *k, const void *v,
                    const int32_t *out_cache_loc, int64_t n_new)
{
    if (layer_id < 0 || layer_id >= n_layers || n_new < 0)
        return ORACLE_ERR_ARG;
    int64_t row = (int64_t)n_kv_heads * head_dim * elem_bytes(dtype);
    for (int64_t i = 0; i < n_new; ++i) {
        int64_t loc = out_cache_loc[i];
        if (loc < 0 || loc >= size)
            return ORACLE_ERR_INDEX;
        int64_t dst = ((int64_t)layer_id * size + loc) * row;
        memcpy((char *)k_buffer + dst, (const char *)k + i * row, (size_t)row);
        memcpy((char *)v_buffer + dst, (const char *)v + i * row, (size_t)row);
    }
    return ORACLE_OK;
}

/*
 * Attention of one query row over the first n logical positions of request
 * row r:  s_j = scale * sum_e q[e] K[slot_j, g, e];  w_j = exp(s_j - max s);
 * out[e] = sum_j w_j V[slot_j, g, e] / sum_j w_j,  slot_j = req_to_token[r, j].
 * `scores` has room for n doubles.
 */
static int attend(const void *k_buffer, const void *v_buffer, int dtype, int64_t size,
                  int n_kv_heads, int head_dim, int layer_id, const int32_t *req_to_token,
                  int max_ctx_len, int r, int n, int g, const void *q, int64_t q_off,
                  double scale, double *scores, double *out)
{
    for (int e = 0; e < head_dim; ++e)
        out[e] = 0.0;
    if (n == 0)
        return ORACLE_OK;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        int64_t slot = req_to_token[(int64_t)r * max_ctx_len + j];
        if (slot < 0 || slot >= size)
            return ORACLE_ERR_INDEX;
        int64_t k_off = (((int64_t)layer_id * size + slot) * n_kv_heads + g) * head_dim;
        double dot = 0.0;
        for (int e = 0; e < head_dim; ++e)
            dot += elem(q, dtype, q_off + e) * elem(k_buffer, dtype, k_off + e);
        scores[j] = scale * dot;
        if (scores[j] > m)
            m = scores[j];
    }
    double denom = 0.0;
    for (int j = 0; j < n; ++j) {
        double w = exp(scores[j] - m);
        denom += w;
        int64_t slot = req_to_token[(int64_t)r * max_ctx_len + j];
        int64_t v_off = (((int64_t)layer_id * size + slot) * n_kv_heads + g) * head_dim;
        for (int e = 0; e < head_dim; ++e)
            out[e] += w * elem(v_buffer, dtype, v_off + e);
    }
    for (int e = 0; e < head_dim; ++e)
        out[e] /= denom;
    return ORACLE_OK;
}

/*
 * Decode attention: one query token per request.  For batch entry b, request
 * row r = req_pool_indices[b], context n = seq_lens[b] (the token written this
 * step included), query head h of q [batch, n_heads, head_dim]:
 * o[b, h] = attention of q[b, h] over positions [0, n) of row r with kv head
 * h / (n_heads / n_kv_heads).  When kv_indptr is given, its differences must
 * equal seq_lens.  o is [batch, n_heads, head_dim] doubles.
 */
int oracle_decode(const void *k_buffer, const void *v_buffer, int dtype, int n_layers,
                  int64_t size, int n_kv_heads, int head_dim, const int32_t *req_to_token,
                  int num_reqs, int max_ctx_len, const int32_t *req_pool_indices,
                  const int32_t *seq_lens, const int32_t *kv_indptr, int batch, int layer_id,
                  const void *q, int n_heads, double scale, double *o)
{
    if (layer_id < 0 || layer_id >= n_layers || n_kv_heads <= 0 || n_heads % n_kv_heads)
        return ORACLE_ERR_ARG;
    int group = n_heads / n_kv_heads;
    double *scores = malloc(sizeof(double) * (size_t)(max_ctx_len > 0 ? max_ctx_len : 1));
    if (!scores)
        return ORACLE_ERR_NOMEM;
    int rc = ORACLE_OK;
    for (int b = 0; b < batch && rc == ORACLE_OK; ++b) {
        int r = req_pool_indices[b];
        int n = seq_lens[b];
        if (r < 0 || r >= num_reqs || n < 0 || n > max_ctx_len) {
            rc = ORACLE_ERR_INDEX;
            break;
        }
        if (kv_indptr && kv_indptr[b + 1] - kv_indptr[b] != n) {
            rc = ORACLE_ERR_ARG;
            break;
        }
        for (int h = 0; h < n_heads && rc == ORACLE_OK; ++h) {
            int64_t row = (int64_t)b * n_heads + h;
            rc = attend(k_buffer, v_buffer, dtype, size, n_kv_heads, head_dim, layer_id,
                        req_to_token, max_ctx_len, r, n, h / group, q, row * head_dim, scale,
                        scores, o + row * head_dim);
        }
    }
    free(scores);
    return rc;
}

/*
 * Ragged prefill.  q and the output are packed [sum q_len, n_heads, head_dim];
 * request b owns packed rows [qo_indptr[b], qo_indptr[b+1]) and has
 * kv_len = kv_indptr[b+1] - kv_indptr[b] cached positions, of which the last
 * q_len are the new tokens (already written), so its prefix is P = kv_len - q_len.
 * Row i of request b sees positions [0, P + i] when causal, else [0, kv_len).
 * `rows` selects which packed rows to compute (NULL: all, in order); o is
 * [n_rows, n_heads, head_dim] doubles.
 */
int oracle_prefill(const void *k_buffer, const void *v_buffer, int dtype, int n_layers,
                   int64_t size, int n_kv_heads, int head_dim, const int32_t *req_to_token,
                   int num_reqs, int max_ctx_len, const int32_t *req_pool_indices,
                   const int32_t *qo_indptr, const int32_t *kv_indptr, int batch, int layer_id,
                   const void *q, int n_heads, int causal, double scale, const int64_t *rows,
                   int64_t n_rows, double *o)
{
    if (layer_id < 0 || layer_id >= n_layers || n_kv_heads <= 0 || n_heads % n_kv_heads)
        return ORACLE_ERR_ARG;
    int group = n_heads / n_kv_heads;
    int64_t total = qo_indptr[batch];
    if (!rows)
        n_rows = total;
    double *scores = malloc(sizeof(double) * (size_t)(max_ctx_len > 0 ? max_ctx_len : 1));
    if (!scores)
        return ORACLE_ERR_NOMEM;
    int rc = ORACLE_OK;
    for (int64_t t = 0; t < n_rows && rc == ORACLE_OK; ++t) {
        int64_t p = rows ? rows[t] : t;
        if (p < 0 || p >= total) {
            rc = ORACLE_ERR_ARG;
            break;
        }
        int b = 0;
        while (qo_indptr[b + 1] <= p)
            ++b;
        int r = req_pool_indices[b];
        int q_len = qo_indptr[b + 1] - qo_indptr[b];
        int kv_len = kv_indptr[b + 1] - kv_indptr[b];
        int i = (int)(p - qo_indptr[b]);
        if (r < 0 || r >= num_reqs || kv_len < q_len || kv_len > max_ctx_len) {
            rc = ORACLE_ERR_INDEX;
            break;
        }
        int visible = causal ? (kv_len - q_len) + i + 1 : kv_len;
        for (int h = 0; h < n_heads && rc == ORACLE_OK; ++h) {
            rc = attend(k_buffer, v_buffer, dtype, size, n_kv_heads, head_dim, layer_id,
                        req_to_token, max_ctx_len, r, visible, h / group, q,
                        (p * n_heads + h) * head_dim, scale, scores,
                        o + (t * n_heads + h) * head_dim);
        }
    }
    free(scores);
    return rc;
}

/*
 * Rotary embedding of one row set, as a complex multiply: for each row n with
 * position pos[n], head h and pair i, (x[2i] + i x[2i+1]) * (cos + i sin) where
 * (cos, sin) = freqs_cis[pos[n], i, 0..1].  x is [n_rows, n_heads, head_dim] of
 * `dtype`; out is the same shape in double.
 */
int oracle_rope(const void *x, int dtype, int64_t n_rows, int n_heads, int head_dim,
                const float *freqs_cis, int max_pos, const int32_t *pos, double *out)
{
    if (head_dim % 2)
        return ORACLE_ERR_ARG;
    for (int64_t n = 0; n < n_rows; ++n) {
        if (pos[n] < 0 || pos[n] >= max_pos)
            return ORACLE_ERR_INDEX;
        const float *cs = freqs_cis + (int64_t)pos[n] * head_dim;
        for (int h = 0; h < n_heads; ++h) {
            int64_t base = (n * n_heads + h) * head_dim;
            for (int i = 0; i < head_dim / 2; ++i) {
                double re = elem(x, dtype, base + 2 * i);
                double im = elem(x, dtype, base + 2 * i + 1);
                double c = cs[2 * i], s = cs[2 * i + 1];
                out[base + 2 * i] = re * c - im * s;
                out[base + 2 * i + 1] = re * s + im * c;
            }
        }
    }
    return ORACLE_OK;
}
