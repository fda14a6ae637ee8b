/*
 * oracle.c -- the oracle for the paged KV-cache write and the PagedAttention
 * decode step: a plain, slow, single-threaded CPU statement of what the two
 * operations compute, accumulated in double precision.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The product (the CUDA library and its
 * Python binding) never links, loads or calls it, and it shares no code,
 * header, table or helper with the product. It is pinned against the
 * mathematics by the CPU tests (permutation and block-size invariance, dense
 * equivalence, closed forms, brute force, format definitions), not against the
 * CUDA path.
 *
 * Sources (cited by page title and section):
 *  [TGI] "TGI PagedAttention deep-dive: block KV cache, prefix reuse and
 *        continuous batching" (lpnh.cn), sec. 4.1 (the decode kernel walks the
 *        block table; long sequences are split into 512-token partitions and
 *        merged; the write scatters new K/V by `slots`, optionally as FP8),
 *        sec. 4.2 (cache layout and block sizes), sec. 4.3 (block table,
 *        div_ceil block accounting, block 0 reserved).
 *  [L3]  "Lecture 3: PagedAttention and vLLM" (124.221.106.7), sections
 *        "Core data structure: Block Table" and "the paged implementation of
 *        attention" (logical block -> physical block, then softmax and the
 *        weighted sum), and its architecture figure (logical 0,1,2 ->
 *        physical 7,3,9).
 *  [CB]  "Continuous Batching and PagedAttention" (ai-engineering.cn),
 *        sec. 3.2 (PagedKVCache: ceil block count, fork shares blocks by
 *        reference).
 *  [OCP] OCP 8-bit Floating Point Specification (OFP8), E4M3 format: sign,
 *        4 exponent bits with bias 7, 3 mantissa bits; no infinities; the
 *        all-ones exponent+mantissa pattern is NaN; largest finite 448.
 *
 * The pages do not write out the decode arithmetic. The oracle takes the
 * textbook reading: for query head h (served by KV head floor(h / G),
 * G = Hq / Hkv), s_i = scale * <q_h, k_i> over the sequence's context_len
 * tokens, p = softmax(s), out = sum_i p_i v_i. An empty context (length 0)
 * yields a zero vector.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element type codes of the oracle's own interface. */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3 };

/* Return codes. */
enum { OR_OK = 0, OR_BAD_ARG = 1, OR_BAD_SLOT = 2, OR_BAD_BLOCK = 3, OR_NOMEM = 4 };

/* ---------------------------------------------------------------- formats */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits. */
double or_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent bits
 * with bias 127, 7 mantissa bits). */
double or_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);                /* m * 2^-7 * 2^-126 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134);     /* (1 + m/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* OCP E4M3: exponent field 0 is subnormal (m/8 * 2^-6); otherwise
 * (1 + m/8) * 2^(e-7); S.1111.111 is NaN; there is no infinity. */
double or_e4m3_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int m = c & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* E4M3 encoding of a binary32 value: round to nearest, ties to the code with
 * an even mantissa, saturating every finite or infinite magnitude above the
 * largest finite value (448) to 448 ("satfinite"). NaN maps to the NaN code
 * with the input's sign. The nearest code is found by a binary search over the
 * 127 non-negative finite codes 0x00..0x7E, whose values increase with the
 * code. */
uint8_t or_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return (uint8_t)(sign | 0x7f);
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    /* largest code lo with value(lo) <= a; value(0) = 0 <= a always */
    int lo = 0, hi = 0x7e;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (or_e4m3_to_double((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int code = lo;
    if (lo < 0x7e) {
        double below = or_e4m3_to_double((uint8_t)lo);
        double above = or_e4m3_to_double((uint8_t)(lo + 1));
        double dlo = a - below, dhi = above - a;   /* both exact in double */
        if (dhi < dlo || (dhi == dlo && ((lo + 1) & 1) == 0))
            code = lo + 1;
    }
    return (uint8_t)(sign | code);
}

static double or_read(const void* base, int dtype, int64_t i)
{
    switch (dtype) {
    case OR_F32: { float f; memcpy(&f, (const char*)base + 4 * i, 4); return (double)f; }
    case OR_F16: { uint16_t h; memcpy(&h, (const char*)base + 2 * i, 2); return or_f16_to_double(h); }
    case OR_BF16: { uint16_t b; memcpy(&b, (const char*)base + 2 * i, 2); return or_bf16_to_double(b); }
    case OR_E4M3: return or_e4m3_to_double(((const uint8_t*)base)[i]);
    }
    return NAN;
}

static int or_elem_bytes(int dtype)
{
    switch (dtype) {
    case OR_F32: return 4;
    case OR_F16: case OR_BF16: return 2;
    case OR_E4M3: return 1;
    }
    return 0;
}

/* Byte-level encoders used by tests to turn a double into the stored bits. */
void or_decode_array(const void* src, int dtype, int64_t n, double* dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_read(src, dtype, i);
}

void or_e4m3_encode_array(const float* src, int64_t n, uint8_t* dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_e4m3_encode(src[i]);
}

/* ---------------------------------------------------------------- layout */

/* A cache element (block b, KV head h, position-in-block i, component e) sits
 * at element offset b*st[0] + h*st[1] + i*st[2] + e*st[3]. The caller gives
 * the strides, so the same oracle runs any layout the pages describe. */
static int64_t or_cache_index(const int64_t* st, int64_t b, int64_t h, int64_t i, int64_t e)
{
    return b * st[0] + h * st[1] + i * st[2] + e * st[3];
}

/* ---------------------------------------------------------------- write */

/*
 * The KV write ([TGI] sec. 4.1): for each new token t with slot = slots[t],
 * block = slot / B and offset = slot mod B; copy key[t, h, :] into
 * k_cache[block, h, offset, :] and value[t, h, :] into v_cache likewise.
 * A negative slot marks a padding token and is skipped. A slot at or past
 * num_blocks * B is an error: nothing more is written and OR_BAD_SLOT is
 * returned.
 * When the cache type equals the input type the element bits are copied.
 * When the cache is E4M3 the stored code is encode(x / scale), the quotient a
 * binary32 division (k_scale for keys, v_scale for values).
 */
int or_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slots, int64_t num_tokens, int num_kv_heads, int head_size,
                         int block_size, int64_t num_blocks, int in_dtype, int cache_dtype,
                         float k_scale, float v_scale, const int64_t* cache_strides)
{
    if (num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0 || num_tokens < 0)
        return OR_BAD_ARG;
    int same = (in_dtype == cache_dtype);
    if (!same && cache_dtype != OR_E4M3)
        return OR_BAD_ARG;
    if (in_dtype == OR_E4M3)
        return OR_BAD_ARG;
    int eb = or_elem_bytes(cache_dtype);
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slots[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * (int64_t)block_size)
            return OR_BAD_SLOT;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int e = 0; e < head_size; ++e) {
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_size + e;
                int64_t dst = or_cache_index(cache_strides, blk, h, off, e);
                if (same) {
                    memcpy((char*)k_cache + dst * eb, (const char*)key + src * eb, eb);
                    memcpy((char*)v_cache + dst * eb, (const char*)value + src * eb, eb);
                } else {
                    float xk = (float)or_read(key, in_dtype, src);
                    float xv = (float)or_read(value, in_dtype, src);
                    float qk = xk / k_scale;
                    float qv = xv / v_scale;
                    ((uint8_t*)k_cache)[dst] = or_e4m3_encode(qk);
                    ((uint8_t*)v_cache)[dst] = or_e4m3_encode(qv);
                }
            }
        }
    }
    return OR_OK;
}

/* ---------------------------------------------------------------- decode */

/* Materialise the logical K and V of sequence s ([L3] "the paged
 * implementation of attention"; [TGI] sec. 4.3): logical block j < ceil(L/B)
 * lives in physical block block_tables[s][j]; logical position j*B + i is its
 * i-th slot. Output K, V are [L, Hkv, d] doubles, dequantised by the per-tensor
 * scale when the cache holds E4M3 codes. */
static int or_gather_sequence(double* K, double* V, const void* k_cache, const void* v_cache,
                              int cache_dtype, const int64_t* st, const int32_t* table, int L,
                              int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                              double k_scale, double v_scale)
{
    int nblk = (L + block_size - 1) / block_size;
    double ks = cache_dtype == OR_E4M3 ? k_scale : 1.0;
    double vs = cache_dtype == OR_E4M3 ? v_scale : 1.0;
    for (int j = 0; j < nblk; ++j) {
        int64_t p = table[j];
        if (p < 0 || p >= num_blocks)
            return OR_BAD_BLOCK;
        for (int i = 0; i < block_size; ++i) {
            int pos = j * block_size + i;
            if (pos >= L)
                break;
            for (int h = 0; h < num_kv_heads; ++h)
                for (int e = 0; e < head_size; ++e) {
                    int64_t ci = or_cache_index(st, p, h, i, e);
                    int64_t li = ((int64_t)pos * num_kv_heads + h) * head_size + e;
                    K[li] = or_read(k_cache, cache_dtype, ci) * ks;
                    V[li] = or_read(v_cache, cache_dtype, ci) * vs;
                }
        }
    }
    return OR_OK;
}

/* Softmax-weighted sum over positions [t0, t1) for one query head: returns the
 * maximum score m, the sum l of exp(s_i - m) and the normalised output
 * o = sum exp(s_i - m) v_i / l. */
static void or_attend_range(double* o, double* m_out, double* l_out, const double* q,
                            const double* K, const double* V, int t0, int t1, int kvh,
                            int num_kv_heads, int head_size, double scale, double* scores)
{
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        const double* k = K + ((int64_t)t * num_kv_heads + kvh) * head_size;
        double dot = 0.0;
        for (int e = 0; e < head_size; ++e)
            dot += q[e] * k[e];
        scores[t - t0] = scale * dot;
        if (scores[t - t0] > m)
            m = scores[t - t0];
    }
    double l = 0.0;
    for (int e = 0; e < head_size; ++e)
        o[e] = 0.0;
    for (int t = t0; t < t1; ++t) {
        double p = exp(scores[t - t0] - m);
        l += p;
        const double* v = V + ((int64_t)t * num_kv_heads + kvh) * head_size;
        for (int e = 0; e < head_size; ++e)
            o[e] += p * v[e];
    }
    for (int e = 0; e < head_size; ++e)
        o[e] /= l;
    *m_out = m;
    *l_out = l;
}

static int or_check_shape(int num_q_heads, int num_kv_heads, int head_size, int block_size)
{
    if (num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0)
        return 0;
    return num_q_heads % num_kv_heads == 0;
}

/*
 * Single-pass decode: out[s, h, :] (doubles) for every sequence s and query
 * head h. query is [S, Hq, d] of q_dtype; block_tables is [S, max_blocks].
 */
int or_decode(double* out, const void* query, int q_dtype, const void* k_cache, const void* v_cache,
              int cache_dtype, const int64_t* cache_strides, const int32_t* block_tables,
              int max_blocks, const int32_t* context_lens, int num_seqs, int num_q_heads,
              int num_kv_heads, int head_size, int block_size, int64_t num_blocks, double scale,
              double k_scale, double v_scale)
{
    if (!or_check_shape(num_q_heads, num_kv_heads, head_size, block_size))
        return OR_BAD_ARG;
    int G = num_q_heads / num_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        int L = context_lens[s];
        if (L < 0 || L > (int64_t)max_blocks * block_size)
            return OR_BAD_ARG;
        double* o_s = out + (int64_t)s * num_q_heads * head_size;
        if (L == 0) {
            for (int64_t i = 0; i < (int64_t)num_q_heads * head_size; ++i)
                o_s[i] = 0.0;
            continue;
        }
        size_t n = (size_t)L * num_kv_heads * head_size;
        double* K = malloc(n * sizeof(double));
        double* V = malloc(n * sizeof(double));
        double* sc = malloc((size_t)L * sizeof(double));
        double* q = malloc((size_t)head_size * sizeof(double));
        if (!K || !V || !sc || !q) {
            free(K); free(V); free(sc); free(q);
            return OR_NOMEM;
        }
        int rc = or_gather_sequence(K, V, k_cache, v_cache, cache_dtype, cache_strides,
                                    block_tables + (int64_t)s * max_blocks, L, num_kv_heads,
                                    head_size, block_size, num_blocks, k_scale, v_scale);
        if (rc == OR_OK) {
            for (int h = 0; h < num_q_heads; ++h) {
                for (int e = 0; e < head_size; ++e)
                    q[e] = or_read(query, q_dtype, ((int64_t)s * num_q_heads + h) * head_size + e);
                double m, l;
                or_attend_range(o_s + (int64_t)h * head_size, &m, &l, q, K, V, 0, L, h / G,
                                num_kv_heads, head_size, scale, sc);
            }
        }
        free(K); free(V); free(sc); free(q);
        if (rc != OR_OK)
            return rc;
    }
    return OR_OK;
}

/*
 * The partition merge ([TGI] sec. 4.1: partitions computed in parallel, then
 * reduced). For each (s, h) with n = ceil(L / P) partitions, given per
 * partition p its maximum score m_p, its sum l_p of exp(s_i - m_p) and its
 * normalised output o_p: M = max_p m_p, w_p = l_p * exp(m_p - M),
 * out = sum_p w_p o_p / sum_p w_p. Partials are laid out
 * part_o[s][h][p][d], part_m[s][h][p], part_l[s][h][p] with p < max_parts.
 */
int or_merge(double* out, const double* part_o, const double* part_m, const double* part_l,
             const int32_t* context_lens, int num_seqs, int num_q_heads, int head_size,
             int partition_size, int max_parts)
{
    if (partition_size <= 0 || max_parts < 0)
        return OR_BAD_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        int L = context_lens[s];
        int n = (L + partition_size - 1) / partition_size;
        if (n > max_parts)
            return OR_BAD_ARG;
        for (int h = 0; h < num_q_heads; ++h) {
            int64_t sh = (int64_t)s * num_q_heads + h;
            double* o = out + sh * head_size;
            for (int e = 0; e < head_size; ++e)
                o[e] = 0.0;
            if (n == 0)
                continue;
            double M = -INFINITY;
            for (int p = 0; p < n; ++p)
                if (part_m[sh * max_parts + p] > M)
                    M = part_m[sh * max_parts + p];
            double wsum = 0.0;
            for (int p = 0; p < n; ++p) {
                double w = part_l[sh * max_parts + p] * exp(part_m[sh * max_parts + p] - M);
                wsum += w;
                const double* op = part_o + (sh * max_parts + p) * head_size;
                for (int e = 0; e < head_size; ++e)
                    o[e] += w * op[e];
            }
            for (int e = 0; e < head_size; ++e)
                o[e] /= wsum;
        }
    }
    return OR_OK;
}

/*
 * Partitioned decode ([TGI] sec. 4.1, the 512-token partitions): partition p
 * of sequence s covers logical positions [p*P, min((p+1)*P, L)). Each partition
 * is attended on its own (m_p, l_p, normalised o_p), then or_merge combines
 * them. The partials are returned so that tests can compare them one by one.
 * Any of part_o / part_m / part_l may be NULL, in which case scratch is used.
 */
int or_decode_partitioned(double* out, double* part_o, double* part_m, double* part_l,
                          const void* query, int q_dtype, const void* k_cache, const void* v_cache,
                          int cache_dtype, const int64_t* cache_strides, const int32_t* block_tables,
                          int max_blocks, const int32_t* context_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                          double scale, double k_scale, double v_scale, int partition_size,
                          int max_parts)
{
    if (!or_check_shape(num_q_heads, num_kv_heads, head_size, block_size) || partition_size <= 0)
        return OR_BAD_ARG;
    int G = num_q_heads / num_kv_heads;
    size_t nparts = (size_t)num_seqs * num_q_heads * max_parts;
    double* po = part_o ? part_o : malloc(nparts * head_size * sizeof(double) + 1);
    double* pm = part_m ? part_m : malloc(nparts * sizeof(double) + 1);
    double* pl = part_l ? part_l : malloc(nparts * sizeof(double) + 1);
    int rc = OR_OK;
    if (!po || !pm || !pl) {
        rc = OR_NOMEM;
        goto done;
    }
    for (size_t i = 0; i < nparts; ++i) {
        pm[i] = -INFINITY;
        pl[i] = 0.0;
    }
    for (size_t i = 0; i < nparts * head_size; ++i)
        po[i] = 0.0;
    for (int s = 0; s < num_seqs && rc == OR_OK; ++s) {
        int L = context_lens[s];
        if (L < 0 || L > (int64_t)max_blocks * block_size) {
            rc = OR_BAD_ARG;
            break;
        }
        int n = (L + partition_size - 1) / partition_size;
        if (n > max_parts) {
            rc = OR_BAD_ARG;
            break;
        }
        if (L == 0)
            continue;
        size_t cnt = (size_t)L * num_kv_heads * head_size;
        double* K = malloc(cnt * sizeof(double));
        double* V = malloc(cnt * sizeof(double));
        double* sc = malloc((size_t)partition_size * sizeof(double));
        double* q = malloc((size_t)head_size * sizeof(double));
        if (!K || !V || !sc || !q) {
            free(K); free(V); free(sc); free(q);
            rc = OR_NOMEM;
            break;
        }
        rc = or_gather_sequence(K, V, k_cache, v_cache, cache_dtype, cache_strides,
                                block_tables + (int64_t)s * max_blocks, L, num_kv_heads, head_size,
                                block_size, num_blocks, k_scale, v_scale);
        for (int h = 0; h < num_q_heads && rc == OR_OK; ++h) {
            int64_t sh = (int64_t)s * num_q_heads + h;
            for (int e = 0; e < head_size; ++e)
                q[e] = or_read(query, q_dtype, sh * head_size + e);
            for (int p = 0; p < n; ++p) {
                int t0 = p * partition_size;
                int t1 = t0 + partition_size < L ? t0 + partition_size : L;
                or_attend_range(po + (sh * max_parts + p) * head_size, &pm[sh * max_parts + p],
                                &pl[sh * max_parts + p], q, K, V, t0, t1, h / G, num_kv_heads,
                                head_size, scale, sc);
            }
        }
        free(K); free(V); free(sc); free(q);
    }
    if (rc == OR_OK)
        rc = or_merge(out, po, pm, pl, context_lens, num_seqs, num_q_heads, head_size,
                      partition_size, max_parts);
done:
    if (!part_o) free(po);
    if (!part_m) free(pm);
    if (!part_l) free(pl);
    return rc;
}

/*
 * Multi-query paged attention (chunked prefill, speculative verification):
 * sequence s brings Q_s = query_start[s+1] - query_start[s] query tokens, the
 * last Q_s positions of its context of L_s tokens; query i sits at position
 * p = L_s - Q_s + i and attends to the keys at positions 0..p (causal), through
 * the block table exactly as the decode does ("Lecture 3: PagedAttention and
 * vLLM", "the paged implementation of attention", whose listing already takes
 * queries [num_queries, num_heads, head_dim]). query and out are
 * [total_queries, Hq, d]. Q_s > L_s is an error. With Q_s = 1 this is the
 * decode.
 */
int or_paged_prefill(double* out, const void* query, int q_dtype, const int32_t* query_start,
                     const void* k_cache, const void* v_cache, int cache_dtype,
                     const int64_t* cache_strides, const int32_t* block_tables, int max_blocks,
                     const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_size, int block_size, int64_t num_blocks, double scale,
                     double k_scale, double v_scale)
{
    if (!or_check_shape(num_q_heads, num_kv_heads, head_size, block_size))
        return OR_BAD_ARG;
    int G = num_q_heads / num_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        int L = context_lens[s];
        int q0 = query_start[s], Q = query_start[s + 1] - q0;
        if (L < 0 || Q < 0 || Q > L || L > (int64_t)max_blocks * block_size)
            return OR_BAD_ARG;
        if (Q == 0)
            continue;
        size_t n = (size_t)L * num_kv_heads * head_size;
        double* K = malloc(n * sizeof(double));
        double* V = malloc(n * sizeof(double));
        double* sc = malloc((size_t)L * sizeof(double));
        double* q = malloc((size_t)head_size * sizeof(double));
        if (!K || !V || !sc || !q) {
            free(K); free(V); free(sc); free(q);
            return OR_NOMEM;
        }
        int rc = or_gather_sequence(K, V, k_cache, v_cache, cache_dtype, cache_strides,
                                    block_tables + (int64_t)s * max_blocks, L, num_kv_heads,
                                    head_size, block_size, num_blocks, k_scale, v_scale);
        for (int i = 0; i < Q && rc == OR_OK; ++i) {
            int pos = L - Q + i;
            for (int h = 0; h < num_q_heads; ++h) {
                int64_t row = ((int64_t)(q0 + i) * num_q_heads + h) * head_size;
                for (int e = 0; e < head_size; ++e)
                    q[e] = or_read(query, q_dtype, row + e);
                double m, l;
                or_attend_range(out + row, &m, &l, q, K, V, 0, pos + 1, h / G, num_kv_heads,
                                head_size, scale, sc);
            }
        }
        free(K); free(V); free(sc); free(q);
        if (rc != OR_OK)
            return rc;
    }
    return OR_OK;
}

/* The copy of copy-on-write ("vLLM Page Attention Continuous Batching"
 * (lbrq.cn), "Sharing KV Cache-COW"): for each (src, dst) pair, every element
 * of block src of both caches is copied to block dst. block_elems =
 * Hkv * B * d elements of elem_bytes each, blocks contiguous. Pairs are applied
 * in order. Returns OR_BAD_BLOCK (and stops) on an id outside the pool. */
int or_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int64_t num_pairs,
                   int64_t num_blocks, int64_t block_elems, int elem_bytes)
{
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return OR_BAD_BLOCK;
        for (int64_t e = 0; e < block_elems * elem_bytes; ++e) {
            ((char*)k_cache)[dst * block_elems * elem_bytes + e] =
                ((const char*)k_cache)[src * block_elems * elem_bytes + e];
            ((char*)v_cache)[dst * block_elems * elem_bytes + e] =
                ((const char*)v_cache)[src * block_elems * elem_bytes + e];
        }
    }
    return OR_OK;
}

/* ceil(tokens / block_size): the number of blocks a sequence of `tokens`
 * tokens occupies ([TGI] sec. 4.3 div_ceil; [CB] sec. 3.2). */
int64_t or_blocks_needed(int64_t tokens, int block_size)
{
    return (tokens + block_size - 1) / block_size;
}
