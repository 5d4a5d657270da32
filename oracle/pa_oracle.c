/*
 * ORACLE -- test infrastructure only.  A plain, slow, fp64 CPU statement of
 * what the paged-attention hot path computes.  It shares no code with the
 * CUDA library; only the tests, the smoke check and the benchmark's CPU
 * baseline may call it.
 *
 * Sources (the three PagedAttention pages):
 *   - "Q32: vLLM PagedAttention 原理" (agentalpha.top), §2 "PagedAttention的解决方案":
 *     the KV cache is cut into fixed-size blocks (16 tokens by default); a
 *     per-request block table maps logical block i to a physical block
 *     (example: logical 0 -> physical 5, logical 1 -> physical 12).
 *   - data.6616ai.com/article/vllm, "把虚拟内存搬进 KV Cache": the attention
 *     kernel reads KV by block index, logically contiguous and physically
 *     scattered.
 *   - ohmygp.com "batch-008-day-02-interview-1", "破局思路": one token takes one
 *     slot; a new block is taken only when the current one is full.
 *
 * What the oracle computes is the plain definition: for sequence b, walk its
 * block table to rebuild the contiguous keys K^[t] and values V^[t],
 * t < len_b (token t lives in physical block table[b][t / bs] at offset
 * t % bs), widen them exactly to double, and for each query head h of KV
 * head g = h / (Hq / Hkv) form
 *     s_t = scale * sum_i q[b,h,i] K^[t,i],   w = softmax(s),   out = sum_t w_t V^[t].
 * An empty sequence gives a zero output.
 *
 * Layouts (row-major): pools [num_blocks][Hkv][bs][D]; q [B][Hq][D];
 * block_tables [B][max_blocks_per_seq]; out [B][Hq][D] (double).
 * Element type: dtype 0 = fp32, 1 = bf16 (uint16 bit patterns).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_BAD_BLOCK = -2, ORACLE_BAD_SLOT = -3, ORACLE_NOMEM = -4 };

double oracle_e4m3_value(uint8_t c);

/* dtype: 0 fp32, 1 bf16 bits, 3 OCP E4M3 codes (their value; the pool scale is applied by the caller) */
static double load_elem(int dtype, const void* base, size_t idx) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    if (dtype == 3) return oracle_e4m3_value(((const uint8_t*)base)[idx]);
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16; /* bf16 -> fp32 is exact */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Gather K^ and V^ of (sequence b, KV head g) into contiguous [len][D] arrays; element values
   times the pool scales (1 unless the pools hold FP8 codes). */
static int gather_kv(int dtype, const void* k_pool, const void* v_pool, const int32_t* table,
                     int32_t len, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                     int32_t num_blocks, int32_t g, double k_scale, double v_scale, double* K, double* V) {
    for (int32_t t = 0; t < len; ++t) {
        int32_t phys = table[t / block_size];
        if (phys < 0 || phys >= num_blocks) return ORACLE_BAD_BLOCK;
        size_t row = (((size_t)phys * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * head_dim;
        for (int32_t i = 0; i < head_dim; ++i) {
            K[(size_t)t * head_dim + i] = load_elem(dtype, k_pool, row + i) * k_scale;
            V[(size_t)t * head_dim + i] = load_elem(dtype, v_pool, row + i) * v_scale;
        }
    }
    return ORACLE_OK;
}

static int check_common(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t seq_begin, int32_t seq_end) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return ORACLE_BAD_ARG;
    if (head_dim <= 0 || block_size <= 0) return ORACLE_BAD_ARG;
    if (seq_begin < 0 || seq_end > num_seqs || seq_begin > seq_end) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/* Decode attention with separate element types for q and for the pools. */
static int decode_impl(int q_dtype, const void* q, int kv_dtype, const void* k_pool, const void* v_pool,
                       double k_scale, double v_scale, const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks, double scale, int32_t seq_begin,
                       int32_t seq_end, double* out);

/* Decode attention for sequences [seq_begin, seq_end); writes out[b] for those b only. */
int oracle_decode_attention(int dtype, const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, double scale, int32_t seq_begin, int32_t seq_end,
                            double* out) {
    return decode_impl(dtype, q, dtype, k_pool, v_pool, 1.0, 1.0, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, seq_begin,
                       seq_end, out);
}

static int decode_impl(int q_dtype, const void* q, int kv_dtype, const void* k_pool, const void* v_pool,
                       double k_scale, double v_scale, const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks, double scale, int32_t seq_begin,
                       int32_t seq_end, double* out) {
    int rc = check_common(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, seq_begin, seq_end);
    if (rc) return rc;
    const int32_t G = num_q_heads / num_kv_heads;
    for (int32_t b = seq_begin; b < seq_end; ++b) {
        const int32_t len = seq_lens[b];
        if (len < 0 || (int64_t)len > (int64_t)max_blocks_per_seq * block_size) return ORACLE_BAD_ARG;
        double* outb = out + (size_t)b * num_q_heads * head_dim;
        if (len == 0) {
            memset(outb, 0, sizeof(double) * (size_t)num_q_heads * head_dim);
            continue;
        }
        double* K = (double*)malloc(sizeof(double) * (size_t)len * head_dim);
        double* V = (double*)malloc(sizeof(double) * (size_t)len * head_dim);
        double* s = (double*)malloc(sizeof(double) * (size_t)len);
        if (!K || !V || !s) {
            free(K); free(V); free(s);
            return ORACLE_NOMEM;
        }
        const int32_t* table = block_tables + (size_t)b * max_blocks_per_seq;
        for (int32_t g = 0; g < num_kv_heads && rc == ORACLE_OK; ++g) {
            rc = gather_kv(kv_dtype, k_pool, v_pool, table, len, num_kv_heads, head_dim, block_size,
                           num_blocks, g, k_scale, v_scale, K, V);
            if (rc) break;
            for (int32_t h = g * G; h < (g + 1) * G; ++h) {
                size_t qrow = ((size_t)b * num_q_heads + h) * head_dim;
                double m = -INFINITY;
                for (int32_t t = 0; t < len; ++t) {
                    double dot = 0.0;
                    for (int32_t i = 0; i < head_dim; ++i)
                        dot += load_elem(q_dtype, q, qrow + i) * K[(size_t)t * head_dim + i];
                    s[t] = scale * dot;
                    if (s[t] > m) m = s[t];
                }
                double denom = 0.0;
                for (int32_t t = 0; t < len; ++t) {
                    s[t] = exp(s[t] - m);
                    denom += s[t];
                }
                double* o = outb + (size_t)h * head_dim;
                for (int32_t i = 0; i < head_dim; ++i) o[i] = 0.0;
                for (int32_t t = 0; t < len; ++t) {
                    double w = s[t] / denom;
                    for (int32_t i = 0; i < head_dim; ++i) o[i] += w * V[(size_t)t * head_dim + i];
                }
            }
        }
        free(K); free(V); free(s);
        if (rc) return rc;
    }
    return ORACLE_OK;
}

/*
 * Split-sequence form (flash-decoding): the tokens of each sequence are cut
 * into partitions of P tokens; partition p yields, per query head,
 *   m_p = max_t s_t,  l_p = sum_t exp(s_t - m_p),  o_p = sum_t exp(s_t - m_p) V^[t]
 * (unnormalised).  Partitions past the end of the sequence hold m = -inf,
 * l = 0, o = 0.  Arrays: m, l [B][Hq][n_part]; o [B][Hq][n_part][D].
 */
int oracle_decode_partials(int dtype, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int32_t num_blocks, double scale, int32_t partition_tokens, int32_t n_part,
                           double* m_out, double* l_out, double* o_out) {
    int rc = check_common(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 0, num_seqs);
    if (rc) return rc;
    if (partition_tokens <= 0 || n_part <= 0) return ORACLE_BAD_ARG;
    const int32_t G = num_q_heads / num_kv_heads;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t len = seq_lens[b];
        if (len < 0 || (int64_t)len > (int64_t)max_blocks_per_seq * block_size) return ORACLE_BAD_ARG;
        if ((int64_t)n_part * partition_tokens < len) return ORACLE_BAD_ARG;
        double* K = (double*)malloc(sizeof(double) * ((size_t)len + 1) * head_dim);
        double* V = (double*)malloc(sizeof(double) * ((size_t)len + 1) * head_dim);
        if (!K || !V) {
            free(K); free(V);
            return ORACLE_NOMEM;
        }
        const int32_t* table = block_tables + (size_t)b * max_blocks_per_seq;
        for (int32_t g = 0; g < num_kv_heads && rc == ORACLE_OK; ++g) {
            rc = gather_kv(dtype, k_pool, v_pool, table, len, num_kv_heads, head_dim, block_size,
                           num_blocks, g, 1.0, 1.0, K, V);
            if (rc) break;
            for (int32_t h = g * G; h < (g + 1) * G; ++h) {
                size_t qrow = ((size_t)b * num_q_heads + h) * head_dim;
                for (int32_t p = 0; p < n_part; ++p) {
                    size_t pi = ((size_t)b * num_q_heads + h) * n_part + p;
                    double* o = o_out + pi * head_dim;
                    for (int32_t i = 0; i < head_dim; ++i) o[i] = 0.0;
                    int64_t t0 = (int64_t)p * partition_tokens;
                    int64_t t1 = t0 + partition_tokens < len ? t0 + partition_tokens : len;
                    double m = -INFINITY, l = 0.0;
                    for (int64_t t = t0; t < t1; ++t) {
                        double dot = 0.0;
                        for (int32_t i = 0; i < head_dim; ++i)
                            dot += load_elem(dtype, q, qrow + i) * K[(size_t)t * head_dim + i];
                        if (scale * dot > m) m = scale * dot;
                    }
                    for (int64_t t = t0; t < t1; ++t) {
                        double dot = 0.0;
                        for (int32_t i = 0; i < head_dim; ++i)
                            dot += load_elem(dtype, q, qrow + i) * K[(size_t)t * head_dim + i];
                        double e = exp(scale * dot - m);
                        l += e;
                        for (int32_t i = 0; i < head_dim; ++i) o[i] += e * V[(size_t)t * head_dim + i];
                    }
                    m_out[pi] = m;
                    l_out[pi] = l;
                }
            }
        }
        free(K); free(V);
        if (rc) return rc;
    }
    return ORACLE_OK;
}

/* Reduce of the partitions: M = max_p m_p, out = sum_p e^{m_p-M} o_p / sum_p e^{m_p-M} l_p. */
int oracle_combine_partials(int32_t rows, int32_t n_part, int32_t head_dim, const double* m_in,
                            const double* l_in, const double* o_in, double* out) {
    if (rows < 0 || n_part <= 0 || head_dim <= 0) return ORACLE_BAD_ARG;
    for (int32_t r = 0; r < rows; ++r) {
        const double* m = m_in + (size_t)r * n_part;
        const double* l = l_in + (size_t)r * n_part;
        double M = -INFINITY;
        for (int32_t p = 0; p < n_part; ++p)
            if (m[p] > M) M = m[p];
        double* o = out + (size_t)r * head_dim;
        for (int32_t i = 0; i < head_dim; ++i) o[i] = 0.0;
        if (M == -INFINITY) continue; /* every partition empty: zero output */
        double L = 0.0;
        for (int32_t p = 0; p < n_part; ++p) {
            if (m[p] == -INFINITY) continue;
            double w = exp(m[p] - M);
            L += w * l[p];
            const double* op = o_in + ((size_t)r * n_part + p) * head_dim;
            for (int32_t i = 0; i < head_dim; ++i) o[i] += w * op[i];
        }
        for (int32_t i = 0; i < head_dim; ++i) o[i] /= L;
    }
    return ORACLE_OK;
}

/*
 * Slot-mapped append: token i with slot s >= 0 is written to physical block
 * s / bs at offset s % bs, every KV head, K and V.  A negative slot is
 * skipped.  Plain element copies.
 */
int oracle_reshape_and_cache(int32_t elem_bytes, const void* k_new, const void* v_new, void* k_pool,
                             void* v_pool, const int64_t* slot_mapping, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks) {
    if (elem_bytes != 2 && elem_bytes != 4) return ORACLE_BAD_ARG;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0) continue;
        int64_t blk = s / block_size, off = s % block_size;
        if (blk >= num_blocks) return ORACLE_BAD_SLOT;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            for (int32_t e = 0; e < head_dim; ++e) {
                size_t src = ((size_t)i * num_kv_heads + h) * head_dim + e;
                size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * head_dim + e;
                memcpy((char*)k_pool + dst * elem_bytes, (const char*)k_new + src * elem_bytes, elem_bytes);
                memcpy((char*)v_pool + dst * elem_bytes, (const char*)v_new + src * elem_bytes, elem_bytes);
            }
        }
    }
    return ORACLE_OK;
}

/* Copy-on-write block copy: pool[dst] <- pool[src] for each pair, K and V, the whole block. */
int oracle_copy_blocks(int32_t elem_bytes, void* k_pool, void* v_pool, const int32_t* pairs,
                       int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int32_t num_blocks) {
    if (elem_bytes != 2 && elem_bytes != 4) return ORACLE_BAD_ARG;
    const size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
    for (int32_t p = 0; p < num_pairs; ++p) {
        int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORACLE_BAD_BLOCK;
        for (size_t e = 0; e < block_elems; ++e) {
            memcpy((char*)k_pool + ((size_t)dst * block_elems + e) * elem_bytes,
                   (const char*)k_pool + ((size_t)src * block_elems + e) * elem_bytes, elem_bytes);
            memcpy((char*)v_pool + ((size_t)dst * block_elems + e) * elem_bytes,
                   (const char*)v_pool + ((size_t)src * block_elems + e) * elem_bytes, elem_bytes);
        }
    }
    return ORACLE_OK;
}

/*
 * Paged prefill (chunked append) attention.  The pages put the same block
 * table in front of every attention read ("把虚拟内存搬进 KV Cache": the
 * attention kernel reads KV by block index; "Q32" follow-up 3: FlashAttention
 * loads the KV cache block by block, adapted to non-contiguous storage), and
 * prefill is the step that computes a prompt's queries against that cache.
 *
 * Sequence b holds seq_lens[b] tokens in the cache; the last
 * n_b = cu_q_lens[b+1] - cu_q_lens[b] of them are the chunk whose queries are
 * given.  Chunk token i sits at position p = seq_lens[b] - n_b + i and, as in
 * any causal language model, attends to the keys at positions 0..p:
 *     s_t = scale * q . K^[t] (t <= p),  w = softmax(s),  out = sum_t w_t V^[t].
 * q and out are [T][Hq][D] with T = cu_q_lens[num_seqs]; chunk token i of
 * sequence b is row cu_q_lens[b] + i.  Writes the rows of sequences
 * [seq_begin, seq_end) only.
 */
int oracle_prefill_attention(int dtype, const void* q, const void* k_pool, const void* v_pool,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t num_seqs,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks, double scale, int32_t seq_begin, int32_t seq_end, double* out) {
    int rc = check_common(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, seq_begin, seq_end);
    if (rc) return rc;
    const int32_t G = num_q_heads / num_kv_heads;
    for (int32_t b = seq_begin; b < seq_end; ++b) {
        const int32_t len = seq_lens[b];
        const int32_t n = cu_q_lens[b + 1] - cu_q_lens[b];
        if (n < 0 || len < n || (int64_t)len > (int64_t)max_blocks_per_seq * block_size) return ORACLE_BAD_ARG;
        if (n == 0) continue;
        double* K = (double*)malloc(sizeof(double) * (size_t)len * head_dim);
        double* V = (double*)malloc(sizeof(double) * (size_t)len * head_dim);
        double* s = (double*)malloc(sizeof(double) * (size_t)len);
        if (!K || !V || !s) {
            free(K); free(V); free(s);
            return ORACLE_NOMEM;
        }
        const int32_t* table = block_tables + (size_t)b * max_blocks_per_seq;
        for (int32_t g = 0; g < num_kv_heads && rc == ORACLE_OK; ++g) {
            rc = gather_kv(dtype, k_pool, v_pool, table, len, num_kv_heads, head_dim, block_size,
                           num_blocks, g, 1.0, 1.0, K, V);
            if (rc) break;
            for (int32_t i = 0; i < n; ++i) {
                const int32_t p = len - n + i; /* this token's position: keys 0..p are visible */
                const size_t row = (size_t)cu_q_lens[b] + (size_t)i;
                for (int32_t h = g * G; h < (g + 1) * G; ++h) {
                    const size_t qrow = (row * num_q_heads + h) * head_dim;
                    double m = -INFINITY;
                    for (int32_t t = 0; t <= p; ++t) {
                        double dot = 0.0;
                        for (int32_t d = 0; d < head_dim; ++d)
                            dot += load_elem(dtype, q, qrow + d) * K[(size_t)t * head_dim + d];
                        s[t] = scale * dot;
                        if (s[t] > m) m = s[t];
                    }
                    double denom = 0.0;
                    for (int32_t t = 0; t <= p; ++t) {
                        s[t] = exp(s[t] - m);
                        denom += s[t];
                    }
                    double* o = out + qrow;
                    for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
                    for (int32_t t = 0; t <= p; ++t) {
                        const double w = s[t] / denom;
                        for (int32_t d = 0; d < head_dim; ++d) o[d] += w * V[(size_t)t * head_dim + d];
                    }
                }
            }
        }
        free(K); free(V); free(s);
        if (rc) return rc;
    }
    return ORACLE_OK;
}

/*
 * FP8 KV pool (an extrapolation: the pages name FP8 only among the quantisation
 * formats the ecosystem supports, data.6616ai.com "PagedAttention 之外").
 *
 * Codes are OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent field 0 holds subnormals m * 2^-9; the all-ones exponent with
 * mantissa 7 is NaN and there is no infinity; the largest finite magnitude is
 * 448).  A pool holds codes of x / scale, one fp32 scale per pool (K and V):
 * the append computes y = x / scale in fp32 and rounds y to the nearest
 * finite E4M3 value, ties to the code with an even mantissa, magnitudes past
 * 448 saturating to 448.  Decode reads x^ = value(code) * scale.
 */
double oracle_e4m3_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round an fp32 value to E4M3 as above, by search over the 127 finite magnitudes. */
uint8_t oracle_e4m3_encode(float y) {
    if (isnan(y)) return 0x7F;
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    const double a = fabs((double)y);
    int best = 0;
    for (int c = 1; c <= 0x7E; ++c) {
        const double dc = fabs(oracle_e4m3_value((uint8_t)c) - a), db = fabs(oracle_e4m3_value((uint8_t)best) - a);
        if (dc < db || (dc == db && (c & 1) == 0 && (best & 1) == 1)) best = c;
    }
    return (uint8_t)(sign | best);
}

/* Slot-mapped append into FP8 pools: pool code = encode(fp32(x / scale)) (x fp32, or bf16 bits when dtype = 1). */
int oracle_reshape_and_cache_fp8(int dtype, const void* k_new, const void* v_new, uint8_t* k_pool,
                                 uint8_t* v_pool, const int64_t* slots, int32_t num_tokens, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t block_size, int32_t num_blocks, float k_scale,
                                 float v_scale) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORACLE_BAD_ARG;
    for (int32_t i = 0; i < num_tokens; ++i) {
        const int64_t s = slots[i];
        if (s < 0) continue;
        if (s >= (int64_t)num_blocks * block_size) return ORACLE_BAD_SLOT;
        const int64_t blk = s / block_size, off = s % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h)
            for (int32_t d = 0; d < head_dim; ++d) {
                const size_t src = ((size_t)i * num_kv_heads + h) * head_dim + d;
                const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * head_dim + d;
                k_pool[dst] = oracle_e4m3_encode((float)load_elem(dtype, k_new, src) / k_scale);
                v_pool[dst] = oracle_e4m3_encode((float)load_elem(dtype, v_new, src) / v_scale);
            }
    }
    return ORACLE_OK;
}

/* Decode attention over FP8 pools: the decode definition above with K^ = value * k_scale, V^ = value * v_scale. */
int oracle_decode_attention_fp8(int q_dtype, const void* q, const uint8_t* k_pool, const uint8_t* v_pool,
                                float k_scale, float v_scale, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int32_t num_blocks, double scale,
                                int32_t seq_begin, int32_t seq_end, double* out) {
    int rc = check_common(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, seq_begin, seq_end);
    if (rc) return rc;
    /* each code's value times its pool's scale, in double (exact: a 4-bit significand times an fp32
       scale), then the definition; the values are widened per sequence as the definition reads them */
    return decode_impl(q_dtype, q, 3, k_pool, v_pool, (double)k_scale, (double)v_scale, block_tables,
                       max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, scale, seq_begin, seq_end, out);
}

/* Element-wise forms for the tests: out[i] = encode(x[i]); val[i] = value(codes[i]). */
void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}
void oracle_e4m3_value_array(const uint8_t* codes, int64_t n, double* val) {
    for (int64_t i = 0; i < n; ++i) val[i] = oracle_e4m3_value(codes[i]);
}
