/*
 * Paged-KV-cache attention oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded float64 restatement of what the paged attention
 * path computes.  Only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg may load this file; the library under paged_kv_cache_99_gb300/
 * never does, and the two share no code, header, table or helper.
 *
 * Sources (web pages; cited by title and section):
 *   [P1] "Basics of LLM Inference and vLLM Internals: KV Cache, PagedAttention,
 *        and Scheduler" (ttlab.hopto.org), sections 2, 4, 6.
 *   [P2] drpranayjha.com, Red Hat AI Inference Server part, section
 *        "How PagedAttention pages the KV cache".
 *   [P3] "The Memory Trick Behind Fast LLM Serving" (tarundecipher.com),
 *        sections "PagedAttention changes the shape of the problem" and
 *        "Batching does not merge the conversations".
 *
 * What the pages fix, restated:
 *   - attention at a new token revisits the keys and values of every preceding
 *     token of the same request [P1 s.2];
 *   - K/V are stored in fixed blocks of 16 tokens; a per-request block table maps
 *     logical block j to a physical block anywhere in the pool; only the tail of
 *     the last block is unused [P1 s.4][P2][P3];
 *   - several tables may name the same physical block (shared prefix) [P1 s.4][P2];
 *   - GQA: query heads are grouped, one K/V head per group [P1 s.2];
 *   - FP8 cache stores one byte per element [P1 s.2, s.7];
 *   - a flattened batch keeps requests separate: no request attends to another [P3];
 *   - a prefill chunk is a slice of a prompt processed in one step while other
 *     requests decode [P1 s.6].
 * Readings where the pages are silent (layout, slot formula, grouping order,
 * causal positions of a chunk, FP8 encoding rule, empty sequences) are listed in
 * the repository's design notes and repeated next to each function below.
 *
 * Nothing here is blocked, fused or reordered: each output is the textbook
 *   softmax(scale * q . K^T) . V
 * over the gathered keys, computed in float64 with left-to-right sums.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Storage type codes used by the Python shim (same numbering is chosen freely
 * by the library; nothing is shared). */
#define OR_BF16 0
#define OR_FP16 1
#define OR_FP8_E4M3 2

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_RANGE 2
#define OR_ERR_NOMEM 3

/* ------------------------------------------------------------------------ */
/* Element formats, written from their bit-level definitions.               */
/* ------------------------------------------------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double or_bf16_to_double(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double or_fp16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1F;
    int m = bits & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return sign ? -v : v;
}

/* FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities, NaN = S.1111.111, largest finite 448, smallest subnormal 2^-9. */
double or_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) {
        v = ldexp((double)m, -9);
    } else {
        v = ldexp((double)(8 + m), e - 10);
    }
    return sign ? -v : v;
}

/* Round a binary32 value to E4M3 with round-to-nearest, ties to the even
 * mantissa, then clamp magnitudes above 448 to 448 ("satfinite").  NaN keeps its
 * sign and becomes S.1111.111; infinities saturate; -0 stays -0. */
uint8_t or_e4m3_encode(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint8_t)(sign | 0x7E);
    /* binade exponent k with 2^k <= a < 2^(k+1); below 2^-6 the grid is the
     * subnormal one, whose spacing equals that of the binade [2^-6, 2^-5). */
    int e2;
    frexp(a, &e2);
    int k = e2 - 1;
    if (k < -6) k = -6;
    double quantum = ldexp(1.0, k - 3);
    double r = a / quantum; /* exact: scaling by a power of two */
    double fl = floor(r);
    double frac = r - fl;
    double n;
    if (frac > 0.5) {
        n = fl + 1.0;
    } else if (frac < 0.5) {
        n = fl;
    } else {
        n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    }
    double v = n * quantum;
    if (v > 448.0) return (uint8_t)(sign | 0x7E);
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) {
        /* subnormal: v = m * 2^-9, m in 1..7 */
        int m = (int)(v / ldexp(1.0, -9));
        return (uint8_t)(sign | m);
    }
    int ev;
    frexp(v, &ev);
    int kv = ev - 1; /* 2^kv <= v < 2^(kv+1), kv in -6..8 */
    int mant = (int)(v / ldexp(1.0, kv - 3)) - 8;
    return (uint8_t)(sign | ((kv + 7) << 3) | mant);
}

/* The slot-write rule for one element: the quotient fl32(x) / scale (IEEE
 * binary32 division), rounded to E4M3 as above.  A NaN quotient takes the sign
 * of the source element x, so the code does not depend on how a platform
 * propagates NaN signs through division (reading; the pages do not cover NaN). */
uint8_t or_slot_code(float x, float scale) {
    float q = x / scale;
    if (isnan(q)) return (uint8_t)((signbit(x) ? 0x80 : 0x00) | 0x7F);
    return or_e4m3_encode(q);
}

static double or_load(const void* base, int64_t idx, int dtype) {
    switch (dtype) {
        case OR_BF16: return or_bf16_to_double(((const uint16_t*)base)[idx]);
        case OR_FP16: return or_fp16_to_double(((const uint16_t*)base)[idx]);
        case OR_FP8_E4M3: return or_e4m3_to_double(((const uint8_t*)base)[idx]);
        default: return NAN;
    }
}

/* ------------------------------------------------------------------------ */
/* Slot write (reshape_and_cache).                                          */
/* ------------------------------------------------------------------------ */

/*
 * For every new token t with slot s = slot_mapping[t] >= 0, copy its K and V
 * vectors of every KV head into the cache at physical block s / block_size,
 * offset s % block_size [P1 s.4][P3 "PagedAttention changes the shape"].
 * Cache layout [num_blocks][num_kv_heads][block_size][head_dim]; a negative slot
 * is padding and writes nothing (readings; the pages do not fix either).
 * A 16-bit cache receives the source bits unchanged (source and cache type must
 * then agree).  An FP8 cache receives or_slot_code(x, scale): e4m3(fl32(x) /
 * scale), the quotient rounded once to binary32, with separate K and V scales.
 * All other cache bytes are left untouched.  Returns OR_ERR_RANGE if a slot
 * lies beyond the pool (nothing is written for that token).
 */
int or_reshape_and_cache(const uint16_t* k, const uint16_t* v, int src_dtype,
                         void* k_cache, void* v_cache, int cache_dtype,
                         const int64_t* slot_mapping, int num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, float k_scale, float v_scale) {
    if (src_dtype != OR_BF16 && src_dtype != OR_FP16) return OR_ERR_ARG;
    if (cache_dtype != OR_FP8_E4M3 && cache_dtype != src_dtype) return OR_ERR_ARG;
    int status = OR_OK;
    int64_t pool_slots = (int64_t)num_blocks * block_size;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            status = OR_ERR_RANGE;
            continue;
        }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int i = 0; i < head_dim; ++i) {
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + i;
                int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim + i;
                if (cache_dtype == OR_FP8_E4M3) {
                    float xk = (float)or_load(k, src, src_dtype);
                    float xv = (float)or_load(v, src, src_dtype);
                    ((uint8_t*)k_cache)[dst] = or_slot_code(xk, k_scale);
                    ((uint8_t*)v_cache)[dst] = or_slot_code(xv, v_scale);
                } else {
                    ((uint16_t*)k_cache)[dst] = k[src];
                    ((uint16_t*)v_cache)[dst] = v[src];
                }
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Attention over the paged cache.                                          */
/* ------------------------------------------------------------------------ */

/*
 * Gather the first n tokens of sequence `seq`, KV head `kvh`, into contiguous
 * [n][head_dim] float64 arrays: token t lives in physical block
 * block_tables[seq][t / block_size] at offset t % block_size [P1 s.4 diagram:
 * logical block -> physical block].  FP8 elements are dequantised as
 * decode(c) * scale.
 */
static int or_gather(double* K, double* V, const void* k_cache, const void* v_cache,
                     int cache_dtype, double k_scale, double v_scale,
                     const int32_t* block_tables, int max_blocks_per_seq, int seq,
                     int n, int kvh, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks) {
    for (int t = 0; t < n; ++t) {
        int j = t / block_size;
        if (j >= max_blocks_per_seq) return OR_ERR_RANGE;
        int64_t phys = block_tables[(int64_t)seq * max_blocks_per_seq + j];
        if (phys < 0 || phys >= num_blocks) return OR_ERR_RANGE;
        int off = t % block_size;
        int64_t base = ((phys * num_kv_heads + kvh) * block_size + off) * head_dim;
        for (int i = 0; i < head_dim; ++i) {
            double kk = or_load(k_cache, base + i, cache_dtype);
            double vv = or_load(v_cache, base + i, cache_dtype);
            if (cache_dtype == OR_FP8_E4M3) {
                kk *= k_scale;
                vv *= v_scale;
            }
            K[(int64_t)t * head_dim + i] = kk;
            V[(int64_t)t * head_dim + i] = vv;
        }
    }
    return OR_OK;
}

/* softmax(scale * q . K[t] for t < nk) . V, with the maximum subtracted before
 * exponentiation; plain left-to-right float64 sums. */
static void or_attend_one(double* out, const double* q, const double* K, const double* V,
                          int nk, int head_dim, double scale, double* logits) {
    if (nk <= 0) {
        for (int i = 0; i < head_dim; ++i) out[i] = 0.0;
        return;
    }
    double mx = -INFINITY;
    for (int t = 0; t < nk; ++t) {
        double dot = 0.0;
        for (int i = 0; i < head_dim; ++i) dot += q[i] * K[(int64_t)t * head_dim + i];
        logits[t] = scale * dot;
        if (logits[t] > mx) mx = logits[t];
    }
    double z = 0.0;
    for (int t = 0; t < nk; ++t) {
        logits[t] = exp(logits[t] - mx);
        z += logits[t];
    }
    for (int i = 0; i < head_dim; ++i) {
        double acc = 0.0;
        for (int t = 0; t < nk; ++t) acc += logits[t] * V[(int64_t)t * head_dim + i];
        out[i] = acc / z;
    }
}

/*
 * Decode: one query token per sequence.  out[s][h][:] for query head h uses KV
 * head h / (num_q_heads / num_kv_heads) -- consecutive query heads form a group
 * (reading of GQA [P1 s.2]) -- and attends over all seq_lens[s] cached tokens
 * (reading: the cache already holds this step's token, written first).  An empty
 * sequence (seq_lens[s] == 0) yields zeros (reading).
 * q: [num_seqs][num_q_heads][head_dim] 16-bit bits of q_dtype.
 * out: [num_seqs][num_q_heads][head_dim] float64.
 */
int or_decode(double* out, const uint16_t* q, int q_dtype, const void* k_cache,
              const void* v_cache, int cache_dtype, double k_scale, double v_scale,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
              int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
              int block_size, int num_blocks, double scale) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return OR_ERR_ARG;
    int group = num_q_heads / num_kv_heads;
    int max_n = 0;
    for (int s = 0; s < num_seqs; ++s) {
        if (seq_lens[s] < 0) return OR_ERR_ARG;
        if (seq_lens[s] > max_n) max_n = seq_lens[s];
    }
    size_t kv_elems = (size_t)(max_n > 0 ? max_n : 1) * head_dim;
    double* K = (double*)malloc(kv_elems * sizeof(double));
    double* V = (double*)malloc(kv_elems * sizeof(double));
    double* logits = (double*)malloc((size_t)(max_n > 0 ? max_n : 1) * sizeof(double));
    double* qd = (double*)malloc((size_t)head_dim * sizeof(double));
    if (!K || !V || !logits || !qd) {
        free(K); free(V); free(logits); free(qd);
        return OR_ERR_NOMEM;
    }
    int status = OR_OK;
    for (int s = 0; s < num_seqs && status == OR_OK; ++s) {
        int n = seq_lens[s];
        for (int kvh = 0; kvh < num_kv_heads && status == OR_OK; ++kvh) {
            status = or_gather(K, V, k_cache, v_cache, cache_dtype, k_scale, v_scale,
                               block_tables, max_blocks_per_seq, s, n, kvh, num_kv_heads,
                               head_dim, block_size, num_blocks);
            if (status != OR_OK) break;
            for (int g = 0; g < group; ++g) {
                int h = kvh * group + g;
                int64_t row = ((int64_t)s * num_q_heads + h) * head_dim;
                for (int i = 0; i < head_dim; ++i) qd[i] = or_load(q, row + i, q_dtype);
                or_attend_one(out + row, qd, K, V, n, head_dim, scale, logits);
            }
        }
    }
    free(K); free(V); free(logits); free(qd);
    return status;
}

/*
 * Mixed batch: the query rows of all sequences are flattened into one array,
 * sequence s owning rows query_start_loc[s] .. query_start_loc[s+1]-1 [P3
 * "Batching does not merge the conversations"].  A sequence with q_len = 1 is a
 * decode row; a longer one is a prefill chunk [P1 s.6].  seq_lens[s] counts the
 * cached tokens including this step's q_len new ones, so chunk row j sits at
 * absolute position seq_lens[s] - q_len + j and attends causally to keys
 * 0 .. that position (reading: tokens are processed so that the computed count
 * catches up with the total count [P1 s.3]).
 * q/out: [total_q][num_q_heads][head_dim].
 */
int or_mixed(double* out, const uint16_t* q, int q_dtype, const int32_t* query_start_loc,
             const void* k_cache, const void* v_cache, int cache_dtype, double k_scale,
             double v_scale, const int32_t* block_tables, int max_blocks_per_seq,
             const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
             int head_dim, int block_size, int num_blocks, double scale) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return OR_ERR_ARG;
    int group = num_q_heads / num_kv_heads;
    int max_n = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int q_len = query_start_loc[s + 1] - query_start_loc[s];
        if (q_len < 0 || seq_lens[s] < q_len) return OR_ERR_ARG;
        if (seq_lens[s] > max_n) max_n = seq_lens[s];
    }
    size_t kv_elems = (size_t)(max_n > 0 ? max_n : 1) * head_dim;
    double* K = (double*)malloc(kv_elems * sizeof(double));
    double* V = (double*)malloc(kv_elems * sizeof(double));
    double* logits = (double*)malloc((size_t)(max_n > 0 ? max_n : 1) * sizeof(double));
    double* qd = (double*)malloc((size_t)head_dim * sizeof(double));
    if (!K || !V || !logits || !qd) {
        free(K); free(V); free(logits); free(qd);
        return OR_ERR_NOMEM;
    }
    int status = OR_OK;
    for (int s = 0; s < num_seqs && status == OR_OK; ++s) {
        int n = seq_lens[s];
        int q0 = query_start_loc[s];
        int q_len = query_start_loc[s + 1] - q0;
        if (q_len == 0) continue;
        for (int kvh = 0; kvh < num_kv_heads && status == OR_OK; ++kvh) {
            status = or_gather(K, V, k_cache, v_cache, cache_dtype, k_scale, v_scale,
                               block_tables, max_blocks_per_seq, s, n, kvh, num_kv_heads,
                               head_dim, block_size, num_blocks);
            if (status != OR_OK) break;
            for (int j = 0; j < q_len; ++j) {
                int pos = n - q_len + j;
                for (int g = 0; g < group; ++g) {
                    int h = kvh * group + g;
                    int64_t row = ((int64_t)(q0 + j) * num_q_heads + h) * head_dim;
                    for (int i = 0; i < head_dim; ++i) qd[i] = or_load(q, row + i, q_dtype);
                    or_attend_one(out + row, qd, K, V, pos + 1, head_dim, scale, logits);
                }
            }
        }
    }
    free(K); free(V); free(logits); free(qd);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Array forms of the element conversions (used by the tests' pins).        */
/* ------------------------------------------------------------------------ */

void or_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_encode(x[i]);
}

/* e4m3(fl32(x) / scale) for 16-bit source bits, the exact rule of the slot write. */
void or_quantize_array(const uint16_t* x, int src_dtype, float scale, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        float xf = (float)or_load(x, i, src_dtype);
        out[i] = or_slot_code(xf, scale);
    }
}

void or_decode_array(const void* x, int dtype, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_load(x, i, dtype);
}
