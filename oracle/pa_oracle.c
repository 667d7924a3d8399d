/*
 * pa_oracle.c -- fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers of this library. The
 * product path (the CUDA library under paged_kv_decode_18_gb300/) never
 * links, loads or calls it, and the two share no code, header, table or
 * helper. Everything here is deliberately plain and slow: scalar loops, fp64
 * arithmetic, no tiling, no fusion, no reordering beyond the definitions.
 *
 * What it computes, and where the definitions come from:
 *
 *   Cache write ("S06/S11" of the course README "Build an LLM Inference Engine
 *   From Scratch", section "The code asserts its own claims"; and the
 *   "KV Cache > The Idea" section of the LLM inference engine work-log,
 *   shehab-ashraf.github.io/posts/llm-inference): every new token's K and V
 *   rows are stored once, at the physical slot its block manager handed out.
 *   A slot is phys_block * block_size + offset_in_block. Negative slot = skip.
 *
 *   Attention (same work-log section, "Decode: ... this single Q attends over
 *   the whole history"; course README curriculum row "Memory & KV Cache":
 *   PagedAttention, GQA): for sequence s, query token j and query head h,
 *     K_s[p] = k_cache[block_tables[s][p / BS]][h / G][p % BS][:]  (V alike)
 *     pos(j) = c_s - Lq_s + j        (the query's own position in the context)
 *     z_p    = scale * <q[j,h], K_s[p]>   for 0 <= p <= pos(j) (causal), or
 *              for 0 <= p < c_s (non-causal)
 *     M = max z, L = sum exp(z - M), out = sum exp(z - M) V_s[p] / L,
 *     lse = M + ln L.
 *   This is the plain two-pass softmax attention over the gathered context.
 *
 *   Split-K merge (course README, "s12: online softmax is exact; paged and
 *   split-K variants agree"): given P partial results (o_i, lse_i) over
 *   disjoint key ranges, LSE = M + ln sum_i exp(lse_i - M) with M = max lse_i,
 *   out = sum_i exp(lse_i - LSE) o_i. Partials with lse_i = -inf are empty.
 *
 *   Online softmax (course README, "S12 ... FlashAttention"; "online softmax is
 *   exact"): a second, independent attention routine that streams the keys in
 *   tiles with a running max and running sum. It exists only so the tests can
 *   check it against the two-pass routine.
 *
 *   INT8 KV rows (course README, curriculum row "Memory & KV Cache":
 *   quantization; the "INT8 KV" configuration; claim "s08": grouping keeps
 *   outliers in check). The pages fix no formula; the reading used here is
 *   the plainest one: symmetric quantisation with one group per (token, KV
 *   head) row of head_dim values, every step one IEEE fp32 operation:
 *     amax = max_d |x_d|;  amax == 0 -> all codes 0 and scale 0; else
 *     inv = 127 / amax,  code_d = clamp(rint(x_d * inv), -127, 127),
 *     scale = amax / 127   (rint: nearest, ties to even).
 *   A row dequantises to code_d * scale (exact in fp64). Attention over an
 *   int8 pool is the attention above over the dequantised rows.
 *
 *   FP8 KV rows (the same curriculum row names FP8 beside INT8; the format
 *   is the OCP 8-bit float E4M3: 1 sign, 4 exponent bits with bias 7, 3
 *   mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448).
 *   The plainest reading, as for INT8: one group per (token, KV head) row,
 *     amax = max_d |x_d|;  amax == 0 -> all codes 0 and scale 0; else
 *     inv = 448 / amax,  code_d = e4m3(x_d * inv),  scale = amax / 448,
 *   each one IEEE fp32 operation, where e4m3(y) is the finite E4M3 value
 *   nearest to y (ties to the even code, i.e. the even last mantissa bit)
 *   and |y| beyond 448 gives +-448. A row dequantises to value(code_d) *
 *   scale (exact in fp64).
 *
 * Numbers: bf16 inputs are bit patterns (uint16). They are widened to fp64
 * exactly (bf16 -> fp32 is a 16-bit shift; fp32 -> fp64 is exact).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_RANGE (-2)
#define ORACLE_ERR_NOMEM (-3)

/* bf16 bit pattern -> double, exactly. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_bits_to_float(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int pa_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Cache write: k_cache[slot / BS][h][slot % BS][:] = k[t][h][:] (V alike).  */
/* Byte copy; tokens with a negative slot are skipped. A slot beyond the pool */
/* is an error and nothing further is written.                               */
/* ------------------------------------------------------------------------ */
int pa_oracle_reshape_and_cache(const uint16_t *k, const uint16_t *v,
                                const int64_t *slot_mapping, int64_t num_tokens,
                                int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, uint16_t *k_cache,
                                uint16_t *v_cache) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0)
        return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) return ORACLE_ERR_RANGE;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t src = ((t * num_kv_heads) + h) * (int64_t)head_dim + d;
                int64_t dst = (((block * num_kv_heads) + h) * (int64_t)block_size + offset) *
                                  (int64_t)head_dim + d;
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* INT8 quantisation of one row of D bf16 values (rule in the header).       */
/* ------------------------------------------------------------------------ */
static void quantize_row_i8(const uint16_t *x, int D, int8_t *codes, float *scale) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(bf16_bits_to_float(x[d]));
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int d = 0; d < D; ++d) codes[d] = 0;
        *scale = 0.0f;
        return;
    }
    float inv = 127.0f / amax;
    for (int d = 0; d < D; ++d) {
        float t = rintf(bf16_bits_to_float(x[d]) * inv);
        if (t > 127.0f) t = 127.0f;
        if (t < -127.0f) t = -127.0f;
        codes[d] = (int8_t)t;
    }
    *scale = amax / 127.0f;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 codes (format and rule in the header).                           */
/* ------------------------------------------------------------------------ */
static double e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (c & 0x80) ? -v : v;
}

/* the finite E4M3 code nearest to y, ties to the even code, saturating at 448:
   a search over the 127 non-negative finite codes, in increasing order */
static uint8_t e4m3_code(float y) {
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    const double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double d = fabs(e4m3_value((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best_d = d;
            best = c;
        }
    }
    return (uint8_t)(sign | best);
}

int pa_oracle_e4m3_values(const uint8_t *codes, int64_t n, double *values) {
    if (n < 0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) values[i] = e4m3_value(codes[i]);
    return ORACLE_OK;
}

int pa_oracle_e4m3_codes(const float *y, int64_t n, uint8_t *codes) {
    if (n < 0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_code(y[i]);
    return ORACLE_OK;
}

static void quantize_row_f8(const uint16_t *x, int D, uint8_t *codes, float *scale) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(bf16_bits_to_float(x[d]));
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int d = 0; d < D; ++d) codes[d] = 0;
        *scale = 0.0f;
        return;
    }
    const float inv = 448.0f / amax;
    for (int d = 0; d < D; ++d) {
        const float y = bf16_bits_to_float(x[d]) * inv;
        codes[d] = e4m3_code(y);
    }
    *scale = amax / 448.0f;
}

/* rows [rows][D] bf16 -> codes [rows][D] e4m3, scales [rows] fp32 */
int pa_oracle_quantize_rows_f8(const uint16_t *x, int64_t rows, int D, uint8_t *codes,
                               float *scales) {
    if (rows < 0 || D <= 0) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r)
        quantize_row_f8(x + r * D, D, codes + r * D, scales + r);
    return ORACLE_OK;
}

/* Cache write into the fp8 pool, laid out as the int8 one. */
int pa_oracle_reshape_and_cache_f8(const uint16_t *k, const uint16_t *v,
                                   const int64_t *slot_mapping, int64_t num_tokens,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int64_t num_blocks, uint8_t *k_cache, uint8_t *v_cache,
                                   float *k_scale, float *v_scale) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0)
        return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) return ORACLE_ERR_RANGE;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = (t * num_kv_heads + h) * (int64_t)head_dim;
            int64_t row = (block * num_kv_heads + h) * (int64_t)block_size + offset;
            quantize_row_f8(k + src, head_dim, k_cache + row * head_dim, k_scale + row);
            quantize_row_f8(v + src, head_dim, v_cache + row * head_dim, v_scale + row);
        }
    }
    return ORACLE_OK;
}

/* rows [rows][D] bf16 -> codes [rows][D] int8, scales [rows] fp32 */
int pa_oracle_quantize_rows_i8(const uint16_t *x, int64_t rows, int D, int8_t *codes,
                               float *scales) {
    if (rows < 0 || D <= 0) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r)
        quantize_row_i8(x + r * D, D, codes + r * D, scales + r);
    return ORACLE_OK;
}

/* Cache write into the int8 pool: row k[t][h][:] is quantised into         */
/* k_cache[slot / BS][h][slot % BS][:] and k_scale[slot / BS][h][slot % BS]. */
int pa_oracle_reshape_and_cache_i8(const uint16_t *k, const uint16_t *v,
                                   const int64_t *slot_mapping, int64_t num_tokens,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int64_t num_blocks, int8_t *k_cache, int8_t *v_cache,
                                   float *k_scale, float *v_scale) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0)
        return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) return ORACLE_ERR_RANGE;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = (t * num_kv_heads + h) * (int64_t)head_dim;
            int64_t row = (block * num_kv_heads + h) * (int64_t)block_size + offset;
            quantize_row_i8(k + src, head_dim, k_cache + row * head_dim, k_scale + row);
            quantize_row_i8(v + src, head_dim, v_cache + row * head_dim, v_scale + row);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Two-pass softmax attention of one query over n dense fp64 keys/values.    */
/* n == 0 gives out = 0 and lse = -inf (softmax over nothing).               */
/* ------------------------------------------------------------------------ */
static void attend_two_pass(const double *q, const double *K, const double *V, int64_t n,
                            int D, double scale, double *z, double *out, double *lse) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    /* logits */
    for (int64_t p = 0; p < n; ++p) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * K[p * D + d];
        z[p] = scale * dot;
    }
    /* pass 1: max */
    double M = z[0];
    for (int64_t p = 1; p < n; ++p)
        if (z[p] > M) M = z[p];
    /* pass 2: normaliser and weighted sum of V */
    double L = 0.0;
    for (int64_t p = 0; p < n; ++p) {
        double w = exp(z[p] - M);
        L += w;
        for (int d = 0; d < D; ++d) out[d] += w * V[p * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= L;
    *lse = M + log(L);
}

/* Online softmax over the same inputs: keys streamed in tiles of `tile`,  */
/* with a running max m, running sum l and a rescaled accumulator.         */
static void attend_online(const double *q, const double *K, const double *V, int64_t n, int D,
                          double scale, int64_t tile, double *acc, double *out, double *lse) {
    double m = -INFINITY, l = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int64_t t0 = 0; t0 < n; t0 += tile) {
        int64_t t1 = t0 + tile < n ? t0 + tile : n;
        double tile_max = -INFINITY;
        for (int64_t p = t0; p < t1; ++p) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q[d] * K[p * D + d];
            double s = scale * dot;
            if (s > tile_max) tile_max = s;
        }
        double m_new = m > tile_max ? m : tile_max;
        double alpha = exp(m - m_new); /* m = -inf on the first tile: alpha = 0 */
        l *= alpha;
        for (int d = 0; d < D; ++d) acc[d] *= alpha;
        for (int64_t p = t0; p < t1; ++p) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q[d] * K[p * D + d];
            double w = exp(scale * dot - m_new);
            l += w;
            for (int d = 0; d < D; ++d) acc[d] += w * V[p * D + d];
        }
        m = m_new;
    }
    if (n == 0) {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    for (int d = 0; d < D; ++d) out[d] = acc[d] / l;
    *lse = m + log(l);
}

/* ------------------------------------------------------------------------ */
/* Dense attention over contiguous bf16 keys/values, one query vector.       */
/*   q: [D] bf16, K/V: [n, D] bf16 rows (row stride D).                      */
/*   mode 0 = two-pass, mode 1 = online with the given tile.                 */
/* ------------------------------------------------------------------------ */
int pa_oracle_attention_dense(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                              int64_t n, int D, double scale, int mode, int64_t tile,
                              double *out, double *lse) {
    if (n < 0 || D <= 0 || (mode == 1 && tile <= 0)) return ORACLE_ERR_ARG;
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *Kd = (double *)malloc(sizeof(double) * (size_t)(n * D + 1));
    double *Vd = (double *)malloc(sizeof(double) * (size_t)(n * D + 1));
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(n > D ? n + 1 : D + 1));
    if (!qd || !Kd || !Vd || !tmp) {
        free(qd); free(Kd); free(Vd); free(tmp);
        return ORACLE_ERR_NOMEM;
    }
    for (int d = 0; d < D; ++d) qd[d] = bf16_bits_to_double(q[d]);
    for (int64_t i = 0; i < n * D; ++i) {
        Kd[i] = bf16_bits_to_double(K[i]);
        Vd[i] = bf16_bits_to_double(V[i]);
    }
    if (mode == 0)
        attend_two_pass(qd, Kd, Vd, n, D, scale, tmp, out, lse);
    else
        attend_online(qd, Kd, Vd, n, D, scale, tile, tmp, out, lse);
    free(qd); free(Kd); free(Vd); free(tmp);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Paged attention. Shapes:                                                  */
/*   q            [Tq, Hq, D] bf16, Tq = cu_seqlens_q[S]                     */
/*   k/v_cache    [num_blocks, Hkv, BS, D] bf16                              */
/*   block_tables [S, max_blocks] int32                                      */
/*   context_lens [S] int32 (includes the sequence's own query tokens)       */
/*   cu_seqlens_q [S + 1] int32 (row offsets of each sequence's queries)     */
/*   out          [Tq, Hq, D] fp64;  lse [Tq, Hq] fp64 (natural log)         */
/* Query head h reads KV head h / (Hq / Hkv).                                */
/* mode 0 = two-pass (the oracle proper); mode 1 = online with `tile` keys.  */
/* ------------------------------------------------------------------------ */
/* Pool element formats: bf16 (k16/v16) or int8 rows with one scale per row. */
static int paged_attention_core(const uint16_t *q, const uint16_t *k16, const uint16_t *v16,
                                const int8_t *k8, const int8_t *v8, int f8, const float *k_scale,
                                const float *v_scale, const int32_t *block_tables,
                                const int32_t *context_lens, const int32_t *cu_seqlens_q,
                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                double scale, int causal, int mode, int64_t tile,
                                int num_threads, double *out, double *lse) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq < 0 || num_q_heads % num_kv_heads != 0 ||
        (mode == 1 && tile <= 0))
        return ORACLE_ERR_ARG;
    const int G = num_q_heads / num_kv_heads;
    const int D = head_dim;
    /* argument checks first, so the parallel loop cannot fail half way */
    for (int s = 0; s < num_seqs; ++s) {
        int c = context_lens[s];
        int lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        /* causal: the window cannot be longer than the context; non-causal
           queries see the whole (non-empty) context */
        if (c < 0 || lq < 0 || (lq > c && (causal || c == 0)) ||
            c > max_blocks_per_seq * block_size)
            return ORACLE_ERR_RANGE;
        int nb = (c + block_size - 1) / block_size;
        for (int b = 0; b < nb; ++b) {
            int32_t phys = block_tables[(int64_t)s * max_blocks_per_seq + b];
            if (phys < 0 || phys >= num_blocks) return ORACLE_ERR_RANGE;
        }
    }
    const int64_t pairs = (int64_t)num_seqs * num_kv_heads;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t pr = 0; pr < pairs; ++pr) {
        const int s = (int)(pr / num_kv_heads);
        const int kvh = (int)(pr % num_kv_heads);
        const int64_t c = context_lens[s];
        const int64_t q0 = cu_seqlens_q[s];
        const int64_t lq = cu_seqlens_q[s + 1] - q0;
        if (lq == 0) continue;
        double *K = (double *)malloc(sizeof(double) * (size_t)(c * D + 1));
        double *V = (double *)malloc(sizeof(double) * (size_t)(c * D + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *tmp = (double *)malloc(sizeof(double) * (size_t)(c > D ? c + 1 : D + 1));
        if (!K || !V || !qd || !tmp) {
            free(K); free(V); free(qd); free(tmp);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
            continue;
        }
        /* gather this sequence's context for KV head kvh, in position order */
        for (int64_t p = 0; p < c; ++p) {
            int64_t phys = block_tables[(int64_t)s * max_blocks_per_seq + p / block_size];
            int64_t srow = (phys * num_kv_heads + kvh) * block_size + p % block_size;
            int64_t row = srow * D;
            for (int d = 0; d < D; ++d) {
                if (k16) {
                    K[p * D + d] = bf16_bits_to_double(k16[row + d]);
                    V[p * D + d] = bf16_bits_to_double(v16[row + d]);
                } else if (f8) {  /* dequantised fp8 row: value(code) * scale */
                    K[p * D + d] = e4m3_value((uint8_t)k8[row + d]) * (double)k_scale[srow];
                    V[p * D + d] = e4m3_value((uint8_t)v8[row + d]) * (double)v_scale[srow];
                } else {  /* dequantised int8 row: code * scale, exact in fp64 */
                    K[p * D + d] = (double)k8[row + d] * (double)k_scale[srow];
                    V[p * D + d] = (double)v8[row + d] * (double)v_scale[srow];
                }
            }
        }
        for (int g = 0; g < G; ++g) {
            const int h = kvh * G + g;
            for (int64_t j = 0; j < lq; ++j) {
                const int64_t row = q0 + j;
                const int64_t pos = c - lq + j;          /* this query's position */
                const int64_t n = causal ? pos + 1 : c;  /* keys it may see */
                for (int d = 0; d < D; ++d)
                    qd[d] = bf16_bits_to_double(q[(row * num_q_heads + h) * (int64_t)D + d]);
                double *o = out + (row * num_q_heads + h) * (int64_t)D;
                double *l = lse + row * num_q_heads + h;
                if (mode == 0)
                    attend_two_pass(qd, K, V, n, D, scale, tmp, o, l);
                else
                    attend_online(qd, K, V, n, D, scale, tile, tmp, o, l);
            }
        }
        free(K); free(V); free(qd); free(tmp);
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

int pa_oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *block_tables,
                              const int32_t *context_lens, const int32_t *cu_seqlens_q,
                              int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_blocks_per_seq, int64_t num_blocks,
                              double scale, int causal, int mode, int64_t tile,
                              int num_threads, double *out, double *lse) {
    return paged_attention_core(q, k_cache, v_cache, NULL, NULL, 0, NULL, NULL, block_tables,
                                context_lens, cu_seqlens_q, num_seqs, num_q_heads,
                                num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                num_blocks, scale, causal, mode, tile, num_threads, out, lse);
}

/* Paged attention over an int8 pool (rows dequantised as code * scale). */
int pa_oracle_paged_attention_i8(const uint16_t *q, const int8_t *k_cache,
                                 const int8_t *v_cache, const float *k_scale,
                                 const float *v_scale, const int32_t *block_tables,
                                 const int32_t *context_lens, const int32_t *cu_seqlens_q,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                 double scale, int causal, int num_threads, double *out,
                                 double *lse) {
    if (!k_cache || !v_cache || !k_scale || !v_scale) return ORACLE_ERR_ARG;
    return paged_attention_core(q, NULL, NULL, k_cache, v_cache, 0, k_scale, v_scale,
                                block_tables, context_lens, cu_seqlens_q, num_seqs,
                                num_q_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, num_blocks, scale, causal, 0, 0,
                                num_threads, out, lse);
}

/* Paged attention over an fp8 pool (rows dequantised as value(code) * scale). */
int pa_oracle_paged_attention_f8(const uint16_t *q, const uint8_t *k_cache,
                                 const uint8_t *v_cache, const float *k_scale,
                                 const float *v_scale, const int32_t *block_tables,
                                 const int32_t *context_lens, const int32_t *cu_seqlens_q,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                 double scale, int causal, int num_threads, double *out,
                                 double *lse) {
    if (!k_cache || !v_cache || !k_scale || !v_scale) return ORACLE_ERR_ARG;
    return paged_attention_core(q, NULL, NULL, (const int8_t *)k_cache,
                                (const int8_t *)v_cache, 1, k_scale, v_scale, block_tables,
                                context_lens, cu_seqlens_q, num_seqs, num_q_heads,
                                num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                num_blocks, scale, causal, 0, 0, num_threads, out, lse);
}

/* ------------------------------------------------------------------------ */
/* Split-K merge of P partials per row.                                      */
/*   part_out [rows, P, D] fp64, part_lse [rows, P] fp64 -> out [rows, D],   */
/*   lse [rows]. Rows whose partials are all empty give 0 and -inf.          */
/* ------------------------------------------------------------------------ */
int pa_oracle_splitk_merge(const double *part_out, const double *part_lse, int64_t rows,
                           int P, int D, double *out, double *lse) {
    if (rows < 0 || P <= 0 || D <= 0) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const double *li = part_lse + r * P;
        double M = -INFINITY;
        for (int i = 0; i < P; ++i)
            if (li[i] > M) M = li[i];
        double *o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int i = 0; i < P; ++i) sum += exp(li[i] - M);
        const double LSE = M + log(sum);
        for (int i = 0; i < P; ++i) {
            double w = exp(li[i] - LSE);
            const double *oi = part_out + (r * P + i) * (int64_t)D;
            for (int d = 0; d < D; ++d) o[d] += w * oi[d];
        }
        lse[r] = LSE;
    }
    return ORACLE_OK;
}
