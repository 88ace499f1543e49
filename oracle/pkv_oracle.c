/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for paged KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; it exists so the tests, the smoke check and the CPU
 * baseline of the benchmark have an independent definition to compare the
 * CUDA kernels against.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (sources are the pages' titles and sections):
 *   - "PagedAttention" (deepconcepts.dev), sections "PagedAttention" (the
 *     per-sequence block table maps logical block n to a physical block) and
 *     the closing note on FlashAttention (paged attention is numerically
 *     exact attention; splitting the softmax sum over blocks and recombining
 *     it does not change the result).
 *   - "Paged attention" (danielfleming.xyz), section "What changed": decode
 *     touches, for each row, just the blocks named in the row's table, up to
 *     the row's true length.
 *   - "SLM paged attention" (aicassindra.com), section "The architecture":
 *     a row's table turns a logical block index (position / block_size) into
 *     a physical block id, and a slot count says how far the final block is
 *     filled.
 *
 * So the oracle is the plain definition of attention over a row's tokens in
 * logical order, in double precision:
 *     K_t = k_pool[table[r][t / bs]][t % bs][kvh][:]      t in [0, L_r)
 *     s_t = scale * sum_d q[r][h][d] * K_t[d]
 *     o[r][h][:] = sum_t softmax(s)_t * V_t[:]
 * with kvh = h / (q_heads / kv_heads) (contiguous query-head groups).
 *
 * Readings taken where the pages are silent:
 *   - seq_len == 0 gives an all-zero output row.
 *   - table entries past ceil(L/bs) are never read; an entry that is read and
 *     lies outside [0, num_blocks) is an error (return code ORACLE_BAD_TABLE).
 *   - no causal mask inside a row (the query is the newest position), no
 *     window, no bias.
 *
 * fp16 inputs are passed as raw IEEE binary16 bit patterns (uint16) and
 * widened exactly to double by oracle_half_to_double, written from the
 * binary16 definition.  Results are double.
 *
 * Threading: the (row, q-head) loop may run on several OpenMP threads
 * (num_threads > 1); each output element is still computed by one thread in
 * the same order, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_TABLE 5
#define ORACLE_NO_MEMORY 6

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  exponent 0 = zero/subnormal (fraction * 2^-24), exponent 31 =
 * infinity (fraction 0) or NaN. */
double oracle_half_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac + 1024), expo - 25);
    }
    return sign ? -v : v;
}

void oracle_half_array_to_double(double* dst, const uint16_t* src, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_half_to_double(src[i]);
}

static int64_t idx4(int64_t a, int64_t b, int64_t c, int64_t d,
                    int64_t nb, int64_t nc, int64_t nd) {
    return ((a * nb + b) * nc + c) * nd + d;
}

/* Attention of one query vector over n key/value vectors given by pointer
 * lists.  out[d] = sum_t exp(s_t - max s) V_t[d] / sum_t exp(s_t - max s). */
static void attend_one(double* out, const uint16_t* qv, const uint16_t* const* kp,
                       const uint16_t* const* vp, int n, int head_dim,
                       double scale, double* s) {
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (n == 0) return;
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
            acc += oracle_half_to_double(qv[d]) * oracle_half_to_double(kp[t][d]);
        s[t] = scale * acc;
        if (s[t] > m) m = s[t];
    }
    double z = 0.0;
    for (int t = 0; t < n; ++t) {
        s[t] = exp(s[t] - m);
        z += s[t];
    }
    for (int t = 0; t < n; ++t) {
        const double w = s[t] / z;
        for (int d = 0; d < head_dim; ++d)
            out[d] += w * oracle_half_to_double(vp[t][d]);
    }
}

static int check_heads(int q_heads, int kv_heads, int head_dim) {
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0) return 0;
    if (q_heads % kv_heads) return 0;
    return 1;
}

static void set_threads(int num_threads) {
#ifdef _OPENMP
    omp_set_num_threads(num_threads > 0 ? num_threads : 1);
#else
    (void)num_threads;
#endif
}

/*
 * Paged decode: out[rows][q_heads][head_dim] (double).
 * q: [rows][q_heads][head_dim] fp16 bits.
 * k_pool, v_pool: [num_blocks][block_size][kv_heads][head_dim] fp16 bits.
 * block_tables: [rows][max_blocks_per_row] int32.  seq_lens: [rows].
 */
int oracle_paged_decode(double* out, const uint16_t* q, const uint16_t* k_pool,
                        const uint16_t* v_pool, const int32_t* block_tables,
                        const int32_t* seq_lens, int rows, int q_heads,
                        int kv_heads, int head_dim, int block_size, double scale,
                        int max_blocks_per_row, int num_blocks, int num_threads) {
    if (!check_heads(q_heads, kv_heads, head_dim) || block_size <= 0 || rows < 0)
        return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        const int L = seq_lens[r];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks_per_row * block_size)
            return ORACLE_BAD_ARG;
        for (int lb = 0; lb < (L + block_size - 1) / block_size; ++lb) {
            const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + lb];
            if (pb < 0 || pb >= num_blocks) return ORACLE_BAD_TABLE;
        }
    }
    const int group = q_heads / kv_heads;
    int failed = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < q_heads; ++h) {
            const int L = seq_lens[r];
            const int kvh = h / group;
            const uint16_t** kp = (const uint16_t**)malloc(sizeof(void*) * (L + 1));
            const uint16_t** vp = (const uint16_t**)malloc(sizeof(void*) * (L + 1));
            double* s = (double*)malloc(sizeof(double) * (L + 1));
            if (!kp || !vp || !s) {
#pragma omp atomic write
                failed = 1;
            } else {
                for (int t = 0; t < L; ++t) {
                    const int64_t pb = block_tables[(int64_t)r * max_blocks_per_row + t / block_size];
                    const int64_t off = idx4(pb, t % block_size, kvh, 0, block_size, kv_heads, head_dim);
                    kp[t] = k_pool + off;
                    vp[t] = v_pool + off;
                }
                attend_one(out + ((int64_t)r * q_heads + h) * head_dim,
                           q + ((int64_t)r * q_heads + h) * head_dim, kp, vp, L,
                           head_dim, scale, s);
            }
            free(kp);
            free(vp);
            free(s);
        }
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Contiguous decode over a padded slab, the layout the paged cache replaced
 * ("Continuous batching", section "What changed": every row owns a slot as
 * wide as the widest row).  k_slab, v_slab: [rows][width][kv_heads][head_dim]; row r uses its
 * first seq_lens[r] tokens.
 */
int oracle_contiguous_decode(double* out, const uint16_t* q, const uint16_t* k_slab,
                             const uint16_t* v_slab, const int32_t* seq_lens,
                             int rows, int width, int q_heads, int kv_heads,
                             int head_dim, double scale, int num_threads) {
    if (!check_heads(q_heads, kv_heads, head_dim) || width < 0 || rows < 0)
        return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r)
        if (seq_lens[r] < 0 || seq_lens[r] > width) return ORACLE_BAD_ARG;
    const int group = q_heads / kv_heads;
    int failed = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < q_heads; ++h) {
            const int L = seq_lens[r];
            const int kvh = h / group;
            const uint16_t** kp = (const uint16_t**)malloc(sizeof(void*) * (L + 1));
            const uint16_t** vp = (const uint16_t**)malloc(sizeof(void*) * (L + 1));
            double* s = (double*)malloc(sizeof(double) * (L + 1));
            if (!kp || !vp || !s) {
#pragma omp atomic write
                failed = 1;
            } else {
                for (int t = 0; t < L; ++t) {
                    const int64_t off = idx4(r, t, kvh, 0, width, kv_heads, head_dim);
                    kp[t] = k_slab + off;
                    vp[t] = v_slab + off;
                }
                attend_one(out + ((int64_t)r * q_heads + h) * head_dim,
                           q + ((int64_t)r * q_heads + h) * head_dim, kp, vp, L,
                           head_dim, scale, s);
            }
            free(kp);
            free(vp);
            free(s);
        }
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Blockwise decode: the softmax sum of each row is cut into chunks of
 * chunk_tokens logical tokens; each chunk c yields its normalised partial
 * output o_c and its log-sum-exp lse_c = m_c + ln(sum_{t in c} exp(s_t - m_c));
 * the chunks are then combined:
 *     lse = M + ln sum_c exp(lse_c - M),  M = max_c lse_c
 *     o   = sum_c exp(lse_c - lse) * o_c
 * This is the exact block-wise rescaling the "PagedAttention" page's note on
 * FlashAttention describes; it must agree with oracle_paged_decode to
 * rounding.  lse_out (nullable) receives lse per (row, head); for L == 0 it
 * is -inf.
 */
int oracle_blockwise_decode(double* out, double* lse_out, const uint16_t* q,
                            const uint16_t* k_pool, const uint16_t* v_pool,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            int rows, int q_heads, int kv_heads, int head_dim,
                            int block_size, double scale, int max_blocks_per_row,
                            int num_blocks, int chunk_tokens) {
    if (!check_heads(q_heads, kv_heads, head_dim) || block_size <= 0 || chunk_tokens <= 0)
        return ORACLE_BAD_ARG;
    const int group = q_heads / kv_heads;
    for (int r = 0; r < rows; ++r) {
        const int L = seq_lens[r];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks_per_row * block_size)
            return ORACLE_BAD_ARG;
        const int nchunk = (L + chunk_tokens - 1) / chunk_tokens;
        for (int h = 0; h < q_heads; ++h) {
            const int kvh = h / group;
            const uint16_t* qv = q + ((int64_t)r * q_heads + h) * head_dim;
            double* o = out + ((int64_t)r * q_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            double* oc = (double*)calloc((size_t)(nchunk ? nchunk : 1) * head_dim, sizeof(double));
            double* lc = (double*)calloc((size_t)(nchunk ? nchunk : 1), sizeof(double));
            double* s = (double*)calloc((size_t)chunk_tokens, sizeof(double));
            if (!oc || !lc || !s) {
                free(oc); free(lc); free(s);
                return ORACLE_NO_MEMORY;
            }
            for (int c = 0; c < nchunk; ++c) {
                const int t0 = c * chunk_tokens;
                const int t1 = (t0 + chunk_tokens < L) ? t0 + chunk_tokens : L;
                double m = -INFINITY;
                for (int t = t0; t < t1; ++t) {
                    const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + t / block_size];
                    if (pb < 0 || pb >= num_blocks) {
                        free(oc); free(lc); free(s);
                        return ORACLE_BAD_TABLE;
                    }
                    const uint16_t* kv = k_pool + idx4(pb, t % block_size, kvh, 0, block_size, kv_heads, head_dim);
                    double acc = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        acc += oracle_half_to_double(qv[d]) * oracle_half_to_double(kv[d]);
                    s[t - t0] = scale * acc;
                    if (s[t - t0] > m) m = s[t - t0];
                }
                double z = 0.0;
                for (int t = t0; t < t1; ++t) {
                    s[t - t0] = exp(s[t - t0] - m);
                    z += s[t - t0];
                }
                for (int t = t0; t < t1; ++t) {
                    const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + t / block_size];
                    const uint16_t* vv = v_pool + idx4(pb, t % block_size, kvh, 0, block_size, kv_heads, head_dim);
                    for (int d = 0; d < head_dim; ++d)
                        oc[(int64_t)c * head_dim + d] += (s[t - t0] / z) * oracle_half_to_double(vv[d]);
                }
                lc[c] = m + log(z);
            }
            double M = -INFINITY;
            for (int c = 0; c < nchunk; ++c) if (lc[c] > M) M = lc[c];
            double lse = -INFINITY;
            if (nchunk > 0) {
                double z = 0.0;
                for (int c = 0; c < nchunk; ++c) z += exp(lc[c] - M);
                lse = M + log(z);
                for (int c = 0; c < nchunk; ++c) {
                    const double w = exp(lc[c] - lse);
                    for (int d = 0; d < head_dim; ++d) o[d] += w * oc[(int64_t)c * head_dim + d];
                }
            }
            if (lse_out) lse_out[(int64_t)r * q_heads + h] = lse;
            free(oc); free(lc); free(s);
        }
    }
    return ORACLE_OK;
}

/*
 * Append: for each row r with positions[r] >= 0, the new token's K and V go
 * to slot (pos % bs) of physical block table[r][pos / bs], for every KV head
 * ("SLM paged attention", section "The architecture": a row's table
 * turns position / block_size into a physical block, and the final block
 * takes one slot after another).  Operates in place on k_pool / v_pool, as a plain copy of
 * the fp16 bit patterns.  Rows with a negative position are skipped.
 */
int oracle_paged_append(uint16_t* k_pool, uint16_t* v_pool, const int32_t* block_tables,
                        const int32_t* positions, const uint16_t* k_new,
                        const uint16_t* v_new, int rows, int kv_heads, int head_dim,
                        int block_size, int max_blocks_per_row, int num_blocks) {
    if (kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || rows < 0) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        const int pos = positions[r];
        if (pos < 0) continue;
        const int lb = pos / block_size;
        if (lb >= max_blocks_per_row) return ORACLE_BAD_TABLE;
        const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + lb];
        if (pb < 0 || pb >= num_blocks) return ORACLE_BAD_TABLE;
    }
    for (int r = 0; r < rows; ++r) {
        const int pos = positions[r];
        if (pos < 0) continue;
        const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + pos / block_size];
        for (int h = 0; h < kv_heads; ++h) {
            const int64_t dst = idx4(pb, pos % block_size, h, 0, block_size, kv_heads, head_dim);
            const int64_t src = ((int64_t)r * kv_heads + h) * head_dim;
            memcpy(k_pool + dst, k_new + src, sizeof(uint16_t) * (size_t)head_dim);
            memcpy(v_pool + dst, v_new + src, sizeof(uint16_t) * (size_t)head_dim);
        }
    }
    return ORACLE_OK;
}

/*
 * Copy-on-write block copy: for i < n, block dst_ids[i] of both pools becomes
 * a byte copy of block src_ids[i] ("SLM paged attention", section "The
 * architecture": a writer about to modify a shared block gets a private
 * copy of that one block, and its table entry is switched to the copy).  In place; pairs are
 * applied in order.  Ids outside [0, num_blocks) are an error.
 */
int oracle_copy_blocks(uint16_t* k_pool, uint16_t* v_pool, const int32_t* src_ids,
                       const int32_t* dst_ids, int n, int block_size, int kv_heads,
                       int head_dim, int num_blocks) {
    if (n < 0 || block_size <= 0 || kv_heads <= 0 || head_dim <= 0) return ORACLE_BAD_ARG;
    for (int i = 0; i < n; ++i)
        if (src_ids[i] < 0 || src_ids[i] >= num_blocks || dst_ids[i] < 0 || dst_ids[i] >= num_blocks)
            return ORACLE_BAD_TABLE;
    const int64_t per_block = (int64_t)block_size * kv_heads * head_dim;
    for (int i = 0; i < n; ++i) {
        memmove(k_pool + dst_ids[i] * per_block, k_pool + src_ids[i] * per_block,
                sizeof(uint16_t) * (size_t)per_block);
        memmove(v_pool + dst_ids[i] * per_block, v_pool + src_ids[i] * per_block,
                sizeof(uint16_t) * (size_t)per_block);
    }
    return ORACLE_OK;
}

/*
 * Prefill scatter: a batched prefill pads its rows on the left to the longest
 * prompt of the batch; afterwards each row's K/V moves into the row's blocks
 * without the padding ("Paged attention", section "What changed").  Source
 * k_src, v_src: [rows][width][kv_heads][head_dim]; row r's tokens are columns
 * src_start[r] .. src_start[r] + lengths[r] - 1 and go to logical positions
 * dst_start[r] .. dst_start[r] + lengths[r] - 1 of the row's table.  Rows
 * with lengths[r] <= 0 are skipped.  A position whose logical block is past
 * the table or whose id is out of range is an error.
 */
int oracle_prefill_scatter(uint16_t* k_pool, uint16_t* v_pool, const int32_t* block_tables,
                           const int32_t* src_start, const int32_t* dst_start,
                           const int32_t* lengths, const uint16_t* k_src, const uint16_t* v_src,
                           int rows, int width, int kv_heads, int head_dim, int block_size,
                           int max_blocks_per_row, int num_blocks) {
    if (rows < 0 || width < 0 || kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return ORACLE_BAD_ARG;
    const int64_t tok = (int64_t)kv_heads * head_dim;
    for (int r = 0; r < rows; ++r) {
        if (lengths[r] <= 0) continue;
        if (src_start[r] < 0 || src_start[r] + lengths[r] > width || dst_start[r] < 0)
            return ORACLE_BAD_ARG;
        for (int t = 0; t < lengths[r]; ++t) {
            const int pos = dst_start[r] + t;
            if (pos / block_size >= max_blocks_per_row) return ORACLE_BAD_TABLE;
            const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + pos / block_size];
            if (pb < 0 || pb >= num_blocks) return ORACLE_BAD_TABLE;
        }
    }
    for (int r = 0; r < rows; ++r) {
        for (int t = 0; t < lengths[r]; ++t) {
            const int pos = dst_start[r] + t;
            const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + pos / block_size];
            const int64_t dst = ((int64_t)pb * block_size + pos % block_size) * tok;
            const int64_t src = ((int64_t)r * width + src_start[r] + t) * tok;
            memcpy(k_pool + dst, k_src + src, sizeof(uint16_t) * (size_t)tok);
            memcpy(v_pool + dst, v_src + src, sizeof(uint16_t) * (size_t)tok);
        }
    }
    return ORACLE_OK;
}

/*
 * FP8 KV pools.  "PagedAttention" (deepconcepts.dev), section "Checking it
 * on a real system", names FP8 KV as a way to change the bytes per token;
 * the pages fix no format.  The reading taken here: the OCP 8-bit floating
 * point E4M3 format, one float scale per KV head (given by the caller); a
 * stored code c stands for e4m3(c) * scale[head].
 *
 * E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent 0
 * is subnormal: mantissa * 2^-9.  Otherwise (8 + mantissa) * 2^(exponent-10).
 * The codes with all exponent and mantissa bits set (0x7F, 0xFF) are NaN;
 * there is no infinity, so the largest magnitude is 0x7E = 448.
 */
double oracle_fp8_e4m3_to_double(uint8_t c) {
    const int sign = (c >> 7) & 1;
    const int expo = (c >> 3) & 0xf;
    const int mant = c & 7;
    double v;
    if (expo == 15 && mant == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)mant, -9);
    else
        v = ldexp((double)(8 + mant), expo - 10);
    return sign ? -v : v;
}

/*
 * Nearest E4M3 code to y, ties to the even code (the code's lowest bit is
 * the mantissa's), magnitudes above 448 saturating to 448, NaN to 0x7F.
 * Written as a search over the 127 non-negative finite codes, which are
 * exact in double, so every comparison is exact.
 */
uint8_t oracle_fp8_e4m3_from_float(float y) {
    if (isnan(y)) return 0x7F;
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    const double a = fabs((double)y);
    int best = 0;
    double best_err = a;  /* code 0 is +0 */
    for (int c = 1; c <= 0x7E; ++c) {
        const double err = fabs(oracle_fp8_e4m3_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    if (a > 448.0) best = 0x7E;
    return (uint8_t)(sign | best);
}

/* Quantisation of one fp16 value with scale s: the quotient x / s is formed
 * in binary32 (IEEE division, rounded to nearest) and then encoded. */
static uint8_t quantize_fp8(uint16_t xh, float s) {
    const float x = (float)oracle_half_to_double(xh);
    const float y = x / s;
    return oracle_fp8_e4m3_from_float(y);
}

void oracle_fp8_quantize_array(uint8_t* dst, const uint16_t* src, int64_t n, float s) {
    for (int64_t i = 0; i < n; ++i) dst[i] = quantize_fp8(src[i], s);
}

/*
 * Append into FP8 pools: as oracle_paged_append, with every element of head
 * h of the new token stored as its quantisation with k_scale[h] (K) or
 * v_scale[h] (V).  Pools: [num_blocks][block_size][kv_heads][head_dim] bytes.
 */
int oracle_paged_append_fp8(uint8_t* k_pool, uint8_t* v_pool, const float* k_scale,
                            const float* v_scale, const int32_t* block_tables,
                            const int32_t* positions, const uint16_t* k_new,
                            const uint16_t* v_new, int rows, int kv_heads, int head_dim,
                            int block_size, int max_blocks_per_row, int num_blocks) {
    if (rows < 0 || kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        const int pos = positions[r];
        if (pos < 0) continue;
        if (pos / block_size >= max_blocks_per_row) return ORACLE_BAD_TABLE;
        const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + pos / block_size];
        if (pb < 0 || pb >= num_blocks) return ORACLE_BAD_TABLE;
    }
    for (int r = 0; r < rows; ++r) {
        const int pos = positions[r];
        if (pos < 0) continue;
        const int64_t pb = block_tables[(int64_t)r * max_blocks_per_row + pos / block_size];
        for (int h = 0; h < kv_heads; ++h) {
            const int64_t dst = idx4(pb, pos % block_size, h, 0, block_size, kv_heads, head_dim);
            const int64_t src = ((int64_t)r * kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                k_pool[dst + d] = quantize_fp8(k_new[src + d], k_scale[h]);
                v_pool[dst + d] = quantize_fp8(v_new[src + d], v_scale[h]);
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Paged decode over FP8 pools: the definition of oracle_paged_decode with
 * K_t[d] = e4m3(k code) * k_scale[kvh] and V_t[d] = e4m3(v code) *
 * v_scale[kvh], all in double.
 */
int oracle_paged_decode_fp8(double* out, const uint16_t* q, const uint8_t* k_pool,
                            const uint8_t* v_pool, const float* k_scale, const float* v_scale,
                            const int32_t* block_tables, const int32_t* seq_lens, int rows,
                            int q_heads, int kv_heads, int head_dim, int block_size,
                            double scale, int max_blocks_per_row, int num_blocks,
                            int num_threads) {
    if (!check_heads(q_heads, kv_heads, head_dim) || block_size <= 0 || rows < 0)
        return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        const int L = seq_lens[r];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks_per_row * block_size)
            return ORACLE_BAD_ARG;
        for (int lb = 0; lb < (L + block_size - 1) / block_size; ++lb) {
            const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + lb];
            if (pb < 0 || pb >= num_blocks) return ORACLE_BAD_TABLE;
        }
    }
    const int group = q_heads / kv_heads;
    int failed = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < q_heads; ++h) {
            const int L = seq_lens[r];
            const int kvh = h / group;
            double* o = out + ((int64_t)r * q_heads + h) * head_dim;
            const uint16_t* qv = q + ((int64_t)r * q_heads + h) * head_dim;
            double* s = (double*)malloc(sizeof(double) * (L + 1));
            if (!s) {
#pragma omp atomic write
                failed = 1;
                continue;
            }
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (L > 0) {
                double m = -INFINITY;
                for (int t = 0; t < L; ++t) {
                    const int64_t pb = block_tables[(int64_t)r * max_blocks_per_row + t / block_size];
                    const int64_t off = idx4(pb, t % block_size, kvh, 0, block_size, kv_heads, head_dim);
                    double acc = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        acc += oracle_half_to_double(qv[d]) *
                               (oracle_fp8_e4m3_to_double(k_pool[off + d]) * (double)k_scale[kvh]);
                    s[t] = scale * acc;
                    if (s[t] > m) m = s[t];
                }
                double z = 0.0;
                for (int t = 0; t < L; ++t) {
                    s[t] = exp(s[t] - m);
                    z += s[t];
                }
                for (int t = 0; t < L; ++t) {
                    const int64_t pb = block_tables[(int64_t)r * max_blocks_per_row + t / block_size];
                    const int64_t off = idx4(pb, t % block_size, kvh, 0, block_size, kv_heads, head_dim);
                    const double w = s[t] / z;
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += w * (oracle_fp8_e4m3_to_double(v_pool[off + d]) * (double)v_scale[kvh]);
                }
            }
            free(s);
        }
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Chunked prefill: several query tokens per row, causal within the chunk.
 * "Paged attention" (danielfleming.xyz), section "What changed" and the
 * closing paragraphs: the following engine breaks long prompts into pieces of
 * a fixed size (512 tokens) and runs decode steps in between; "Continuous
 * batching", closing section: chunking long prefills is named as the next
 * step.  Reading
 * taken (the pages give no kernel): row r's chunk holds the
 * C_r = q_start[r+1] - q_start[r] newest tokens of the row, at positions
 * p_r + i with p_r = seq_lens[r] - C_r (their K/V already in the row's
 * blocks); query i attends to the row's tokens 0 .. p_r + i (causal), with
 * the same head grouping as decode.
 *
 * q: [q_start[rows]][q_heads][head_dim] fp16 bits (rows' chunks packed in
 * order); out: the same shape, double.
 */
int oracle_paged_prefill(double* out, const uint16_t* q, const uint16_t* k_pool,
                         const uint16_t* v_pool, const int32_t* block_tables,
                         const int32_t* seq_lens, const int32_t* q_start, int rows, int q_heads,
                         int kv_heads, int head_dim, int block_size, double scale,
                         int max_blocks_per_row, int num_blocks, int num_threads) {
    if (!check_heads(q_heads, kv_heads, head_dim) || block_size <= 0 || rows < 0)
        return ORACLE_BAD_ARG;
    if (q_start[0] != 0) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        const int C = q_start[r + 1] - q_start[r];
        const int L = seq_lens[r];
        if (C < 0 || L < C || (int64_t)L > (int64_t)max_blocks_per_row * block_size)
            return ORACLE_BAD_ARG;
        for (int lb = 0; lb < (L + block_size - 1) / block_size; ++lb) {
            const int32_t pb = block_tables[(int64_t)r * max_blocks_per_row + lb];
            if (pb < 0 || pb >= num_blocks) return ORACLE_BAD_TABLE;
        }
    }
    const int group = q_heads / kv_heads;
    const int total = q_start[rows];
    int failed = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int qi = 0; qi < total; ++qi) {
        for (int h = 0; h < q_heads; ++h) {
            int r = 0;
            while (q_start[r + 1] <= qi) ++r;  /* row of packed query qi */
            const int C = q_start[r + 1] - q_start[r];
            const int pos = seq_lens[r] - C + (qi - q_start[r]);
            const int n = pos + 1;  /* tokens 0 .. pos */
            const int kvh = h / group;
            const uint16_t** kp = (const uint16_t**)malloc(sizeof(void*) * (n + 1));
            const uint16_t** vp = (const uint16_t**)malloc(sizeof(void*) * (n + 1));
            double* s = (double*)malloc(sizeof(double) * (n + 1));
            if (!kp || !vp || !s) {
#pragma omp atomic write
                failed = 1;
            } else {
                for (int t = 0; t < n; ++t) {
                    const int64_t pb = block_tables[(int64_t)r * max_blocks_per_row + t / block_size];
                    const int64_t off = idx4(pb, t % block_size, kvh, 0, block_size, kv_heads, head_dim);
                    kp[t] = k_pool + off;
                    vp[t] = v_pool + off;
                }
                attend_one(out + ((int64_t)qi * q_heads + h) * head_dim,
                           q + ((int64_t)qi * q_heads + h) * head_dim, kp, vp, n, head_dim, scale, s);
            }
            free(kp);
            free(vp);
            free(s);
        }
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}
