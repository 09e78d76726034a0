/*
 * Paged KV-cache oracle: a plain, slow, single-threaded CPU restatement of
 * the paged KV-cache write calls and of paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or constant with
 * the CUDA library, and the CUDA library never includes or calls it.
 *
 * Sources (the web pages this path is defined by):
 *   [kv_cache.rs]      spark_model/layers/ops/kv_cache.rs
 *   [kv_cache_fp8k.rs] metrale_model_layers/layers/ops/kv_cache_fp8k.rs
 * Each function names the page and the doc comment or launcher it follows.
 *
 * Precision: integer and byte work is exact; the FP8 encode takes the
 * quotient k / k_scale in IEEE binary32 (the page gives the division, and
 * k_scale is an f32 argument) and rounds it to E4M3 exactly; every other
 * floating-point step runs in binary64 and is rounded once at the store.
 *
 * Pins: every function here is checked by the CPU test suite against facts
 * that do not come from this file (brute force, closed forms, invariants,
 * torch's own conversions and attention). There is no "parity unpinned"
 * function in this file.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math
 *        (no FMA contraction, so x86-64 and aarch64 hosts agree bit for bit).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * Number formats, written from their definitions.
 * ---------------------------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32 word, so widening is exact. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static uint16_t bf16_bits_of_exact_float(float f) {
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(w >> 16);
}

/* Round a binary64 value once to BF16, round-to-nearest-even, directly (no
 * intermediate binary32 rounding). BF16 keeps 8 significant bits; its
 * normal exponents run from -126 to 127 and subnormals are spaced 2^-133.
 * Overflow rounds to infinity; NaN becomes the quiet NaN 0x7FC0 with the
 * input's sign. */
uint16_t oracle_f64_to_bf16(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    double ax = fabs(x);
    if (isinf(ax)) return (uint16_t)(sign | 0x7F80u);
    if (ax == 0.0) return sign;
    int e;
    (void)frexp(ax, &e);            /* ax = m * 2^e, m in [0.5, 1) */
    int unbiased = e - 1;           /* ax in [2^unbiased, 2^(unbiased+1)) */
    if (unbiased < -126) unbiased = -126;
    double quantum = ldexp(1.0, unbiased - 7);
    double n = rint(ax / quantum);  /* exact scaling, then RNE to an integer */
    double y = n * quantum;
    if (y >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | bf16_bits_of_exact_float((float)y));
}

/* FP8 E4M3 ("FN" variant: no infinities): sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits. Exponent field 0 holds subnormals m * 2^-9;
 * exponent field 15 with mantissa 7 is NaN; the largest finite value is
 * 0x7E = 448. */
double oracle_e4m3_to_f64(uint8_t code) {
    int s = (code >> 7) & 1;
    int ef = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (ef == 15 && m == 7) return s ? -NAN : NAN;
    if (ef == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, ef - 7);
    return s ? -v : v;
}

/* Encode a binary64 value to E4M3 with round-to-nearest-even and saturation
 * to the largest finite magnitude (448) for |x| >= 448 and for infinities.
 * NaN encodes as the canonical NaN 0x7F. */
uint8_t oracle_e4m3_encode_f64(double x) {
    uint8_t sign = signbit(x) ? 0x80u : 0u;
    if (isnan(x)) return 0x7Fu;
    double ax = fabs(x);
    if (ax >= 448.0) return (uint8_t)(sign | 0x7Eu);
    if (ax == 0.0) return sign;
    int e;
    (void)frexp(ax, &e);
    int unbiased = e - 1;
    if (unbiased < -6) unbiased = -6;        /* subnormal range shares 2^-9 spacing */
    double quantum = ldexp(1.0, unbiased - 3);
    double y = rint(ax / quantum) * quantum; /* at most 448 since ax < 448 */
    if (y < ldexp(1.0, -6))                  /* subnormal (or zero) */
        return (uint8_t)(sign | (uint8_t)(y / ldexp(1.0, -9)));
    int ye;
    (void)frexp(y, &ye);
    int yexp = ye - 1;
    int mant = (int)((y / ldexp(1.0, yexp) - 1.0) * 8.0);
    return (uint8_t)(sign | (uint8_t)(((yexp + 7) << 3) | mant));
}

/* The same rule for a binary32 input (exactly representable in binary64). */
uint8_t oracle_e4m3_encode(float xf) { return oracle_e4m3_encode_f64((double)xf); }

/* ------------------------------------------------------------------------
 * Slot mapping.  [kv_cache.rs] `fill_slots_from_block_table`: for i < count,
 * position p = start_pos + i lives in logical block p / block_size of the
 * sequence, whose physical block is block_table[p / block_size]; the flat
 * slot is physical_block * block_size + p % block_size. [kv_cache.rs]
 * `reshape_and_cache` doc: slot_mapping is i64[num_tokens].
 * ---------------------------------------------------------------------- */
void oracle_fill_slots(int64_t *slots, const int32_t *block_table, uint32_t start_pos,
                       uint32_t count, uint32_t block_size) {
    for (uint32_t i = 0; i < count; ++i) {
        uint64_t p = (uint64_t)start_pos + i;
        int64_t physical_block = block_table[p / block_size];
        slots[i] = physical_block * (int64_t)block_size + (int64_t)(p % block_size);
    }
}

/* Element index of (slot, head, dim) in a [num_blocks, block_size,
 * num_kv_heads, head_dim] pool: the slot's block is slot / block_size and its
 * row within the block is slot % block_size. */
static int64_t pool_index(int64_t slot, uint32_t block_size, uint32_t num_kv_heads,
                          uint32_t head_dim, uint32_t head, uint32_t d) {
    int64_t block = slot / (int64_t)block_size;
    int64_t offset = slot % (int64_t)block_size;
    return ((block * (int64_t)block_size + offset) * num_kv_heads + head) * (int64_t)head_dim + d;
}

/* ------------------------------------------------------------------------
 * [kv_cache.rs] `reshape_and_cache` (BF16: "no quantization, direct BF16
 * copy") and `reshape_and_cache_flash_v_only` (its V half). Token t's head h
 * row starts at key + t * key_stride + h * head_dim. A negative slot marks a
 * padding token and is skipped.
 * ---------------------------------------------------------------------- */
void oracle_write_v_only(const uint16_t *value, uint16_t *v_cache, const int64_t *slot_mapping,
                         uint32_t num_tokens, uint32_t num_kv_heads, uint32_t head_dim,
                         uint32_t block_size, uint32_t value_stride) {
    for (uint32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        for (uint32_t h = 0; h < num_kv_heads; ++h)
            for (uint32_t d = 0; d < head_dim; ++d)
                v_cache[pool_index(slot, block_size, num_kv_heads, head_dim, h, d)] =
                    value[(int64_t)t * value_stride + (int64_t)h * head_dim + d];
    }
}

void oracle_write_bf16(const uint16_t *key, const uint16_t *value, uint16_t *k_cache,
                       uint16_t *v_cache, const int64_t *slot_mapping, uint32_t num_tokens,
                       uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                       uint32_t key_stride, uint32_t value_stride) {
    oracle_write_v_only(key, k_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                        block_size, key_stride);
    oracle_write_v_only(value, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                        block_size, value_stride);
}

/* Quantised paged write of one tensor: element x of token t, head h is stored
 * as the E4M3 code of the binary32 quotient (float)x / scale, rounded to
 * nearest. */
static void write_rows_e4m3(const uint16_t *src, uint32_t src_stride, uint8_t *cache,
                            const int64_t *slot_mapping, uint32_t num_tokens,
                            uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                            float scale) {
    for (uint32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        for (uint32_t h = 0; h < num_kv_heads; ++h)
            for (uint32_t d = 0; d < head_dim; ++d) {
                float x = (float)oracle_bf16_to_f64(
                    src[(int64_t)t * src_stride + (int64_t)h * head_dim + d]);
                float quotient = x / scale; /* binary32 division, round to nearest */
                cache[pool_index(slot, block_size, num_kv_heads, head_dim, h, d)] =
                    oracle_e4m3_encode(quotient);
            }
    }
}

/* ------------------------------------------------------------------------
 * [kv_cache_fp8k.rs] module invariants: the write stores k / k_scale as
 * E4M3 in the [num_blocks, block_size, num_kv_heads, head_dim] layout; the
 * launcher argument order is that of `reshape_and_cache_fp8k_turbo3v`. V is
 * kept BF16 here (a direct copy, as in [kv_cache.rs] `reshape_and_cache`).
 * ---------------------------------------------------------------------- */
void oracle_write_fp8k(const uint16_t *key, const uint16_t *value, uint8_t *k_cache_fp8,
                       uint16_t *v_cache, const int64_t *slot_mapping, uint32_t num_tokens,
                       uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                       uint32_t key_stride, uint32_t value_stride, float k_scale) {
    write_rows_e4m3(key, key_stride, k_cache_fp8, slot_mapping, num_tokens, num_kv_heads,
                    head_dim, block_size, k_scale);
    oracle_write_v_only(value, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                        block_size, value_stride);
}

/* ------------------------------------------------------------------------
 * [kv_cache.rs] `reshape_and_cache_fp8`: K and V both stored as E4M3, K as
 * k / k_scale and V as v / v_scale, each with the rule above, into two
 * pools of the same layout. Argument order as the launcher's (k_scale,
 * v_scale before the strides); its cache_stride is implied by the layout.
 * ---------------------------------------------------------------------- */
void oracle_write_fp8(const uint16_t *key, const uint16_t *value, uint8_t *k_cache_fp8,
                      uint8_t *v_cache_fp8, const int64_t *slot_mapping, uint32_t num_tokens,
                      uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                      float k_scale, float v_scale, uint32_t key_stride, uint32_t value_stride) {
    write_rows_e4m3(key, key_stride, k_cache_fp8, slot_mapping, num_tokens, num_kv_heads,
                    head_dim, block_size, k_scale);
    write_rows_e4m3(value, value_stride, v_cache_fp8, slot_mapping, num_tokens, num_kv_heads,
                    head_dim, block_size, v_scale);
}

/* ------------------------------------------------------------------------
 * [kv_cache.rs] `fused_k_norm_rope_cache_write_bf16`: RMSNorm, then RoPE,
 * then the BF16 paged write, with K kept at high precision through all three
 * steps and rounded once at the write. The steps are exposed one by one so
 * that the tests can pin each of them.
 * ---------------------------------------------------------------------- */

/* RMSNorm of one head row: y_d = x_d / sqrt(mean(x^2) + eps) * w_d. */
void oracle_rmsnorm_row(const double *x, const double *w, uint32_t head_dim, double eps,
                        double *y) {
    double sum_sq = 0.0;
    for (uint32_t d = 0; d < head_dim; ++d) sum_sq += x[d] * x[d];
    double inv_rms = 1.0 / sqrt(sum_sq / head_dim + eps);
    for (uint32_t d = 0; d < head_dim; ++d) y[d] = x[d] * inv_rms * w[d];
}

/* Rotary embedding of one head row, rotate-half pairing: for
 * i < rotary_dim / 2 the pair (i, i + rotary_dim / 2) turns by the angle
 * p_i * theta^(-2i / rotary_dim); dims >= rotary_dim pass through.
 * [kv_cache.rs] `fused_k_norm_rope_cache_write_bf16_mrope`: the MRoPE
 * variant takes one position per rotation pair, chosen from the three
 * position streams by pair index mod 3, p_i = pos3[i % 3] (pos3[0] = t,
 * pos3[1] = h, pos3[2] = w). */
void oracle_rope_row_mrope(const double *y, uint32_t head_dim, uint32_t rotary_dim,
                           const double *pos3, double theta, double *out) {
    uint32_t half = rotary_dim / 2;
    for (uint32_t d = 0; d < head_dim; ++d) out[d] = y[d];
    for (uint32_t i = 0; i < half; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / (double)rotary_dim);
        double angle = pos3[i % 3] * inv_freq;
        double c = cos(angle), s = sin(angle);
        out[i] = y[i] * c - y[i + half] * s;
        out[i + half] = y[i + half] * c + y[i] * s;
    }
}

/* Plain RoPE at one integer position pos: every pair turns by
 * pos * theta^(-2i / rotary_dim), i.e. the rule above with three equal
 * positions. */
void oracle_rope_row(const double *y, uint32_t head_dim, uint32_t rotary_dim, double pos,
                     double theta, double *out) {
    const double pos3[3] = {pos, pos, pos};
    oracle_rope_row_mrope(y, head_dim, rotary_dim, pos3, theta, out);
}

/* The fused call's result before its single rounding, for one (token, head):
 * used by the pins and by the full write below. */
void oracle_fused_k_row_f64(const uint16_t *k_in, const uint16_t *k_norm_weight,
                            const int32_t *positions, uint32_t t, uint32_t h,
                            uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                            float rms_eps, float theta, double *out) {
    double x[1024], w[1024], y[1024];
    for (uint32_t d = 0; d < head_dim; ++d) {
        x[d] = oracle_bf16_to_f64(k_in[((int64_t)t * num_kv_heads + h) * head_dim + d]);
        w[d] = oracle_bf16_to_f64(k_norm_weight[d]);
    }
    oracle_rmsnorm_row(x, w, head_dim, (double)rms_eps, y);
    oracle_rope_row(y, head_dim, rotary_dim, (double)positions[t], (double)theta, out);
}

void oracle_write_fused_k_norm_rope_bf16(const uint16_t *k_in, const uint16_t *k_norm_weight,
                                         const int32_t *positions, uint16_t *k_cache,
                                         const int64_t *slot_mapping, uint32_t num_tokens,
                                         uint32_t num_kv_heads, uint32_t head_dim,
                                         uint32_t rotary_dim, uint32_t block_size,
                                         float rms_eps, float theta) {
    double out[1024];
    for (uint32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        for (uint32_t h = 0; h < num_kv_heads; ++h) {
            oracle_fused_k_row_f64(k_in, k_norm_weight, positions, t, h, num_kv_heads, head_dim,
                                   rotary_dim, rms_eps, theta, out);
            for (uint32_t d = 0; d < head_dim; ++d)
                k_cache[pool_index(slot, block_size, num_kv_heads, head_dim, h, d)] =
                    oracle_f64_to_bf16(out[d]);
        }
    }
}

/* The MRoPE variant's result before its rounding, for one (token, head). */
void oracle_fused_k_row_f64_mrope(const uint16_t *k_in, const uint16_t *k_norm_weight,
                                  const int32_t *pos_t, const int32_t *pos_h, const int32_t *pos_w,
                                  uint32_t t, uint32_t h, uint32_t num_kv_heads, uint32_t head_dim,
                                  uint32_t rotary_dim, float rms_eps, float theta, double *out) {
    double x[1024], w[1024], y[1024];
    double pos3[3] = {(double)pos_t[t], (double)pos_h[t], (double)pos_w[t]};
    for (uint32_t d = 0; d < head_dim; ++d) {
        x[d] = oracle_bf16_to_f64(k_in[((int64_t)t * num_kv_heads + h) * head_dim + d]);
        w[d] = oracle_bf16_to_f64(k_norm_weight[d]);
    }
    oracle_rmsnorm_row(x, w, head_dim, (double)rms_eps, y);
    oracle_rope_row_mrope(y, head_dim, rotary_dim, pos3, (double)theta, out);
}

void oracle_write_fused_k_norm_rope_bf16_mrope(const uint16_t *k_in, const uint16_t *k_norm_weight,
                                               const int32_t *pos_t, const int32_t *pos_h,
                                               const int32_t *pos_w, uint16_t *k_cache,
                                               const int64_t *slot_mapping, uint32_t num_tokens,
                                               uint32_t num_kv_heads, uint32_t head_dim,
                                               uint32_t rotary_dim, uint32_t block_size,
                                               float rms_eps, float theta) {
    double out[1024];
    for (uint32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        for (uint32_t h = 0; h < num_kv_heads; ++h) {
            oracle_fused_k_row_f64_mrope(k_in, k_norm_weight, pos_t, pos_h, pos_w, t, h, num_kv_heads,
                                         head_dim, rotary_dim, rms_eps, theta, out);
            for (uint32_t d = 0; d < head_dim; ++d)
                k_cache[pool_index(slot, block_size, num_kv_heads, head_dim, h, d)] =
                    oracle_f64_to_bf16(out[d]);
        }
    }
}

/* [kv_cache.rs] `fused_k_norm_rope_cache_write_fp8`: the FP8-output
 * sibling of the fused write. Same RMSNorm and RoPE; the result, without
 * any BF16 rounding, is multiplied by inv_scale and cast to E4M3 with
 * saturation (round to nearest even). */
void oracle_write_fused_k_norm_rope_fp8(const uint16_t *k_in, const uint16_t *k_norm_weight,
                                        const int32_t *positions, uint8_t *k_cache_fp8,
                                        const int64_t *slot_mapping, uint32_t num_tokens,
                                        uint32_t num_kv_heads, uint32_t head_dim,
                                        uint32_t rotary_dim, uint32_t block_size, float rms_eps,
                                        float theta, float inv_scale) {
    double out[1024];
    for (uint32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        for (uint32_t h = 0; h < num_kv_heads; ++h) {
            oracle_fused_k_row_f64(k_in, k_norm_weight, positions, t, h, num_kv_heads, head_dim,
                                   rotary_dim, rms_eps, theta, out);
            for (uint32_t d = 0; d < head_dim; ++d)
                k_cache_fp8[pool_index(slot, block_size, num_kv_heads, head_dim, h, d)] =
                    oracle_e4m3_encode_f64(out[d] * (double)inv_scale);
        }
    }
}

/* ------------------------------------------------------------------------
 * Paged decode attention. [kv_cache.rs] `paged_decode_attn_fp8` doc: one
 * query per (query head, sequence); block_tables is i32[num_seqs *
 * max_blocks_per_seq] and seq_lens is i32[num_seqs]. [kv_cache.rs]
 * `paged_decode_attn_bf16k_turbo3v` gives q_stride and sliding_window;
 * [kv_cache_fp8k.rs] module invariants: decode multiplies the stored FP8 K
 * by k_scale.
 *
 * For sequence s and query head h: the KV head is h / (num_q_heads /
 * num_kv_heads); L = seq_lens[s]; with sliding_window W > 0 the query
 * attends positions p in [max(0, L - W), L), else [0, L). Position p lives
 * in physical block block_tables[s * max_blocks_per_seq + p / block_size] at
 * row p % block_size. score_p = inv_sqrt_d * (q . k_p); the weights are the
 * softmax of the scores; the output is sum_p weight_p * v_p (zeros when no
 * position is attended).
 * ---------------------------------------------------------------------- */

/* Key element d of position p's row, dequantised to binary64: BF16 widened
 * exactly, or the E4M3 code's value times k_scale. */
static double key_at(const uint16_t *k_cache_bf16, const uint8_t *k_cache_fp8, int64_t idx,
                     float k_scale) {
    if (k_cache_fp8) return oracle_e4m3_to_f64(k_cache_fp8[idx]) * (double)k_scale;
    return oracle_bf16_to_f64(k_cache_bf16[idx]);
}

/* Value element d of position p's row: BF16 widened exactly, or, for the
 * FP8 K+V cache ([kv_cache.rs] `paged_decode_attn_fp8`, which takes
 * v_scale), the E4M3 code's value times v_scale. */
static double value_at(const uint16_t *v_cache_bf16, const uint8_t *v_cache_fp8, int64_t idx,
                       float v_scale) {
    if (v_cache_fp8) return oracle_e4m3_to_f64(v_cache_fp8[idx]) * (double)v_scale;
    return oracle_bf16_to_f64(v_cache_bf16[idx]);
}

/* The attention of one query row over positions [start, L) of one sequence,
 * start = max(0, L - sliding_window) when sliding_window > 0, else 0:
 * q_row is the query head's head_dim BF16 values and table the sequence's
 * block-table row. k_cache_fp8 != NULL selects the FP8-K cache (k_cache_bf16
 * is then unused); v_cache_fp8 != NULL likewise selects an FP8 V cache
 * (v_cache unused). out receives head_dim values. weights, when not NULL,
 * has room for L values and receives the softmax weight of each position (0
 * for positions outside the window). head_dim is at most 1024. */
static void attend(const uint16_t *q_row, const uint16_t *k_cache_bf16, const uint8_t *k_cache_fp8,
                   const uint16_t *v_cache, const uint8_t *v_cache_fp8, const int32_t *table,
                   int64_t L, uint32_t num_kv_heads, uint32_t kv_head, uint32_t head_dim,
                   uint32_t block_size, float inv_sqrt_d, float k_scale, float v_scale,
                   uint32_t sliding_window, double *out, double *weights) {
    int64_t start = 0;
    if (sliding_window > 0 && L > (int64_t)sliding_window) start = L - sliding_window;
    for (uint32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
    for (int64_t p = 0; weights && p < L; ++p) weights[p] = 0.0;
    if (L <= start) return;

    double qv[1024], acc[1024];
    for (uint32_t d = 0; d < head_dim; ++d) {
        qv[d] = oracle_bf16_to_f64(q_row[d]);
        acc[d] = 0.0;
    }
    double *scores = (double *)malloc((size_t)(L - start) * sizeof(double));
    int64_t *slots = (int64_t *)malloc((size_t)(L - start) * sizeof(int64_t));

    /* pass 1: walk the block table and score every attended position */
    double max_score = -INFINITY;
    for (int64_t p = start; p < L; ++p) {
        int64_t block = table[p / block_size];
        int64_t slot = block * (int64_t)block_size + p % block_size;
        double dot = 0.0;
        for (uint32_t d = 0; d < head_dim; ++d)
            dot += qv[d] * key_at(k_cache_bf16, k_cache_fp8,
                                  pool_index(slot, block_size, num_kv_heads, head_dim, kv_head, d),
                                  k_scale);
        slots[p - start] = slot;
        scores[p - start] = (double)inv_sqrt_d * dot;
        if (scores[p - start] > max_score) max_score = scores[p - start];
    }
    /* pass 2: softmax weights (max-shifted exponentials over their sum) and
     * the weighted sum of the V rows */
    double denom = 0.0;
    for (int64_t p = start; p < L; ++p) {
        double e = exp(scores[p - start] - max_score);
        scores[p - start] = e;
        denom += e;
        for (uint32_t d = 0; d < head_dim; ++d)
            acc[d] += e * value_at(v_cache, v_cache_fp8,
                                   pool_index(slots[p - start], block_size, num_kv_heads,
                                              head_dim, kv_head, d),
                                   v_scale);
    }
    for (uint32_t d = 0; d < head_dim; ++d) out[d] = acc[d] / denom;
    for (int64_t p = start; weights && p < L; ++p) weights[p] = scores[p - start] / denom;
    free(scores);
    free(slots);
}

/* Decode: the one query of sequence s (at position seq_lens[s] - 1) for
 * query head h, whose KV head is h / (num_q_heads / num_kv_heads). */
void oracle_decode_one(const uint16_t *q, const uint16_t *k_cache_bf16, const uint8_t *k_cache_fp8,
                       const uint16_t *v_cache, const uint8_t *v_cache_fp8,
                       const int32_t *block_tables, const int32_t *seq_lens,
                       uint32_t max_blocks_per_seq, uint32_t num_q_heads, uint32_t num_kv_heads,
                       uint32_t head_dim, uint32_t block_size, float inv_sqrt_d, float k_scale,
                       float v_scale, uint32_t q_stride, uint32_t sliding_window, uint32_t s,
                       uint32_t h, double *out, double *weights) {
    uint32_t group = num_q_heads / num_kv_heads;
    uint32_t kv_head = h / group;
    attend(q + (int64_t)s * q_stride + (int64_t)h * head_dim, k_cache_bf16, k_cache_fp8, v_cache,
           v_cache_fp8, block_tables + (int64_t)s * max_blocks_per_seq, seq_lens[s], num_kv_heads,
           kv_head, head_dim, block_size, inv_sqrt_d, k_scale, v_scale, sliding_window, out,
           weights);
}

static void decode_all(const uint16_t *q, const uint16_t *k_cache_bf16, const uint8_t *k_cache_fp8,
                       const uint16_t *v_cache, const uint8_t *v_cache_fp8, float *output,
                       const int32_t *block_tables, const int32_t *seq_lens,
                       uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                       uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                       float inv_sqrt_d, float k_scale, float v_scale, uint32_t q_stride,
                       uint32_t sliding_window) {
    double out[1024];
    for (uint32_t s = 0; s < num_seqs; ++s)
        for (uint32_t h = 0; h < num_q_heads; ++h) {
            oracle_decode_one(q, k_cache_bf16, k_cache_fp8, v_cache, v_cache_fp8, block_tables,
                              seq_lens, max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim,
                              block_size, inv_sqrt_d, k_scale, v_scale, q_stride, sliding_window,
                              s, h, out, 0);
            for (uint32_t d = 0; d < head_dim; ++d)
                output[((int64_t)s * num_q_heads + h) * head_dim + d] = (float)out[d];
        }
}

void oracle_paged_decode_attn_bf16(const uint16_t *q, const uint16_t *k_cache,
                                   const uint16_t *v_cache, float *output,
                                   const int32_t *block_tables, const int32_t *seq_lens,
                                   uint32_t max_blocks_per_seq, uint32_t num_seqs,
                                   uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                   uint32_t block_size, float inv_sqrt_d, uint32_t q_stride,
                                   uint32_t sliding_window) {
    decode_all(q, k_cache, 0, v_cache, 0, output, block_tables, seq_lens, max_blocks_per_seq,
               num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, 1.0f, 1.0f,
               q_stride, sliding_window);
}

void oracle_paged_decode_attn_fp8k(const uint16_t *q, const uint8_t *k_cache_fp8,
                                   const uint16_t *v_cache, float *output,
                                   const int32_t *block_tables, const int32_t *seq_lens,
                                   uint32_t max_blocks_per_seq, uint32_t num_seqs,
                                   uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                   uint32_t block_size, float inv_sqrt_d, float k_scale,
                                   uint32_t q_stride, uint32_t sliding_window) {
    decode_all(q, 0, k_cache_fp8, v_cache, 0, output, block_tables, seq_lens, max_blocks_per_seq,
               num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, k_scale, 1.0f,
               q_stride, sliding_window);
}

/* [kv_cache.rs] `paged_decode_attn_fp8`: K and V both E4M3, dequantised by
 * k_scale and v_scale. */
void oracle_paged_decode_attn_fp8(const uint16_t *q, const uint8_t *k_cache_fp8,
                                  const uint8_t *v_cache_fp8, float *output,
                                  const int32_t *block_tables, const int32_t *seq_lens,
                                  uint32_t max_blocks_per_seq, uint32_t num_seqs,
                                  uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                  uint32_t block_size, float inv_sqrt_d, float k_scale,
                                  float v_scale, uint32_t q_stride, uint32_t sliding_window) {
    decode_all(q, 0, k_cache_fp8, 0, v_cache_fp8, output, block_tables, seq_lens,
               max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
               inv_sqrt_d, k_scale, v_scale, q_stride, sliding_window);
}

/* ------------------------------------------------------------------------
 * Multi-token (chunked-prefill) paged attention. [kv_cache.rs] "Batched
 * prefill variants (N tokens)" (a heading only): sequence s brings
 * n_s = query_start_loc[s + 1] - query_start_loc[s] query tokens, the last n_s
 * of its seq_lens[s] cached positions. Query j (row query_start_loc[s] + j of
 * q, at position P = seq_lens[s] - n_s + j) attends causally: positions
 * [start, P] with start = max(0, P + 1 - sliding_window) when
 * sliding_window > 0, else 0 -- exactly what a decode of that sequence
 * truncated to length P + 1 attends. A query with P < 0 (n_s > seq_lens[s])
 * attends nothing and gives zeros. Output float32
 * [num_q_tokens, num_q_heads, head_dim]. k_cache_fp8 != NULL selects the
 * FP8-K cache (k_scale as in the FP8-K decode).
 * ---------------------------------------------------------------------- */
void oracle_paged_prefill_attn(const uint16_t *q, const uint16_t *k_cache_bf16,
                               const uint8_t *k_cache_fp8, const uint16_t *v_cache,
                               const uint8_t *v_cache_fp8, float *output,
                               const int32_t *block_tables, const int32_t *seq_lens,
                               const int32_t *query_start_loc, uint32_t max_blocks_per_seq,
                               uint32_t num_seqs, uint32_t num_q_heads, uint32_t num_kv_heads,
                               uint32_t head_dim, uint32_t block_size, float inv_sqrt_d,
                               float k_scale, float v_scale, uint32_t q_stride,
                               uint32_t sliding_window) {
    double out[1024];
    uint32_t group = num_q_heads / num_kv_heads;
    for (uint32_t s = 0; s < num_seqs; ++s) {
        int64_t n = (int64_t)query_start_loc[s + 1] - query_start_loc[s];
        for (int64_t j = 0; j < n; ++j) {
            int64_t row = query_start_loc[s] + j;
            int64_t position = (int64_t)seq_lens[s] - n + j;
            for (uint32_t h = 0; h < num_q_heads; ++h) {
                attend(q + row * q_stride + (int64_t)h * head_dim, k_cache_bf16, k_cache_fp8,
                       v_cache, v_cache_fp8, block_tables + (int64_t)s * max_blocks_per_seq, position + 1,
                       num_kv_heads, h / group, head_dim, block_size, inv_sqrt_d, k_scale, v_scale,
                       sliding_window, out, 0);
                for (uint32_t d = 0; d < head_dim; ++d)
                    output[(row * num_q_heads + h) * head_dim + d] = (float)out[d];
            }
        }
    }
}

/* ------------------------------------------------------------------------
 * Array forms of the format conversions, for the exhaustive tests.
 * ---------------------------------------------------------------------- */
void oracle_bf16_to_f64_array(const uint16_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(in[i]);
}
void oracle_f64_to_bf16_array(const double *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(in[i]);
}
void oracle_e4m3_to_f64_array(const uint8_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f64(in[i]);
}
void oracle_e4m3_encode_array(const float *in, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(in[i]);
}
void oracle_e4m3_encode_f64_array(const double *in, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode_f64(in[i]);
}
