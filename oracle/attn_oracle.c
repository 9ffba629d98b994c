/*
 * attn_oracle.c -- slow, plain fp64 CPU statement of grouped-query attention
 * over a decoder KV cache.  TEST INFRASTRUCTURE ONLY: it is called by the
 * tests, by the package's smoke check and by the benchmark's CPU-baseline leg,
 * never by the product path.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What is computed, and where the pages fix it:
 *
 *  - Attention itself is the plain definition: scores s_t = scale * <q, k_t>,
 *    weights e_t = exp(s_t - max s), out = sum e_t v_t / sum e_t, all in fp64
 *    from exact bf16 -> fp64 widening.  Split-KV and online softmax are exact
 *    reformulations of it (vibevoice.c, "The kernels that matter" and
 *    "Attention backends": every backend is checked against one FP64
 *    reference).
 *  - GQA: query head h reads KV head h / (n_q_heads / n_kv_heads), the
 *    grouping behind `enable_gqa` (Voxtral Realtime -- Architecture & Design
 *    Notes, "SDPA"; vibevoice.c, "Attention backends": the heads of one group
 *    share a KV head).
 *  - Cache kinds (Voxtral Realtime notes, "KV cache"; vibevoice.c, "Paged KV
 *    cache"):
 *      linear: key position t of request b lives in slot b*slots_per_seq + t;
 *      paged : slot block_table[b][t / block_size] * block_size + t % block_size;
 *      ring  : slot j of request b's ring holds absolute position
 *              abs_pos = j + floor((total_written - 1 - j) / ring) * ring,
 *              negative meaning never written (Voxtral notes, "Encoder KV
 *              cache", the analytic position formula).  The oracle walks
 *              ring SLOTS and recovers their positions with that formula; it
 *              never computes t % ring.
 *  - Mask: a key at position t is attended by a query at position pos iff
 *    t >= 0, delta = pos - t >= 0 and (window <= 0 or delta < window)
 *    (Voxtral notes, "Encoder KV cache", the `valid = ...` mask).
 *    For linear and paged caches the candidate keys are t = 0..seq_len-1
 *    ("seq_lens[r] -- its length", talker_multiframe, NarrowStep fields:
 *    keys written including this step's rows).
 *  - Append: rows are applied in order, cache[slot_mapping[i]] = new[i],
 *    as raw 16-bit copies; with a repeated slot the last row wins.
 *  - RoPE (for the fused append): interleaved pairs rotated by a float32
 *    angle pos * inv_freq[i], see oracle_rope_bf16.
 *  - FP8 cache (vibevoice.c, "KV cache"): K and V held as 8-bit floats with
 *    no scale factor, K stored relative to a per-layer reference vector
 *    built from the first prefill chunk; see the FP8 section below.
 *  - Prefill: query i of a sequence attends keys 0..i (and i - t < window
 *    when window > 0) of the same sequence (Voxtral notes, "Offline
 *    Encoder": causal SDPA).
 *
 * All bf16 tensors are passed as uint16_t bit patterns, row-major with the
 * last dimension contiguous.  Outputs are fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EMPTY_KEYSET 1
#define ORACLE_BAD_ARGS 2

#define ORACLE_LINEAR 0
#define ORACLE_PAGED 1
#define ORACLE_RING 2

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Floor division for a possibly negative numerator and a positive divisor. */
static int64_t floor_div(int64_t a, int64_t b) {
    int64_t q = a / b;
    if ((a % b != 0) && (a < 0)) q -= 1;
    return q;
}

/* Absolute position held by ring slot j after total_written rows were stored
 * (Voxtral notes, "Encoder KV cache").  Negative: the slot was never written. */
int64_t oracle_ring_abs_pos(int64_t j, int64_t total_written, int64_t ring) {
    return j + floor_div(total_written - 1 - j, ring) * ring;
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* KV append: cache[slot_mapping[i], :] = new[i, :] for i = 0..n-1 in order.
 * row_elems = n_kv_heads * head_dim.  Rows whose slot is outside
 * [0, num_slots) are skipped and counted; the count is returned. */
int64_t oracle_kv_append(uint16_t *k_cache, uint16_t *v_cache, int64_t num_slots,
                         int64_t row_elems, const uint16_t *k_new, const uint16_t *v_new,
                         const int64_t *slot_mapping, int64_t n) {
    int64_t skipped = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0 || s >= num_slots) {
            ++skipped;
            continue;
        }
        for (int64_t e = 0; e < row_elems; ++e) {
            k_cache[s * row_elems + e] = k_new[i * row_elems + e];
            v_cache[s * row_elems + e] = v_new[i * row_elems + e];
        }
    }
    return skipped;
}

/* Round a binary32 value to bf16, nearest even (NaN kept quiet). */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    if ((w & 0x7F800000u) == 0x7F800000u && (w & 0x007FFFFFu) != 0)
        return (uint16_t)((w >> 16) | 0x0040u);
    const uint32_t lsb = (w >> 16) & 1u;
    return (uint16_t)((w + 0x7FFFu + lsb) >> 16);
}

/* Rotary position embedding of interleaved pairs, as the pages state it
 * (Voxtral Realtime notes, "RoPE": frequencies computed on the fly from the
 * stored inv_freq; "Shared Patterns": the pairs are (x[2i], x[2i+1]) of each
 * head, rotated after a float32 upcast and cast back):
 *     theta_i = pos * inv_freq[i]                 (a float32 product)
 *     (x0, x1) -> (x0 cos theta_i - x1 sin theta_i, x0 sin theta_i + x1 cos theta_i)
 * The angle is the float32 product the pages form; its cosine and sine and
 * the rotation are taken in double and rounded once (through binary32) to
 * bf16.  x, out: bf16 bits [n, n_heads, head_dim]; pos[n]; inv_freq[head_dim / 2]. */
void oracle_rope_bf16(const uint16_t *x, int64_t n, int n_heads, int head_dim,
                      const int32_t *pos, const float *inv_freq, uint16_t *out) {
    for (int64_t r = 0; r < n; ++r)
        for (int h = 0; h < n_heads; ++h)
            for (int i = 0; i < head_dim / 2; ++i) {
                const int64_t e = (r * n_heads + h) * head_dim + 2 * i;
                const float theta = (float)pos[r] * inv_freq[i];
                const double c = cos((double)theta), sn = sin((double)theta);
                const double x0 = oracle_bf16_to_f64(x[e]), x1 = oracle_bf16_to_f64(x[e + 1]);
                out[e] = f32_to_bf16_rne((float)(x0 * c - x1 * sn));
                out[e + 1] = f32_to_bf16_rne((float)(x0 * sn + x1 * c));
            }
}

/* ---- FP8 KV cache (vibevoice.c, "KV cache") ----------------------------
 * The page fixes: the cache holds 8-bit floats converted by bit manipulation
 * alone (no scale factor), and K is stored relative to a per-layer reference
 * vector built from the first prefill chunk, which changes no attention
 * output because softmax ignores a shift shared by every key's score.
 * Readings taken where it is silent:
 *   - the format is E4M3 of the OCP 8-bit floating point specification:
 *     sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
 *     holds subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no
 *     infinities; the largest finite magnitude is 1.75 * 2^8 = 448;
 *   - encoding rounds to nearest with ties to an even mantissa and saturates
 *     every larger magnitude (infinity included) to 448; NaN encodes as 0x7F;
 *   - the reference is one float32 vector per KV head (the layer's key
 *     projection output split by head): the mean of the chunk's keys;
 *   - the difference k - ref is formed in binary32 and that value is
 *     encoded. */

/* Value of an E4M3 code, from the format's definition. */
double oracle_fp8_e4m3_to_f64(uint8_t code) {
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest integer to x >= 0, ties to even (x is exact in double). */
static double round_half_even(double x) {
    const double f = floor(x), r = x - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* E4M3 code of a binary32 value: round to nearest even, saturate to 448. */
uint8_t oracle_f32_to_fp8_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; a count of 8 is the smallest
         * normal, whose code is 8 as well */
        return sign | (uint8_t)round_half_even(ldexp(a, 9));
    }
    int E;
    frexp(a, &E); /* a in [2^(E-1), 2^E) */
    int e = E - 1;
    double m = round_half_even((ldexp(a, -e) - 1.0) * 8.0); /* 0 .. 8 */
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    const int field = e + 7;
    if (field > 15 || (field == 15 && m == 7.0)) return sign | 0x7E;
    return sign | (uint8_t)((field << 3) | (int)m);
}

/* E4M3 code -> bf16 bits.  Every E4M3 value is a bf16 value, so this is exact. */
uint16_t oracle_fp8_e4m3_to_bf16(uint8_t code) {
    return f32_to_bf16_rne((float)oracle_fp8_e4m3_to_f64(code));
}

/* FP8 append: for rows i = 0..n-1 in order, with s = slot_mapping[i] in
 * [0, num_slots) (other rows are skipped and counted):
 *     k_cache[s][e] = E4M3(float32(k_new[i][e]) - k_ref[e])   (k_ref NULL: no shift)
 *     v_cache[s][e] = E4M3(float32(v_new[i][e]))
 * e runs over the row's n_kv_heads * head_dim elements; k_ref is float32
 * [n_kv_heads][head_dim].  Caches are byte arrays [num_slots][row_elems]. */
int64_t oracle_kv_append_fp8(uint8_t *k_cache, uint8_t *v_cache, int64_t num_slots,
                             int64_t row_elems, const uint16_t *k_new, const uint16_t *v_new,
                             const float *k_ref, const int64_t *slot_mapping, int64_t n) {
    int64_t skipped = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0 || s >= num_slots) {
            ++skipped;
            continue;
        }
        for (int64_t e = 0; e < row_elems; ++e) {
            const float kf = (float)oracle_bf16_to_f64(k_new[i * row_elems + e]);
            volatile float d = k_ref ? kf - k_ref[e] : kf; /* a binary32 difference */
            k_cache[s * row_elems + e] = oracle_f32_to_fp8_e4m3(d);
            v_cache[s * row_elems + e] =
                oracle_f32_to_fp8_e4m3((float)oracle_bf16_to_f64(v_new[i * row_elems + e]));
        }
    }
    return skipped;
}

/* Reference vector: ref[e] = (1/n) * sum_i k[i][e] over the n rows of a
 * chunk, in fp64.  k: bf16 bits [n][row_elems]. */
void oracle_kv_reference(const uint16_t *k, int64_t n, int64_t row_elems, double *ref) {
    for (int64_t e = 0; e < row_elems; ++e) {
        double acc = 0.0;
        for (int64_t i = 0; i < n; ++i) acc += oracle_bf16_to_f64(k[i * row_elems + e]);
        ref[e] = n > 0 ? acc / (double)n : 0.0;
    }
}

/* The cache as the oracle sees it. */
typedef struct {
    int kind;
    const uint16_t *k, *v; /* [num_slots, n_kv_heads, head_dim] */
    int64_t num_slots;
    int64_t slots_per_seq; /* linear: per-request capacity; ring: ring size */
    const int32_t *block_table;
    int block_size, max_blocks_per_seq;
} oracle_cache;

/* Enumerate the candidate keys of request b as (slot, absolute position)
 * pairs.  Returns the count; slots[] and tpos[] must hold max_cand entries. */
static int64_t candidate_keys(const oracle_cache *c, int b, int64_t seq_len, int64_t *slots,
                              int64_t *tpos, int64_t max_cand, int *bad) {
    int64_t n = 0;
    if (c->kind == ORACLE_RING) {
        int64_t ring = c->slots_per_seq;
        for (int64_t j = 0; j < ring && n < max_cand; ++j) {
            slots[n] = (int64_t)b * ring + j;
            tpos[n] = oracle_ring_abs_pos(j, seq_len, ring);
            ++n;
        }
    } else {
        for (int64_t t = 0; t < seq_len && n < max_cand; ++t) {
            int64_t slot;
            if (c->kind == ORACLE_LINEAR) {
                slot = (int64_t)b * c->slots_per_seq + t;
            } else {
                int64_t blk = t / c->block_size;
                if (blk >= c->max_blocks_per_seq) {
                    *bad = 1;
                    break;
                }
                int64_t page = c->block_table[(int64_t)b * c->max_blocks_per_seq + blk];
                slot = page * c->block_size + t % c->block_size;
            }
            slots[n] = slot;
            tpos[n] = t;
            ++n;
        }
    }
    for (int64_t i = 0; i < n; ++i)
        if (slots[i] < 0 || slots[i] >= c->num_slots) *bad = 1;
    return n;
}

static int key_is_valid(int64_t t, int64_t pos, int window) {
    int64_t delta = pos - t;
    if (t < 0) return 0;
    if (delta < 0) return 0;
    if (window > 0 && delta >= window) return 0;
    return 1;
}

/* Softmax-weighted sum of one query row over a list of keys, all fp64.
 * kv_elem(i) addresses key i's head row.  weights_out (optional) receives the
 * normalised weights of the listed keys.  Returns 0, or 1 on an empty list. */
static int attend_one(const uint16_t *q_row, int head_dim, double scale, const uint16_t *kbase,
                      const uint16_t *vbase, const int64_t *row_off, int64_t nkeys, double *s,
                      double *out_row, double *weights_out) {
    if (nkeys == 0) {
        for (int d = 0; d < head_dim; ++d) out_row[d] = NAN;
        return 1;
    }
    double m = -INFINITY;
    for (int64_t i = 0; i < nkeys; ++i) {
        const uint16_t *kr = kbase + row_off[i];
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
            acc += oracle_bf16_to_f64(q_row[d]) * oracle_bf16_to_f64(kr[d]);
        s[i] = scale * acc;
        if (s[i] > m) m = s[i];
    }
    double denom = 0.0;
    for (int64_t i = 0; i < nkeys; ++i) {
        s[i] = exp(s[i] - m);
        denom += s[i];
    }
    for (int d = 0; d < head_dim; ++d) out_row[d] = 0.0;
    for (int64_t i = 0; i < nkeys; ++i) {
        const uint16_t *vr = vbase + row_off[i];
        double w = s[i] / denom;
        if (weights_out) weights_out[i] = w;
        for (int d = 0; d < head_dim; ++d) out_row[d] += w * oracle_bf16_to_f64(vr[d]);
    }
    return 0;
}

/* Decode attention: for every request b, query row r and query head h,
 * attend the valid keys of b's cache.
 *   q         [batch, q_rows, n_q_heads, head_dim] bf16
 *   seq_lens  [batch]            keys written, including this step's rows
 *   positions [batch * q_rows]   absolute position of each query row
 *   out       [batch, q_rows, n_q_heads, head_dim] fp64
 * Returns ORACLE_OK, ORACLE_EMPTY_KEYSET (some row had no valid key: that
 * row's output is NaN) or ORACLE_BAD_ARGS. */
int oracle_decode(const uint16_t *q, int batch, int q_rows, int n_q_heads, int n_kv_heads,
                  int head_dim, int kind, const uint16_t *k_cache, const uint16_t *v_cache,
                  int64_t num_slots, int64_t slots_per_seq, const int32_t *block_table,
                  int block_size, int max_blocks_per_seq, const int32_t *seq_lens,
                  const int32_t *positions, int window, double scale, double *out) {
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return ORACLE_BAD_ARGS;
    if (kind != ORACLE_LINEAR && kind != ORACLE_PAGED && kind != ORACLE_RING)
        return ORACLE_BAD_ARGS;
    if (kind == ORACLE_PAGED && block_size <= 0) return ORACLE_BAD_ARGS;
    oracle_cache c = {kind, k_cache, v_cache, num_slots, slots_per_seq,
                      block_table, block_size, max_blocks_per_seq};
    const int group = n_q_heads / n_kv_heads;
    const int64_t row_elems = (int64_t)n_kv_heads * head_dim;
    int status = ORACLE_OK;
    const int64_t items = (int64_t)batch * q_rows * n_q_heads;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < items; ++it) {
        int h = (int)(it % n_q_heads);
        int r = (int)((it / n_q_heads) % q_rows);
        int b = (int)(it / ((int64_t)n_q_heads * q_rows));
        int g = h / group;
        int64_t seq_len = seq_lens[b];
        int64_t pos = positions[(int64_t)b * q_rows + r];
        int64_t max_cand = kind == ORACLE_RING ? slots_per_seq : seq_len;
        if (max_cand < 1) max_cand = 1;
        int64_t *slots = (int64_t *)malloc(sizeof(int64_t) * max_cand);
        int64_t *tpos = (int64_t *)malloc(sizeof(int64_t) * max_cand);
        int64_t *off = (int64_t *)malloc(sizeof(int64_t) * max_cand);
        double *s = (double *)malloc(sizeof(double) * max_cand);
        int bad = 0;
        int64_t ncand = candidate_keys(&c, b, seq_len, slots, tpos, max_cand, &bad);
        int64_t nkeys = 0;
        double *o = out + it * head_dim;
        if (!bad) {
            for (int64_t i = 0; i < ncand; ++i)
                if (key_is_valid(tpos[i], pos, window))
                    off[nkeys++] = slots[i] * row_elems + (int64_t)g * head_dim;
        }
        int rc = bad ? ORACLE_BAD_ARGS
                     : attend_one(q + it * head_dim, head_dim, scale, k_cache, v_cache, off, nkeys,
                                  s, o, NULL);
        if (bad)
            for (int d = 0; d < head_dim; ++d) o[d] = NAN;
        if (rc != 0) {
#pragma omp critical
            {
                if (status == ORACLE_OK) status = bad ? ORACLE_BAD_ARGS : ORACLE_EMPTY_KEYSET;
            }
        }
        free(slots);
        free(tpos);
        free(off);
        free(s);
    }
    return status;
}

/* The attention weights of one decode row (request b, row r, head h): for
 * each candidate key, its absolute position and its weight (0 for masked
 * keys).  Returns the number of candidates written (<= cap), or -1. */
int64_t oracle_decode_weights(const uint16_t *q, int batch, int q_rows, int n_q_heads,
                              int n_kv_heads, int head_dim, int kind, const uint16_t *k_cache,
                              const uint16_t *v_cache, int64_t num_slots, int64_t slots_per_seq,
                              const int32_t *block_table, int block_size, int max_blocks_per_seq,
                              const int32_t *seq_lens, const int32_t *positions, int window,
                              double scale, int b, int r, int h, int64_t *tpos_out,
                              double *w_out, int64_t cap) {
    if (b < 0 || b >= batch || r < 0 || r >= q_rows || h < 0 || h >= n_q_heads) return -1;
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
    oracle_cache c = {kind, k_cache, v_cache, num_slots, slots_per_seq,
                      block_table, block_size, max_blocks_per_seq};
    int g = h / (n_q_heads / n_kv_heads);
    int64_t row_elems = (int64_t)n_kv_heads * head_dim;
    int64_t seq_len = seq_lens[b];
    int64_t pos = positions[(int64_t)b * q_rows + r];
    int64_t max_cand = kind == ORACLE_RING ? slots_per_seq : seq_len;
    if (max_cand > cap) return -1;
    if (max_cand < 1) max_cand = 1;
    int64_t *slots = (int64_t *)malloc(sizeof(int64_t) * max_cand);
    int64_t *tp = (int64_t *)malloc(sizeof(int64_t) * max_cand);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * max_cand);
    int64_t *which = (int64_t *)malloc(sizeof(int64_t) * max_cand);
    double *s = (double *)malloc(sizeof(double) * max_cand);
    double *w = (double *)malloc(sizeof(double) * max_cand);
    double *o = (double *)malloc(sizeof(double) * head_dim);
    int bad = 0;
    int64_t ncand = candidate_keys(&c, b, seq_len, slots, tp, max_cand, &bad);
    int64_t nkeys = 0;
    for (int64_t i = 0; i < ncand; ++i) {
        tpos_out[i] = tp[i];
        w_out[i] = 0.0;
        if (key_is_valid(tp[i], pos, window)) {
            which[nkeys] = i;
            off[nkeys++] = slots[i] * row_elems + (int64_t)g * head_dim;
        }
    }
    int64_t it = ((int64_t)b * q_rows + r) * n_q_heads + h;
    int64_t result = ncand;
    if (bad || attend_one(q + it * head_dim, head_dim, scale, k_cache, v_cache, off, nkeys, s, o,
                          w) != 0)
        result = -1;
    else
        for (int64_t i = 0; i < nkeys; ++i) w_out[which[i]] = w[i];
    free(slots);
    free(tp);
    free(off);
    free(which);
    free(s);
    free(w);
    free(o);
    return result;
}

/* Causal (optionally windowed) prefill attention.
 *   q   [batch, seq_len, n_q_heads, head_dim] bf16
 *   k,v [batch, seq_len, n_kv_heads, head_dim] bf16
 *   out [batch, n_rows or seq_len, n_q_heads, head_dim] fp64
 * rows (optional, n_rows entries) restricts the computation to those query
 * positions of every sequence; out then holds them in that order. */
int oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int batch,
                   int seq_len, int window, int n_q_heads, int n_kv_heads, int head_dim,
                   double scale, const int32_t *rows, int n_rows, double *out) {
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return ORACLE_BAD_ARGS;
    const int group = n_q_heads / n_kv_heads;
    const int nr = rows ? n_rows : seq_len;
    for (int i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= seq_len) return ORACLE_BAD_ARGS;
    const int64_t items = (int64_t)batch * nr * n_q_heads;
    const int64_t kv_row = (int64_t)n_kv_heads * head_dim;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < items; ++it) {
        int h = (int)(it % n_q_heads);
        int ri = (int)((it / n_q_heads) % nr);
        int b = (int)(it / ((int64_t)n_q_heads * nr));
        int i = rows ? rows[ri] : ri;
        int g = h / group;
        int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (i + 1));
        double *s = (double *)malloc(sizeof(double) * (i + 1));
        int64_t nkeys = 0;
        for (int64_t t = 0; t <= i; ++t)
            if (key_is_valid(t, i, window))
                off[nkeys++] = ((int64_t)b * seq_len + t) * kv_row + (int64_t)g * head_dim;
        const uint16_t *q_row = q + (((int64_t)b * seq_len + i) * n_q_heads + h) * head_dim;
        int rc = attend_one(q_row, head_dim, scale, k, v, off, nkeys, s, out + it * head_dim,
                            NULL);
        if (rc != 0) {
#pragma omp critical
            {
                status = ORACLE_EMPTY_KEYSET;
            }
        }
        free(off);
        free(s);
    }
    return status;
}
