/*
 * CPU oracle for one paged-attention step. TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this code. The CUDA library neither links nor calls it, and it shares no
 * source with the library.
 *
 * Everything here is plain and slow on purpose: fp64 arithmetic, an explicit
 * gather through the block table, and a two-pass softmax (maximum, then
 * normalised weights, then the weighted sum of V). No tiling, no online
 * softmax, no reordering.
 *
 * Sources (vLLM inference notes, "AI Infra入门干货总结：大模型是如何高效推理的"):
 *   - §Paged Attention, KV cache layout: per layer and per K/V, the cache is
 *     [num_blocks, block_size, num_kv_heads, head_dim].
 *   - §Paged Attention, block_table: [max_num_reqs, max_num_blocks_per_req],
 *     the physical block of each logical block of a request.
 *   - §Paged Attention, slot_mapping and address computation:
 *     slot = block * block_size + offset; block = slot / block_size;
 *     offset = slot % block_size.
 *   - §LLM 推理全流程 3, Attention: K/V are [seq_lens, num_kv_heads, head_dim]
 *     read discretely from the paged cache; Q is [query_lens, num_heads,
 *     head_dim]; GQA maps one KV head to a group of query heads by index.
 *   - §Continuous Batching: a request schedules num_tokens - num_computed_tokens
 *     query tokens, so query i of a chunk sits at absolute position
 *     (seq_len - query_len) + i and sees keys 0 .. that position (causal).
 * The plain attention definition softmax(q k^T / sqrt(d)) v is the one the
 * operators article ("lpnh.cn/news/2669538", §2.1) prints as its naive
 * reference; here the scale is an argument.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes):
 *   - seq_lens counts every KV token, including this step's new ones.
 *   - GQA groups are contiguous: kv_head = head / (num_heads / num_kv_heads).
 *   - slot_mapping is int64; a negative entry means "skip this token".
 *   - two tokens of one call may not name the same slot.
 *   - block_table entries past ceil(seq_len / block_size) are never read.
 *   - the scale is used as the exact double value of the float argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_SLOT_RANGE (-2)
#define ORACLE_ERR_SLOT_DUPLICATE (-3)
#define ORACLE_ERR_BLOCK_RANGE (-4)
#define ORACLE_ERR_LENGTHS (-5)
#define ORACLE_ERR_NOMEM (-6)

#define ORACLE_BF16 0
#define ORACLE_FP16 1
#define ORACLE_FP8_E4M3 2 /* 8-bit cache codes (see the FP8 section below) */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * IEEE 754 binary16: sign bit, 5-bit exponent with bias 15, 10-bit fraction.
 * Exponent 0 holds zero and the subnormals fraction * 2^-24; exponent 31
 * holds the infinities (fraction 0) and NaNs; otherwise the value is
 * (1024 + fraction) * 2^(exponent - 25). Every value is exact in a double.
 */
static double fp16_to_double(uint16_t h)
{
    const int sign = h >> 15;
    const int e = (h >> 10) & 0x1f;
    const int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

static double elem_to_double(int32_t dtype, uint16_t h)
{
    return dtype == ORACLE_FP16 ? fp16_to_double(h) : bf16_to_double(h);
}

/*
 * Round a double to the nearest element of a binary floating-point format
 * with `mant` stored fraction bits, exponent bias `bias` and largest exponent
 * `emax` (bf16: 7, 127, 127; fp16: 10, 15, 15), ties to even, directly from
 * the double (no intermediate float). Overflow goes to infinity, NaN to the
 * format's quiet NaN. Returns the 16-bit pattern.
 */
static uint16_t round_to_format(double x, int mant, int bias, int emax)
{
    const int ebits = (mant == 7) ? 8 : 5;
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
    const uint16_t inf = (uint16_t)(((1u << ebits) - 1) << mant);
    if (isnan(x))
        return (uint16_t)(inf | (1u << (mant - 1)));
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | inf);
    if (a == 0.0)
        return sign;
    const int emin = 1 - bias;
    int k;
    (void)frexp(a, &k); /* a = f * 2^k, f in [0.5, 1): exponent e = k - 1 */
    int e = k - 1;
    if (e < emin)
        e = emin; /* subnormal range: fixed quantum */
    const double q = ldexp(1.0, e - mant);
    const double n = a / q; /* exact: q is a power of two */
    double r = floor(n);
    const double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    const double v = r * q;
    if (v == 0.0)
        return sign;
    (void)frexp(v, &k);
    int ev = k - 1;
    if (ev > emax)
        return (uint16_t)(sign | inf);
    if (ev < emin) /* subnormal: exponent field 0 */
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, emin - mant)));
    const uint32_t frac_bits = (uint32_t)(v / ldexp(1.0, ev - mant)) - (1u << mant);
    return (uint16_t)(sign | (uint16_t)((uint32_t)(ev + bias) << mant) | frac_bits);
}

static uint16_t double_to_elem(int32_t dtype, double x)
{
    return dtype == ORACLE_FP16 ? round_to_format(x, 10, 15, 15) : round_to_format(x, 7, 127, 127);
}

/* The rounding over an array, for the tests that pin it. */
int oracle_round_elements(const double *x, int64_t n, int32_t dtype, uint16_t *out)
{
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP16)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = double_to_elem(dtype, x[i]);
    return 0;
}

/* The element decoders over an array, for the tests that pin them. */
int oracle_decode_elements(const uint16_t *bits, int64_t n, int32_t dtype, double *out)
{
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP16)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = elem_to_double(dtype, bits[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 (E4M3) cache codes                                                    */
/* ------------------------------------------------------------------------ */

/*
 * KV-cache quantisation (LLM-infra reading map, §4.2): the cache is stored in
 * 8 bits instead of 16, quantised online as K/V are written and dequantised
 * as attention reads them. The page fixes neither the 8-bit format nor the
 * scale, so the readings are: the E4M3 format (sign, 4-bit exponent with bias
 * 7, 3-bit fraction; no infinities; S.1111.111 is NaN, so the largest finite
 * value is 1.75 * 2^8 = 448) with one float scale per cache:
 *   code  = E4M3(x / scale), the quotient taken in binary32 (correctly
 *           rounded), then rounded to the nearest E4M3 value, ties to even,
 *           with magnitudes beyond 448 saturating to 448;
 *   value = decode(code) * scale, exact in a double.
 */

/* Exponent 0: the subnormals fraction * 2^-9; otherwise (8 + fraction) * 2^(exponent - 10). */
static double e4m3_to_double(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, f = c & 7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

/*
 * Nearest E4M3 code to x, ties to the even fraction, saturating at 448; a NaN
 * gives the NaN code 0x7F. The spacing of representable values is 2^-9 below
 * 2^-6 (the subnormals) and 2^(E - 3) within the binade [2^E, 2^(E+1)).
 */
static uint8_t e4m3_from_double(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;
    int E;
    frexp(a, &E); /* a = m * 2^E with m in [0.5, 1): a lies in [2^(E-1), 2^E) */
    int e_unb = E - 1;
    if (e_unb < -6)
        e_unb = -6; /* the subnormal range shares the spacing of [2^-6, 2^-5) */
    double quantum = ldexp(1.0, e_unb - 3);
    double n = a / quantum; /* exact: a power-of-two division */
    double fl = floor(n);
    double rem = n - fl;
    double r = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    double v = r * quantum; /* a representable value: exact */
    if (v >= 448.0)
        return sign | 0x7E;
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6))
        return sign | (uint8_t)(v / ldexp(1.0, -9)); /* exponent 0, fraction = v / 2^-9 */
    frexp(v, &E);
    int e = E - 1;                                  /* v in [2^e, 2^(e+1)) */
    int f = (int)(v / ldexp(1.0, e) * 8.0) - 8;     /* 3-bit fraction */
    return sign | (uint8_t)(((e + 7) << 3) | f);
}

/* The binary32 quotient x / scale of one 16-bit element, then its code. */
static uint8_t quantize_elem(int32_t dtype, uint16_t h, float scale)
{
    float xf = (float)elem_to_double(dtype, h); /* exact: 16-bit floats widen exactly */
    float qf = xf / scale;                      /* binary32 division, correctly rounded */
    return e4m3_from_double((double)qf);
}

int oracle_fp8_decode(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_to_double(codes[i]);
    return ORACLE_OK;
}

int oracle_fp8_round(const double *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_from_double(x[i]);
    return ORACLE_OK;
}

int oracle_fp8_quantize(const uint16_t *bits, int64_t n, int32_t dtype, float scale, uint8_t *out)
{
    if ((dtype != ORACLE_BF16 && dtype != ORACLE_FP16) || !(scale > 0.0f) || isinf(scale))
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        out[i] = quantize_elem(dtype, bits[i], scale);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Step 1: reshape_and_cache                                                 */
/* ------------------------------------------------------------------------ */

/*
 * For every token t whose slot s = slot_mapping[t] is not negative, copy the
 * raw bits of key[t, :, :] to key_cache[s / block_size, s % block_size, :, :]
 * and likewise for value (§Paged Attention: slot_mapping tells the kernel
 * where to write new KV; address computation).
 */
int oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                             uint16_t *key_cache, uint16_t *value_cache,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int64_t num_blocks)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return ORACLE_ERR_ARG;
    if (num_tokens == 0)
        return ORACLE_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping)
        return ORACLE_ERR_ARG;

    const int64_t row = (int64_t)num_kv_heads * head_dim; /* elements per token row */
    const int64_t num_slots = num_blocks * block_size;

    /* Reject out-of-range or repeated slots before writing anything. */
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s >= num_slots)
            return ORACLE_ERR_SLOT_RANGE;
        if (s < 0)
            continue;
        for (int64_t u = 0; u < t; ++u)
            if (slot_mapping[u] == s)
                return ORACLE_ERR_SLOT_DUPLICATE;
    }

    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        int64_t block = s / block_size;
        int64_t offset = s % block_size;
        int64_t dst = (block * block_size + offset) * row;
        for (int64_t e = 0; e < row; ++e) {
            key_cache[dst + e] = key[t * row + e];
            value_cache[dst + e] = value[t * row + e];
        }
    }
    return ORACLE_OK;
}

/*
 * reshape_and_cache into 8-bit caches: the same slots as above, each element
 * quantised on the way in (code = E4M3(x / k_scale) for K, v_scale for V;
 * LLM-infra reading map, §4.2: quantise online as the cache is written).
 */
int oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value,
                                 uint8_t *key_cache, uint8_t *value_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int64_t num_blocks, int32_t dtype,
                                 float k_scale, float v_scale)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return ORACLE_ERR_ARG;
    if ((dtype != ORACLE_BF16 && dtype != ORACLE_FP16) || !(k_scale > 0.0f) || !(v_scale > 0.0f) ||
        isinf(k_scale) || isinf(v_scale))
        return ORACLE_ERR_ARG;
    if (num_tokens == 0)
        return ORACLE_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping)
        return ORACLE_ERR_ARG;

    const int64_t row = (int64_t)num_kv_heads * head_dim;
    const int64_t num_slots = num_blocks * block_size;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s >= num_slots)
            return ORACLE_ERR_SLOT_RANGE;
        if (s < 0)
            continue;
        for (int64_t u = 0; u < t; ++u)
            if (slot_mapping[u] == s)
                return ORACLE_ERR_SLOT_DUPLICATE;
    }
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        int64_t dst = ((s / block_size) * block_size + s % block_size) * row;
        for (int64_t e = 0; e < row; ++e) {
            key_cache[dst + e] = quantize_elem(dtype, key[t * row + e], k_scale);
            value_cache[dst + e] = quantize_elem(dtype, value[t * row + e], v_scale);
        }
    }
    return ORACLE_OK;
}

/*
 * Copy-on-write block copy (§2.2 of the LLM-infra reading map: a shared block
 * is copied before a request writes into it): for each pair, the raw bits of
 * physical block mapping[2i] become those of block mapping[2i+1], in both
 * caches. block_elems = block_size * num_kv_heads * head_dim. Rejects ids out
 * of range, repeated destinations and destinations that are also sources.
 */
int oracle_copy_blocks(uint16_t *key_cache, uint16_t *value_cache, const int64_t *mapping,
                       int64_t num_pairs, int64_t block_elems, int64_t num_blocks)
{
    if (num_pairs < 0 || block_elems <= 0 || num_blocks < 0)
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = mapping[2 * i], dst = mapping[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return ORACLE_ERR_BLOCK_RANGE;
        for (int64_t k = 0; k < num_pairs; ++k) {
            if (k != i && mapping[2 * k + 1] == dst)
                return ORACLE_ERR_SLOT_DUPLICATE;
            if (mapping[2 * k] == dst)
                return ORACLE_ERR_ARG;
        }
    }
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = mapping[2 * i], dst = mapping[2 * i + 1];
        memcpy(key_cache + dst * block_elems, key_cache + src * block_elems, sizeof(uint16_t) * block_elems);
        memcpy(value_cache + dst * block_elems, value_cache + src * block_elems, sizeof(uint16_t) * block_elems);
    }
    return ORACLE_OK;
}

/*
 * Rotary position embedding applied on the way into the cache (§LLM 推理全流程
 * 2 of the vLLM notes: a token's position is a rotation angle, with a
 * precomputed cos_sin_cache of shape [max_position, rotary_dim]).
 * Row p of the cache holds cos(p * theta_i) in columns i < rotary_dim / 2 and
 * sin(p * theta_i) in the next rotary_dim / 2. Each rotated pair (x1, x2)
 * becomes (x1 cos - x2 sin, x2 cos + x1 sin); pairs are element i with
 * i + rotary_dim / 2 (is_neox) or elements 2i and 2i + 1, for
 * i < rotary_dim / 2; elements at rotary_dim and above are unchanged. The
 * rotation is computed in double from the decoded elements and the float
 * cache entries and rounded once to the element type.
 * For each token t with positions[t] in [0, max_position): q[t] (every head)
 * is rotated in place; if slot_mapping[t] >= 0, the rotated key[t] and the
 * unchanged value[t] are written to the slot as reshape_and_cache does.
 * A token whose position is out of range is an error (ORACLE_ERR_ARG).
 */
static void rotate_row(uint16_t *dst, const uint16_t *src, int32_t D, const float *cs, int32_t rot,
                       int32_t is_neox, int32_t dtype)
{
    const int32_t half = rot / 2;
    for (int32_t d = 0; d < D; ++d)
        dst[d] = src[d];
    for (int32_t i = 0; i < half; ++i) {
        const int32_t a = is_neox ? i : 2 * i;
        const int32_t b = is_neox ? i + half : 2 * i + 1;
        const double x1 = elem_to_double(dtype, src[a]), x2 = elem_to_double(dtype, src[b]);
        const double c = (double)cs[i], s = (double)cs[half + i];
        dst[a] = double_to_elem(dtype, x1 * c - x2 * s);
        dst[b] = double_to_elem(dtype, x2 * c + x1 * s);
    }
}

int oracle_rope_reshape_and_cache(uint16_t *q, const uint16_t *key, const uint16_t *value,
                                  uint16_t *key_cache, uint16_t *value_cache, const int64_t *slot_mapping,
                                  const int64_t *positions, const float *cos_sin_cache, int32_t max_position,
                                  int32_t rotary_dim, int32_t is_neox, int64_t num_tokens, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                  int32_t dtype)
{
    if (num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        rotary_dim <= 0 || rotary_dim % 2 || rotary_dim > head_dim || max_position <= 0 ||
        (dtype != ORACLE_BF16 && dtype != ORACLE_FP16))
        return ORACLE_ERR_ARG;
    const int64_t D = head_dim;
    uint16_t *tmp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)D);
    if (!tmp)
        return ORACLE_ERR_NOMEM;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t pos = positions[t];
        if (pos < 0 || pos >= max_position) {
            free(tmp);
            return ORACLE_ERR_ARG;
        }
        const float *cs = cos_sin_cache + pos * rotary_dim;
        for (int32_t h = 0; h < num_heads; ++h) {
            uint16_t *row = q + (t * num_heads + h) * D;
            rotate_row(tmp, row, head_dim, cs, rotary_dim, is_neox, dtype);
            memcpy(row, tmp, sizeof(uint16_t) * (size_t)D);
        }
        const int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_blocks * block_size) {
            free(tmp);
            return ORACLE_ERR_SLOT_RANGE;
        }
        const int64_t row = (int64_t)num_kv_heads * D; /* cache row of slot s starts at s * row */
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            rotate_row(key_cache + s * row + h * D, key + (t * num_kv_heads + h) * D, head_dim, cs, rotary_dim,
                       is_neox, dtype);
            memcpy(value_cache + s * row + h * D, value + (t * num_kv_heads + h) * D, sizeof(uint16_t) * (size_t)D);
        }
    }
    free(tmp);
    return ORACLE_OK;
}

/*
 * The same rotation into 8-bit caches: q is rotated in place as above; the
 * rotated key row (rounded once to the element type, as above) and the value
 * row are stored as E4M3 codes of x / k_scale and x / v_scale, i.e. exactly
 * the rotation followed by oracle_reshape_and_cache_fp8's quantisation.
 */
int oracle_rope_reshape_and_cache_fp8(uint16_t *q, const uint16_t *key, const uint16_t *value,
                                      uint8_t *key_cache, uint8_t *value_cache, const int64_t *slot_mapping,
                                      const int64_t *positions, const float *cos_sin_cache, int32_t max_position,
                                      int32_t rotary_dim, int32_t is_neox, int64_t num_tokens, int32_t num_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                      int32_t dtype, float k_scale, float v_scale)
{
    if (num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        rotary_dim <= 0 || rotary_dim % 2 || rotary_dim > head_dim || max_position <= 0 ||
        (dtype != ORACLE_BF16 && dtype != ORACLE_FP16) || !(k_scale > 0.0f) || !(v_scale > 0.0f) ||
        isinf(k_scale) || isinf(v_scale))
        return ORACLE_ERR_ARG;
    const int64_t D = head_dim;
    uint16_t *tmp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)D);
    if (!tmp)
        return ORACLE_ERR_NOMEM;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t pos = positions[t];
        if (pos < 0 || pos >= max_position) {
            free(tmp);
            return ORACLE_ERR_ARG;
        }
        const float *cs = cos_sin_cache + pos * rotary_dim;
        for (int32_t h = 0; h < num_heads; ++h) {
            uint16_t *row = q + (t * num_heads + h) * D;
            rotate_row(tmp, row, head_dim, cs, rotary_dim, is_neox, dtype);
            memcpy(row, tmp, sizeof(uint16_t) * (size_t)D);
        }
        const int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_blocks * block_size) {
            free(tmp);
            return ORACLE_ERR_SLOT_RANGE;
        }
        const int64_t row = (int64_t)num_kv_heads * D;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            rotate_row(tmp, key + (t * num_kv_heads + h) * D, head_dim, cs, rotary_dim, is_neox, dtype);
            for (int64_t d = 0; d < D; ++d) {
                key_cache[s * row + h * D + d] = quantize_elem(dtype, tmp[d], k_scale);
                value_cache[s * row + h * D + d] = quantize_elem(dtype, value[(t * num_kv_heads + h) * D + d], v_scale);
            }
        }
    }
    free(tmp);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Step 2: attention over the paged cache                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;
    const void *key_cache;   /* 16-bit elements, or 8-bit codes when kv_dtype is ORACLE_FP8_E4M3 */
    const void *value_cache;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    const int32_t *query_start_loc;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int64_t num_blocks;
    double scale;
    int32_t dtype;    /* ORACLE_BF16 or ORACLE_FP16: how q's 16-bit elements decode */
    int32_t kv_dtype; /* dtype (16-bit caches) or ORACLE_FP8_E4M3 */
    double k_scale;   /* 8-bit caches: K value = decode(code) * k_scale */
    double v_scale;
} problem_t;

static int check_problem(const problem_t *p)
{
    if (p->num_seqs < 0 || p->num_heads <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0 ||
        p->block_size <= 0 || p->max_blocks_per_seq < 0 || p->num_blocks < 0)
        return ORACLE_ERR_ARG;
    if (p->num_heads % p->num_kv_heads != 0)
        return ORACLE_ERR_ARG;
    if (p->dtype != ORACLE_BF16 && p->dtype != ORACLE_FP16)
        return ORACLE_ERR_ARG;
    if (p->kv_dtype != p->dtype && p->kv_dtype != ORACLE_FP8_E4M3)
        return ORACLE_ERR_ARG;
    if (p->kv_dtype == ORACLE_FP8_E4M3 &&
        (!(p->k_scale > 0.0) || !(p->v_scale > 0.0) || isinf(p->k_scale) || isinf(p->v_scale)))
        return ORACLE_ERR_ARG;
    if (p->query_start_loc[0] != 0)
        return ORACLE_ERR_LENGTHS;
    for (int32_t b = 0; b < p->num_seqs; ++b) {
        int32_t ql = p->query_start_loc[b + 1] - p->query_start_loc[b];
        int32_t L = p->seq_lens[b];
        if (ql < 0 || L < ql)
            return ORACLE_ERR_LENGTHS;
        if ((int64_t)L > (int64_t)p->max_blocks_per_seq * p->block_size)
            return ORACLE_ERR_LENGTHS;
        int32_t nblk = (L + p->block_size - 1) / p->block_size;
        for (int32_t i = 0; i < nblk; ++i) {
            int32_t blk = p->block_tables[(int64_t)b * p->max_blocks_per_seq + i];
            if (blk < 0 || (int64_t)blk >= p->num_blocks)
                return ORACLE_ERR_BLOCK_RANGE;
        }
    }
    return ORACLE_OK;
}

/* Element idx of a cache as a double: a 16-bit element, or an 8-bit code times its scale. */
static double cache_value(const problem_t *p, const void *cache, int64_t idx, double scale)
{
    if (p->kv_dtype == ORACLE_FP8_E4M3)
        return e4m3_to_double(((const uint8_t *)cache)[idx]) * scale;
    return elem_to_double(p->dtype, ((const uint16_t *)cache)[idx]);
}

/*
 * Gather the logical K and V rows 0..L-1 of request b, KV head kvh, into
 * contiguous [L, head_dim] arrays of doubles. Logical token j lives in
 * physical block block_tables[b][j / block_size] at offset j % block_size.
 */
static void gather_request(const problem_t *p, int32_t b, int32_t kvh, double *K, double *V)
{
    const int32_t L = p->seq_lens[b];
    const int32_t D = p->head_dim;
    for (int32_t j = 0; j < L; ++j) {
        int32_t logical_block = j / p->block_size;
        int32_t offset = j % p->block_size;
        int64_t phys = p->block_tables[(int64_t)b * p->max_blocks_per_seq + logical_block];
        int64_t slot = phys * p->block_size + offset;
        int64_t base = (slot * p->num_kv_heads + kvh) * D;
        for (int32_t d = 0; d < D; ++d) {
            K[(int64_t)j * D + d] = cache_value(p, p->key_cache, base + d, p->k_scale);
            V[(int64_t)j * D + d] = cache_value(p, p->value_cache, base + d, p->v_scale);
        }
    }
}

/*
 * Softmax weights of query token (q0 + i), head h, over its visible keys.
 * Returns the number of visible keys n; w[0..n-1] receives the weights.
 * Two passes: the maximum score first, then exp(s - max) / sum.
 */
static int32_t weights_for_query(const problem_t *p, int32_t b, int32_t i, int32_t h,
                                 const double *K, double *w)
{
    const int32_t D = p->head_dim;
    const int32_t q0 = p->query_start_loc[b];
    const int32_t ql = p->query_start_loc[b + 1] - q0;
    const int32_t L = p->seq_lens[b];
    const int32_t ctx = L - ql;
    const int32_t n = ctx + i + 1; /* keys 0 .. ctx + i */
    const uint16_t *qrow = p->q + ((int64_t)(q0 + i) * p->num_heads + h) * D;

    double qd[1024];
    double *qv = qd;
    double *heap = NULL;
    if (D > 1024) {
        heap = (double *)malloc(sizeof(double) * D);
        qv = heap;
    }
    for (int32_t d = 0; d < D; ++d)
        qv[d] = elem_to_double(p->dtype, qrow[d]);

    for (int32_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += qv[d] * K[(int64_t)j * D + d];
        w[j] = p->scale * dot;
    }
    free(heap);

    double m = -INFINITY;
    for (int32_t j = 0; j < n; ++j)
        if (w[j] > m)
            m = w[j];
    double z = 0.0;
    for (int32_t j = 0; j < n; ++j) {
        w[j] = exp(w[j] - m);
        z += w[j];
    }
    for (int32_t j = 0; j < n; ++j)
        w[j] /= z;
    return n;
}

/* out[d] = sum_j w[j] * V[j][d] */
static void weighted_sum(const double *w, int32_t n, const double *V, int32_t D, double *out)
{
    for (int32_t d = 0; d < D; ++d)
        out[d] = 0.0;
    for (int32_t j = 0; j < n; ++j)
        for (int32_t d = 0; d < D; ++d)
            out[d] += w[j] * V[(int64_t)j * D + d];
}

/* All query rows of request b for head h -> out[(q0 + i), h, :]. */
static int attend_request_head(const problem_t *p, int32_t b, int32_t h, double *out)
{
    const int32_t D = p->head_dim;
    const int32_t G = p->num_heads / p->num_kv_heads;
    const int32_t kvh = h / G;
    const int32_t q0 = p->query_start_loc[b];
    const int32_t ql = p->query_start_loc[b + 1] - q0;
    const int32_t L = p->seq_lens[b];
    if (ql == 0)
        return ORACLE_OK;
    double *K = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
    double *V = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
    double *w = (double *)malloc(sizeof(double) * ((size_t)L + 1));
    if (!K || !V || !w) {
        free(K); free(V); free(w);
        return ORACLE_ERR_NOMEM;
    }
    gather_request(p, b, kvh, K, V);
    for (int32_t i = 0; i < ql; ++i) {
        int32_t n = weights_for_query(p, b, i, h, K, w);
        weighted_sum(w, n, V, D, out + ((int64_t)(q0 + i) * p->num_heads + h) * D);
    }
    free(K); free(V); free(w);
    return ORACLE_OK;
}

/* A tiny thread pool over independent (request, head) items. */
typedef struct {
    const problem_t *p;
    double *out;
    int64_t n_items;
    int64_t next;
    pthread_mutex_t lock;
    int status;
} pool_t;

static void *pool_worker(void *arg)
{
    pool_t *pool = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&pool->lock);
        int64_t it = pool->next++;
        pthread_mutex_unlock(&pool->lock);
        if (it >= pool->n_items)
            break;
        int32_t b = (int32_t)(it / pool->p->num_heads);
        int32_t h = (int32_t)(it % pool->p->num_heads);
        int rc = attend_request_head(pool->p, b, h, pool->out);
        if (rc != ORACLE_OK) {
            pthread_mutex_lock(&pool->lock);
            pool->status = rc;
            pthread_mutex_unlock(&pool->lock);
        }
    }
    return NULL;
}

/*
 * out: [total_q, num_heads, head_dim] doubles. Rows of requests with
 * query_len 0 are absent (total_q counts only scheduled tokens).
 */
int oracle_attention_varlen(const uint16_t *q, const void *key_cache,
                            const void *value_cache, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens,
                            const int32_t *query_start_loc, int32_t num_seqs,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int64_t num_blocks, float scale, int32_t dtype,
                            int32_t kv_dtype, float k_scale, float v_scale,
                            double *out, int32_t num_threads)
{
    problem_t p = {q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                   query_start_loc, num_seqs, num_heads, num_kv_heads, head_dim,
                   block_size, num_blocks, (double)scale, dtype, kv_dtype, (double)k_scale, (double)v_scale};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK)
        return rc;
    pool_t pool;
    pool.p = &p;
    pool.out = out;
    pool.n_items = (int64_t)num_seqs * num_heads;
    pool.next = 0;
    pool.status = ORACLE_OK;
    pthread_mutex_init(&pool.lock, NULL);
    if (num_threads < 1)
        num_threads = 1;
    if (num_threads == 1) {
        pool_worker(&pool);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * num_threads);
        if (!th)
            return ORACLE_ERR_NOMEM;
        for (int32_t t = 0; t < num_threads; ++t)
            pthread_create(&th[t], NULL, pool_worker, &pool);
        for (int32_t t = 0; t < num_threads; ++t)
            pthread_join(th[t], NULL);
        free(th);
    }
    pthread_mutex_destroy(&pool.lock);
    return pool.status;
}

/*
 * The same definition for a chosen list of (query token, head) pairs, so that
 * full-size problems can be checked at sampled outputs. out: [n_samples, head_dim].
 */
int oracle_attention_sampled(const uint16_t *q, const void *key_cache,
                             const void *value_cache, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *seq_lens,
                             const int32_t *query_start_loc, int32_t num_seqs,
                             int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int64_t num_blocks, float scale, int32_t dtype,
                            int32_t kv_dtype, float k_scale, float v_scale,
                             int64_t n_samples, const int64_t *sample_token,
                             const int32_t *sample_head, double *out)
{
    problem_t p = {q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                   query_start_loc, num_seqs, num_heads, num_kv_heads, head_dim,
                   block_size, num_blocks, (double)scale, dtype, kv_dtype, (double)k_scale, (double)v_scale};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK)
        return rc;
    const int32_t D = head_dim;
    const int32_t G = num_heads / num_kv_heads;
    for (int64_t s = 0; s < n_samples; ++s) {
        int64_t t = sample_token[s];
        int32_t h = sample_head[s];
        if (t < 0 || t >= query_start_loc[num_seqs] || h < 0 || h >= num_heads)
            return ORACLE_ERR_ARG;
        int32_t b = 0;
        while (!(query_start_loc[b] <= t && t < query_start_loc[b + 1]))
            ++b;
        int32_t i = (int32_t)(t - query_start_loc[b]);
        int32_t L = seq_lens[b];
        double *K = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
        double *V = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
        double *w = (double *)malloc(sizeof(double) * ((size_t)L + 1));
        if (!K || !V || !w) {
            free(K); free(V); free(w);
            return ORACLE_ERR_NOMEM;
        }
        gather_request(&p, b, h / G, K, V);
        int32_t n = weights_for_query(&p, b, i, h, K, w);
        weighted_sum(w, n, V, D, out + s * D);
        free(K); free(V); free(w);
    }
    return ORACLE_OK;
}

/*
 * Softmax weights of one (query token, head) pair over its visible keys, for
 * the tests' checks of the weights themselves. weights: at least seq_len
 * doubles. Returns the number of visible keys, or a negative error code.
 */
int oracle_attention_weights(const uint16_t *q, const void *key_cache,
                             const void *value_cache, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *seq_lens,
                             const int32_t *query_start_loc, int32_t num_seqs,
                             int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int64_t num_blocks, float scale, int32_t dtype,
                            int32_t kv_dtype, float k_scale, float v_scale,
                             int64_t token, int32_t head, double *weights)
{
    problem_t p = {q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                   query_start_loc, num_seqs, num_heads, num_kv_heads, head_dim,
                   block_size, num_blocks, (double)scale, dtype, kv_dtype, (double)k_scale, (double)v_scale};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK)
        return rc;
    if (token < 0 || token >= query_start_loc[num_seqs] || head < 0 || head >= num_heads)
        return ORACLE_ERR_ARG;
    int32_t b = 0;
    while (!(query_start_loc[b] <= token && token < query_start_loc[b + 1]))
        ++b;
    int32_t L = seq_lens[b];
    const int32_t D = head_dim;
    double *K = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
    double *V = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
    if (!K || !V) {
        free(K); free(V);
        return ORACLE_ERR_NOMEM;
    }
    gather_request(&p, b, head / (num_heads / num_kv_heads), K, V);
    int32_t n = weights_for_query(&p, b, (int32_t)(token - query_start_loc[b]), head, K, weights);
    free(K); free(V);
    return n;
}
