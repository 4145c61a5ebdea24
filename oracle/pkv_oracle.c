/*
 * pkv_oracle.c -- plain, slow, obviously-correct CPU oracle for the paged-KV
 * hot path.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product library never does, and
 * this file shares no code, header, table or helper with the CUDA path.
 *
 * Every floating-point result is computed in IEEE binary64 from inputs widened
 * exactly from their storage type.  Loops follow the definitions on the pages
 * one element at a time; nothing is blocked, fused or reordered.
 *
 * Sources (page title -- section):
 *   [P1] "Block-Paged KV Cache" (Hurray format documentation)
 *        -- "The three buffers", "Element lookup through the block table",
 *           "Validating the storage invariants".
 *   [P3] "Paged KV Cache - AI infra interview lesson"
 *        -- "Walk the Shapes First", "Step 1: slot_mapping and store_kvcache",
 *           "Step 2: paged_attention_decode".
 *
 * Readings where the pages leave a step open are stated beside each function.
 * Every function here is pinned by a CPU test against a value the pages print,
 * a closed form, a library routine or brute force; none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Storage types of q / key / value / caches / page pool. */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ---------------------------------------------------------------------------
 * Exact widening of the storage types to binary64.
 * ------------------------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_widen_f16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1F;
    int frac = bits & 0x3FF;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);              /* zero / subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp(1024.0 + (double)frac, expo - 25); /* (1 + frac/2^10) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
double orc_widen_bf16(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* orc_widen_f16 evaluated once for every bit pattern, so that full-size
 * inputs do not pay an ldexp per element; the values are the function's. */
static double f16_table[1 << 16];
static int f16_table_ready = 0;

static void build_f16_table(void)
{
    if (f16_table_ready) return;
    for (uint32_t b = 0; b < (1u << 16); ++b) f16_table[b] = orc_widen_f16((uint16_t)b);
    f16_table_ready = 1;
}

static double load_elem(const void *base, int64_t idx, int dtype)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char *)base + idx * 4, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)base + idx * 2, 2);
    return dtype == ORC_F16 ? f16_table[h] : orc_widen_bf16(h);
}

/* ---------------------------------------------------------------------------
 * [P3] "Walk the Shapes First": the slot of position p of a sequence is
 * block_table[p // bs] * bs + p % bs.  Returns -1 when the position has no
 * block (beyond the table row, or a negative entry), which the caller reports.
 * ------------------------------------------------------------------------- */
int64_t orc_slot_of_position(const int32_t *bt_row, int32_t max_blocks,
                             int64_t p, int32_t bs)
{
    int64_t logical_block = p / bs;
    if (p < 0 || logical_block >= max_blocks) return -1;
    int32_t phys = bt_row[logical_block];
    if (phys < 0) return -1;
    return (int64_t)phys * bs + p % bs;
}

/* [P3] "Step 1: slot_mapping and store_kvcache": the mapping covers only the
 * tokens computed in this step, positions [start_b, end_b) of every sequence b,
 * laid out sequence after sequence.  The oracle applies the per-position formula
 * above (the page's range-per-block form is checked against it by the tests).
 * Reading: a position with no valid block, or whose block id is >= num_blocks,
 * is written as -1 and counted in the return value.  Returns the number of such
 * errors; writes sum(end-start) entries. */
int64_t orc_compute_slot_mapping(const int32_t *block_tables, int32_t max_blocks,
                                 const int32_t *starts, const int32_t *ends,
                                 int32_t num_seqs, int32_t bs, int32_t num_blocks,
                                 int32_t *slot_mapping)
{
    int64_t k = 0, errors = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t *row = block_tables + (int64_t)b * max_blocks;
        for (int64_t p = starts[b]; p < ends[b]; ++p) {
            int64_t slot = orc_slot_of_position(row, max_blocks, p, bs);
            if (slot < 0 || slot >= (int64_t)num_blocks * bs) {
                slot = -1;
                ++errors;
            }
            slot_mapping[k++] = (int32_t)slot;
        }
    }
    return errors;
}

/* [P3] "Step 1": the cache is viewed as [num_blocks * bs, H_kv * d] rows and
 * row slot_mapping[i] receives token i's key (and value); a slot of -1 is
 * padding and is not written.  Rows are moved as raw bytes.  Reading: any
 * other slot outside [0, num_slots) is not written and is counted. */
int64_t orc_store_kvcache(const void *key, const void *value, void *k_cache, void *v_cache,
                          const int32_t *slot_mapping, int64_t num_tokens,
                          int64_t row_bytes, int64_t num_slots)
{
    int64_t errors = 0;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) { ++errors; continue; }
        memcpy((char *)k_cache + slot * row_bytes, (const char *)key + i * row_bytes, (size_t)row_bytes);
        memcpy((char *)v_cache + slot * row_bytes, (const char *)value + i * row_bytes, (size_t)row_bytes);
    }
    return errors;
}

/* [P3] "Step 2: paged_attention_decode".  For sequence b with context length n:
 * n_blk = ceil(n / bs) blocks are taken from the block-table row (entries past
 * n_blk may be -1 and are never read); token t < n lives in row
 * block_table[b][t // bs] * bs + t % bs of the cache [num_blocks, bs, H_kv, d];
 * query head h reads KV head h // (Hq / H_kv); the output is
 *     softmax_t(scale * q[b,h] . K[t]) . V[t]
 * with the usual max subtraction.  Inputs are widened exactly, everything else
 * is binary64.  The result is written as binary64 to out[B, Hq, d].
 * Readings: n == 0 gives a zero row; a block id outside [0, num_blocks) inside
 * n_blk drops that block's tokens from the softmax and is counted; a context
 * length below 0 gives a zero row and is counted.  Returns the error count. */
int64_t orc_paged_attention_decode(double *out, const void *q,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, int32_t max_blocks,
                                   const int32_t *context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t bs, int32_t num_blocks,
                                   double scale, int dtype)
{
    int64_t errors = 0;
    int32_t group = num_q_heads / num_kv_heads;
    build_f16_table();
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t n = context_lens[b];
        const int32_t *row = block_tables + (int64_t)b * max_blocks;
        if (n < 0 || (n + bs - 1) / bs > max_blocks) {
            ++errors;
            n = -1;
        }
        double *scores = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        char *usable = (char *)malloc((size_t)(n > 0 ? n : 1));
        if (n > 0) {
            for (int64_t j = 0; j < (n + bs - 1) / bs; ++j)
                if (row[j] < 0 || row[j] >= num_blocks) ++errors;
        }
        for (int32_t h = 0; h < num_q_heads; ++h) {
            int32_t g = h / group;
            double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int32_t i = 0; i < head_dim; ++i) o[i] = 0.0;
            if (n <= 0) continue;
            int64_t q_base = ((int64_t)b * num_q_heads + h) * head_dim;
            double m = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                int32_t phys = row[t / bs];
                usable[t] = (phys >= 0 && phys < num_blocks);
                if (!usable[t]) continue;
                int64_t cache_row = (int64_t)phys * bs + t % bs;
                int64_t k_base = (cache_row * num_kv_heads + g) * head_dim;
                double s = 0.0;
                for (int32_t i = 0; i < head_dim; ++i)
                    s += load_elem(q, q_base + i, dtype) * load_elem(k_cache, k_base + i, dtype);
                scores[t] = scale * s;
                if (scores[t] > m) m = scores[t];
            }
            if (m == -INFINITY) continue; /* no usable token */
            double l = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                if (!usable[t]) continue;
                scores[t] = exp(scores[t] - m);
                l += scores[t];
            }
            for (int64_t t = 0; t < n; ++t) {
                if (!usable[t]) continue;
                int64_t cache_row = (int64_t)row[t / bs] * bs + t % bs;
                int64_t v_base = (cache_row * num_kv_heads + g) * head_dim;
                double p = scores[t] / l;
                for (int32_t i = 0; i < head_dim; ++i)
                    o[i] += p * load_elem(v_cache, v_base + i, dtype);
            }
        }
        free(scores);
        free(usable);
    }
    return errors;
}

/* ---------------------------------------------------------------------------
 * [P1] CSR block-paged snapshot: page_pool [num_pages, page_size, H, d],
 * block_table (physical page id of every logical page, sequences concatenated),
 * seq_ptr [num_seqs + 1] delimiting each sequence's slice of block_table.
 * Index buffers are u32 or u64 ("BlockTableIndexType").
 * ------------------------------------------------------------------------- */
static uint64_t load_index(const void *buf, int64_t k, int is_u64)
{
    if (is_u64) {
        uint64_t v;
        memcpy(&v, (const char *)buf + k * 8, 8);
        return v;
    }
    uint32_t v;
    memcpy(&v, (const char *)buf + k * 4, 4);
    return v;
}

/*
 * [P1] "Quantization compatibility": the block-paged layout reuses the
 * quantization schemes with one rule.  Per-block-affine scales (scheme tag
 * 0x03) must run along axis 0, the paged axis, with block_size == page_size,
 * so scales stay per page slot; per-channel scales (0x02) along the paged axis
 * are refused (the page's printed cases).  Reading where the page is silent:
 * a tag with no per-position scales (0x00 none, 0x01 per-tensor) is
 * compatible, per-channel along another axis is compatible, and any other tag
 * is refused.  Returns 0 when compatible, else 1 (per-block-affine off the
 * paged axis), 2 (per-block-affine with block_size != page_size),
 * 3 (per-channel on the paged axis), 4 (unknown tag).
 */
int orc_quantization_compatible(int scheme_tag, int axis, int block_size, int page_size) {
    switch (scheme_tag) {
    case 0x00:
    case 0x01:
        return 0;
    case 0x02:
        return axis == 0 ? 3 : 0;
    case 0x03:
        if (axis != 0) return 1;
        return block_size == page_size ? 0 : 2;
    default:
        return 4;
    }
}

/* [P1] "Validating the storage invariants": seq_ptr[0] == 0; seq_ptr is
 * non-decreasing; seq_ptr[num_seqs] == len(block_table); every block_table
 * entry < num_pages.  The empty batch (num_seqs == 0, seq_ptr == [0]) is
 * valid.  Returns 0 when all hold, else the number (1..4) of the first
 * invariant found broken, in that order. */
int orc_validate_index_buffers(const void *seq_ptr, const void *block_table, int is_u64,
                               int64_t num_seqs, int64_t nnz, uint64_t num_pages)
{
    if (load_index(seq_ptr, 0, is_u64) != 0) return 1;
    for (int64_t s = 0; s < num_seqs; ++s)
        if (load_index(seq_ptr, s + 1, is_u64) < load_index(seq_ptr, s, is_u64)) return 2;
    if (load_index(seq_ptr, num_seqs, is_u64) != (uint64_t)nnz) return 3;
    for (int64_t k = 0; k < nnz; ++k)
        if (load_index(block_table, k, is_u64) >= num_pages) return 4;
    return 0;
}

/* [P1] "Element lookup through the block table":
 *   page_in_seq = token / page_size;  offset_in_page = token % page_size;
 *   phys_page   = block_table[seq_ptr[seq] + page_in_seq];
 *   flat        = ((phys_page * page_size + offset_in_page) * num_heads + head) * head_dim + dim
 * Reading of the lookup's error cases (the page returns a Result): seq out of
 * range, page_in_seq outside the sequence's slice, phys_page >= num_pages,
 * head or dim out of range -> -1. */
int64_t orc_element_offset(int64_t seq, int64_t token, int64_t head, int64_t dim,
                           int64_t page_size, uint64_t num_pages, int64_t num_heads,
                           int64_t head_dim, const void *block_table, const void *seq_ptr,
                           int is_u64, int64_t num_seqs)
{
    if (seq < 0 || seq >= num_seqs || token < 0 || head < 0 || head >= num_heads ||
        dim < 0 || dim >= head_dim || page_size <= 0)
        return -1;
    uint64_t page_in_seq = (uint64_t)(token / page_size);
    uint64_t offset_in_page = (uint64_t)(token % page_size);
    uint64_t lo = load_index(seq_ptr, seq, is_u64);
    uint64_t hi = load_index(seq_ptr, seq + 1, is_u64);
    if (lo + page_in_seq >= hi) return -1;
    uint64_t phys = load_index(block_table, (int64_t)(lo + page_in_seq), is_u64);
    if (phys >= num_pages) return -1;
    return (int64_t)(((phys * (uint64_t)page_size + offset_in_page) * (uint64_t)num_heads +
                      (uint64_t)head) * (uint64_t)head_dim + (uint64_t)dim);
}

/* Unpack the snapshot into the contiguous logical tensor [total_tokens, H, d]
 * ([P1] "The three buffers": the logical shape is [total_tokens, num_heads,
 * head_dim]).  Reading: the CSR buffers do not say how many tokens each
 * sequence holds, so the caller passes token_ptr [num_seqs + 1] (sequence s
 * owns logical rows token_ptr[s] .. token_ptr[s+1]-1, in token order).  Every
 * element is resolved independently with the lookup above and copied as raw
 * bytes; an element whose lookup fails is written as zero bytes and counted.
 * Aliased pages are simply read more than once. */
int64_t orc_unpack_block_paged(void *out, const void *page_pool, const void *block_table,
                               const void *seq_ptr, int is_u64, const int64_t *token_ptr,
                               int64_t num_seqs, int64_t page_size, uint64_t num_pages,
                               int64_t num_heads, int64_t head_dim, int64_t elem_bytes)
{
    int64_t errors = 0;
    for (int64_t s = 0; s < num_seqs; ++s) {
        for (int64_t t = 0; t < token_ptr[s + 1] - token_ptr[s]; ++t) {
            for (int64_t h = 0; h < num_heads; ++h) {
                for (int64_t i = 0; i < head_dim; ++i) {
                    int64_t dst = ((token_ptr[s] + t) * num_heads + h) * head_dim + i;
                    int64_t src = orc_element_offset(s, t, h, i, page_size, num_pages, num_heads,
                                                     head_dim, block_table, seq_ptr, is_u64,
                                                     num_seqs);
                    if (src < 0) {
                        memset((char *)out + dst * elem_bytes, 0, (size_t)elem_bytes);
                        ++errors;
                    } else {
                        memcpy((char *)out + dst * elem_bytes,
                               (const char *)page_pool + src * elem_bytes, (size_t)elem_bytes);
                    }
                }
            }
        }
    }
    return errors;
}

/* ---------------------------------------------------------------------------
 * [P1] "Quantization compatibility": an fp8 cache keeps its scales per page
 * slot (per-block-affine with block_size == page_size), so a shared page
 * carries its own scales.  The pages give that placement rule only.  Readings:
 * the codes are OCP 8-bit E4M3 (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448); each
 * (physical block, KV head) has one binary32 scale for K and one for V, laid
 * out [num_blocks, H_kv]; a stored value is scale * decode(code).
 * ------------------------------------------------------------------------- */

/* E4M3 code -> value, from the format's definition. */
double orc_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* subnormal: (m / 8) * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10); /* normal: (1 + m / 8) * 2^(e - 7) */
    return sign ? -v : v;
}

/* binary32 -> E4M3, round to nearest with ties to even, saturating: magnitudes
 * above 448 (infinities included) give +-448; NaN gives the NaN code with the
 * input's sign.  The magnitude is rounded on the quantum of its binade (2^-9
 * below the smallest normal 2^-6) with rint in the default rounding mode. */
uint8_t orc_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    int E, e;
    double v, n;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    if (a > 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;
    frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
    E = e - 1;             /* a = 1.xxx * 2^E */
    if (E < -6) E = -6;
    n = rint(a / ldexp(1.0, E - 3));   /* exact scaling by a power of two, then RN-even */
    v = n * ldexp(1.0, E - 3);
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6))            /* subnormal */
        return (uint8_t)(sign | (int)(v / ldexp(1.0, -9)));
    frexp(v, &e);
    E = e - 1;
    return (uint8_t)(sign | ((E + 7) << 3) | ((int)(v / ldexp(1.0, E - 3)) - 8));
}

/* ---------------------------------------------------------------------------
 * [P1] "Quantization compatibility" names int8 caches beside fp8 ones, with
 * symmetric per-block-affine scales.  Readings: a code is a signed byte c in
 * [-127, 127] standing for scale * c; the scale of a (block, KV head) is
 * max |x| / 127; encoding rounds x / scale to the nearest integer, ties to
 * even, and clamps to [-127, 127]; NaN encodes as 0.
 * ------------------------------------------------------------------------- */

/* binary32 -> int8 code (as above). */
int8_t orc_int8_encode(float y)
{
    double r;
    if (isnan(y)) return 0;
    r = rint((double)y);  /* y is a binary32 value: exact in binary64, rint ties to even */
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

/* Code formats of the quantized caches. */
enum { Q8_E4M3 = 0, Q8_INT8 = 1 };

/* The largest magnitude of a format: the per-block scale is max |x| / this. */
static float q8_max(int fmt) { return fmt == Q8_INT8 ? 127.0f : 448.0f; }

static double q8_decode(uint8_t code, int fmt)
{
    return fmt == Q8_INT8 ? (double)(int8_t)code : orc_e4m3_decode(code);
}

/* The code of x stored with scale s: encode(x / s), the division in binary32
 * (the precision the kernels use); a zero scale stores +0. */
static uint8_t encode_scaled(double x, float s, int fmt)
{
    if (s == 0.0f) return 0;
    if (fmt == Q8_INT8) return (uint8_t)orc_int8_encode((float)x / s);
    return orc_e4m3_encode((float)x / s);
}

/* Quantizes a [num_blocks, bs, H_kv, d] cache of `dtype`: per (block, head),
 * s = max |x| / 448 (E4M3) or / 127 (int8) in binary32 (NaN entries ignored),
 * then every element becomes encode(x / s).  Writes codes
 * [num_blocks, bs, H_kv, d] and scales [num_blocks, H_kv]. */
void orc_quantize_kvcache_q8(const void *src, uint8_t *codes, float *scales, int64_t num_blocks,
                             int64_t bs, int64_t num_kv_heads, int64_t head_dim, int dtype, int fmt)
{
    build_f16_table();
    for (int64_t blk = 0; blk < num_blocks; ++blk) {
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            float amax = 0.0f;
            for (int64_t t = 0; t < bs; ++t)
                for (int64_t i = 0; i < head_dim; ++i) {
                    float a = (float)fabs(load_elem(src, ((blk * bs + t) * num_kv_heads + h) * head_dim + i, dtype));
                    if (a > amax) amax = a;
                }
            float s = amax / q8_max(fmt);
            scales[blk * num_kv_heads + h] = s;
            for (int64_t t = 0; t < bs; ++t)
                for (int64_t i = 0; i < head_dim; ++i) {
                    int64_t idx = ((blk * bs + t) * num_kv_heads + h) * head_dim + i;
                    codes[idx] = encode_scaled(load_elem(src, idx, dtype), s, fmt);
                }
        }
    }
}

/* [P3] "Step 1" for a quantized cache: row slot_mapping[i] of the code caches
 * receives encode(key[i] / s) per element, s the scale of the row's block and
 * head (slot / bs); -1 is skipped, other slots outside [0, num_slots) are
 * counted and skipped.  key/value are [num_tokens, H_kv, d] of `dtype`. */
int64_t orc_store_kvcache_q8(const void *key, const void *value, uint8_t *k_codes, uint8_t *v_codes,
                             const float *k_scale, const float *v_scale, const int32_t *slot_mapping,
                             int64_t num_tokens, int64_t num_kv_heads, int64_t head_dim, int64_t bs,
                             int64_t num_slots, int dtype, int fmt)
{
    int64_t errors = 0;
    build_f16_table();
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) { ++errors; continue; }
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            float sk = k_scale[(slot / bs) * num_kv_heads + h], sv = v_scale[(slot / bs) * num_kv_heads + h];
            for (int64_t d = 0; d < head_dim; ++d) {
                int64_t src = (i * num_kv_heads + h) * head_dim + d;
                int64_t dst = (slot * num_kv_heads + h) * head_dim + d;
                k_codes[dst] = encode_scaled(load_elem(key, src, dtype), sk, fmt);
                v_codes[dst] = encode_scaled(load_elem(value, src, dtype), sv, fmt);
            }
        }
    }
    return errors;
}

/* [P3] "Step 2" over a quantized cache: as orc_paged_attention_decode, with
 * every K/V element read as scale[block][kv head] * decode(code) in binary64. */
int64_t orc_paged_attention_decode_q8(double *out, const void *q, const uint8_t *k_codes,
                                      const uint8_t *v_codes, const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables, int32_t max_blocks,
                                      const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t bs, int32_t num_blocks,
                                      double scale, int q_dtype, int fmt)
{
    int64_t errors = 0;
    int32_t group = num_q_heads / num_kv_heads;
    build_f16_table();
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t n = context_lens[b];
        const int32_t *row = block_tables + (int64_t)b * max_blocks;
        if (n < 0 || (n + bs - 1) / bs > max_blocks) {
            ++errors;
            n = -1;
        }
        double *scores = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        char *usable = (char *)malloc((size_t)(n > 0 ? n : 1));
        if (n > 0) {
            for (int64_t j = 0; j < (n + bs - 1) / bs; ++j)
                if (row[j] < 0 || row[j] >= num_blocks) ++errors;
        }
        for (int32_t h = 0; h < num_q_heads; ++h) {
            int32_t g = h / group;
            double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int32_t i = 0; i < head_dim; ++i) o[i] = 0.0;
            if (n <= 0) continue;
            int64_t q_base = ((int64_t)b * num_q_heads + h) * head_dim;
            double m = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                int32_t phys = row[t / bs];
                usable[t] = (phys >= 0 && phys < num_blocks);
                if (!usable[t]) continue;
                int64_t cache_row = (int64_t)phys * bs + t % bs;
                int64_t k_base = (cache_row * num_kv_heads + g) * head_dim;
                double sk = k_scale[(int64_t)phys * num_kv_heads + g];
                double s = 0.0;
                for (int32_t i = 0; i < head_dim; ++i)
                    s += load_elem(q, q_base + i, q_dtype) * (sk * q8_decode(k_codes[k_base + i], fmt));
                scores[t] = scale * s;
                if (scores[t] > m) m = scores[t];
            }
            if (m == -INFINITY) continue;
            double l = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                if (!usable[t]) continue;
                scores[t] = exp(scores[t] - m);
                l += scores[t];
            }
            for (int64_t t = 0; t < n; ++t) {
                if (!usable[t]) continue;
                int32_t phys = row[t / bs];
                int64_t cache_row = (int64_t)phys * bs + t % bs;
                int64_t v_base = (cache_row * num_kv_heads + g) * head_dim;
                double sv = v_scale[(int64_t)phys * num_kv_heads + g];
                double p = scores[t] / l;
                for (int32_t i = 0; i < head_dim; ++i)
                    o[i] += p * (sv * q8_decode(v_codes[v_base + i], fmt));
            }
        }
        free(scores);
        free(usable);
    }
    return errors;
}

/* ---------------------------------------------------------------------------
 * [P3] "Step 3: varlen attention and cu_seqlens" names prefill attention over
 * sequences of different lengths and gives no further content.  Reading (the
 * plain one the rest of the page supports): sequence b's new tokens occupy
 * positions [start_b, start_b + n_b), n_b = cu_q[b+1] - cu_q[b]; their K/V are
 * already in the paged cache (stored by "Step 1"), as are the K/V of positions
 * [0, start_b) (a cached prefix or earlier chunks).  Query i of sequence b sits
 * at position p = start_b + i and attends causally over positions 0 .. p
 * through the block table:
 *     out[cu_q[b] + i, h] = softmax_{t <= p}(scale * q . K[t]) . V[t],
 * query head h reading KV head h / (Hq / H_kv).  Binary64 throughout.
 * Readings for bad input: a sequence whose last position needs a table entry
 * past max_blocks, or with start_b < 0, gives zero rows and is counted; a used
 * block id outside [0, num_blocks) drops that block's tokens and is counted
 * once per (sequence, block). */
int64_t orc_paged_attention_prefill(double *out, const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int32_t max_blocks, const int32_t *starts,
                                    const int32_t *cu_q, int32_t num_seqs, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t bs, int32_t num_blocks,
                                    double scale, int dtype)
{
    int64_t errors = 0;
    int32_t group = num_q_heads / num_kv_heads;
    build_f16_table();
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t n = (int64_t)cu_q[b + 1] - cu_q[b];
        int64_t start = starts[b];
        int64_t total = start + n;
        const int32_t *row = block_tables + (int64_t)b * max_blocks;
        int bad = n < 0 || start < 0 || (total + bs - 1) / bs > max_blocks;
        if (bad) ++errors;
        if (!bad) {
            for (int64_t j = 0; j < (total + bs - 1) / bs; ++j)
                if (row[j] < 0 || row[j] >= num_blocks) ++errors;
        }
        double *scores = (double *)malloc(sizeof(double) * (size_t)(total > 0 ? total : 1));
        for (int64_t i = 0; i < (n > 0 ? n : 0); ++i) {
            int64_t p = start + i;
            for (int32_t h = 0; h < num_q_heads; ++h) {
                int32_t g = h / group;
                double *o = out + (((int64_t)cu_q[b] + i) * num_q_heads + h) * head_dim;
                int64_t q_base = (((int64_t)cu_q[b] + i) * num_q_heads + h) * head_dim;
                double m = -INFINITY, l = 0.0;
                for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
                if (bad) continue;
                for (int64_t t = 0; t <= p; ++t) {
                    int32_t phys = row[t / bs];
                    scores[t] = -INFINITY;
                    if (phys < 0 || phys >= num_blocks) continue;
                    int64_t k_base = (((int64_t)phys * bs + t % bs) * num_kv_heads + g) * head_dim;
                    double s = 0.0;
                    for (int32_t d = 0; d < head_dim; ++d)
                        s += load_elem(q, q_base + d, dtype) * load_elem(k_cache, k_base + d, dtype);
                    scores[t] = scale * s;
                    if (scores[t] > m) m = scores[t];
                }
                if (m == -INFINITY) continue;
                for (int64_t t = 0; t <= p; ++t) {
                    if (scores[t] == -INFINITY) continue;
                    scores[t] = exp(scores[t] - m);
                    l += scores[t];
                }
                for (int64_t t = 0; t <= p; ++t) {
                    if (scores[t] == -INFINITY) continue;
                    int32_t phys = row[t / bs];
                    int64_t v_base = (((int64_t)phys * bs + t % bs) * num_kv_heads + g) * head_dim;
                    double w = scores[t] / l;
                    for (int32_t d = 0; d < head_dim; ++d) o[d] += w * load_elem(v_cache, v_base + d, dtype);
                }
            }
        }
        free(scores);
    }
    return errors;
}
