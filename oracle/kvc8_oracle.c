/*
 * kvc8_oracle.c -- plain, slow, single-threaded CPU oracle for the int8 ("C8")
 * paged KV-cache store and dequant-gather.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * with the CUDA library; the two meet only through the seeded inputs that
 * the tests hand to both.
 *
 * Sources (web pages; cited by title and section):
 *   [PR379]  mojo_opset pull request #379, "feat: [MLU] add mlu experimental
 *            ops; fix post norm bug" -- the Gemini Code Assist review and the
 *            four automated github-actions review passes that describe the
 *            torch-native MojoStorePagedKVCacheC8 / MojoDequantFromPagedKVCache.
 *   [README] "Mojo Opset" README, section "Backend Implementations / Torch
 *            native" (the torch-native code is the golden reference).
 *
 * Precision: the pages fix fp32 (the fourth review pass, "Must fix", asks
 * that the store divide in fp32 rather than in the input dtype, and every pass
 * notes that the dequant helper means to upcast the scale to fp32), so every
 * floating-point step below is one IEEE binary32 operation, rounded to nearest
 * even.  Build with -O2 -ffp-contract=off and without -ffast-math so that the
 * compiler neither fuses nor reorders them.
 *
 * Definition (one row = one token of one kv head, head_dim values):
 *   store   x_d   = float(bf16 input)                         (exact widening)
 *           s     = max_d |x_d| / 127          (quant_mode 0, dynamic, per row)
 *           s_d   = static_scale[h][d]         (quant_mode 1, static, per channel)
 *           s     = block_scale[blk][h]        (quant_mode 2, static, per block)
 *           q_d   = clamp(round_half_even(x_d / s), -127, 127), q_d = 0 if s == 0
 *           pos   = context_kv_lens[b] + i     (i-th new token of sequence b)
 *           cache[block_table[b][pos / bs]][h][pos % bs][d] = q_d
 *           scale_cache[same block][h][pos % bs] = s          (quant_mode 0 only)
 *   gather  out[off_b + p][h][d] = bf16_rne(float(q) * s)   for p < context_lengths[b]
 *           off_b = exclusive prefix sum of context_lengths, unless given.
 *
 * Every reading of a point the pages leave open is marked READING below.
 *
 * Function-level parity pins live in the -m "not gpu" tests: hand-worked
 * goldens, exact rational re-derivations, invariants and a brute-force
 * placement model.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_BOUNDS 4

/* ---- bf16 <-> fp32, bit level --------------------------------------------
 * bf16 is the top half of an IEEE binary32 word, so widening is a shift.
 * Narrowing rounds to nearest, ties to even, on the 16 dropped bits: add
 * 0x7FFF plus the lowest kept bit, then truncate.  NaN inputs are outside the
 * contract; they map to the canonical quiet NaN. */
static float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t orc_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)0x7FC0u;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ---- one quantised code ---------------------------------------------------
 * [PR379] review passes 2 and 4 (Notes, "[CHECK]") describe the torch golden
 * as symmetric int8: divide, torch.round, clamp.  torch.round rounds half to
 * even, which is C's nearbyintf under the default FE_TONEAREST mode.
 * READING: the clamp is [-127, 127] (symmetric), as the pass-3 note says some
 * NPU/MLU kernels do, not the torch golden's [-128, 127]; the two agree
 * except when a static scale saturates a negative value.
 * READING: a zero scale (an all-zero row in quant_mode 0) gives code 0 rather
 * than 0/0. */
static int8_t orc_quantize_one(float x, float s)
{
    if (s == 0.0f)
        return 0;
    float r = nearbyintf(x / s); /* one IEEE fp32 division, then half-even */
    if (r > 127.0f)
        r = 127.0f;
    if (r < -127.0f)
        r = -127.0f;
    return (int8_t)r;
}

/* ---- one dequantised value ------------------------------------------------
 * [PR379] every review pass, "Must fix" on dequant_from_cache: the helper is
 * meant to multiply the int8 data, as float, by the fp32 scale and cast the
 * product to the output dtype.  READING: one fp32 multiply (a single rounding)
 * followed by round-to-nearest-even to bf16. */
static uint16_t orc_dequantize_one(int8_t q, float s)
{
    float prod = (float)q * s;
    return orc_f32_to_bf16_rne(prod);
}

/* quant_mode 0: s = max|x| / 127 over one row of head_dim values. */
static float orc_row_scale(const uint16_t *row, int head_dim)
{
    float amax = 0.0f;
    for (int d = 0; d < head_dim; ++d) {
        float a = fabsf(orc_bf16_to_f32(row[d]));
        if (a > amax)
            amax = a;
    }
    return amax / 127.0f;
}

/* Physical (block, slot) of logical position pos of sequence b.
 * [PR379] passes 1 and 3 (Suggestions) describe the store as writing each
 * chunk into key_cache[block, :, offset:offset+len, :] with block taken from
 * the block table; the read side gathers key_cache[block_tables[b, j]] for the
 * sequence's logical blocks j.  Position pos lives in logical block pos / bs
 * at in-block slot pos % bs. */
static int orc_slot(const int32_t *block_table, int max_blocks_per_seq,
                    int block_size, int num_blocks, int b, int64_t pos,
                    int32_t *blk, int32_t *slot)
{
    int64_t lb = pos / block_size;
    if (pos < 0 || lb >= max_blocks_per_seq)
        return ORC_ERR_BOUNDS;
    int32_t pb = block_table[(int64_t)b * max_blocks_per_seq + lb];
    if (pb < 0 || pb >= num_blocks)
        return ORC_ERR_BOUNDS;
    *blk = pb;
    *slot = (int32_t)(pos % block_size);
    return ORC_OK;
}

/* Quantise n rows of one kv-head set.  x: [n][H][D] bf16 bits, dense.
 * quant_mode 0: s_out[n][H] receives the per-row scale.
 * quant_mode 1: static_scale is [H][D]; s_out is not written.
 * quant_mode 2: static_scale is [n][H], the scale of each row (in the cache,
 *               the scale of the row's block); s_out is not written. */
int orc_quantize_rows(int quant_mode, int64_t n, int kv_heads, int head_dim,
                      const uint16_t *x, const float *static_scale,
                      int8_t *q_out, float *s_out)
{
    if (quant_mode < 0 || quant_mode > 2)
        return ORC_ERR_ARG;
    for (int64_t t = 0; t < n; ++t) {
        for (int h = 0; h < kv_heads; ++h) {
            const uint16_t *row = x + (t * kv_heads + h) * head_dim;
            int8_t *qrow = q_out + (t * kv_heads + h) * head_dim;
            if (quant_mode == 0) {
                float s = orc_row_scale(row, head_dim);
                s_out[t * kv_heads + h] = s;
                for (int d = 0; d < head_dim; ++d)
                    qrow[d] = orc_quantize_one(orc_bf16_to_f32(row[d]), s);
            } else if (quant_mode == 1) {
                for (int d = 0; d < head_dim; ++d)
                    qrow[d] = orc_quantize_one(orc_bf16_to_f32(row[d]),
                                               static_scale[h * head_dim + d]);
            } else {
                float s = static_scale[t * kv_heads + h];
                for (int d = 0; d < head_dim; ++d)
                    qrow[d] = orc_quantize_one(orc_bf16_to_f32(row[d]), s);
            }
        }
    }
    return ORC_OK;
}

/* The store: MojoStorePagedKVCacheC8 as the [PR379] reviews describe it.
 *   k_states, v_states : bf16 bits [num_tokens][H][D], dense
 *   k_cache, v_cache   : int8 [num_blocks][H][block_size][D]
 *   k_scale, v_scale   : quant_mode 0 -> fp32 [num_blocks][H][block_size], written
 *                        quant_mode 1 -> fp32 [H][D], read
 *                        quant_mode 2 -> fp32 [num_blocks][H], read
 *                        (READING: [PR379] pass 1, "Must fix", and its
 *                        "[CHECK]" note name per-block scales for
 *                        quant_mode != 0 without a formula; here one static
 *                        scale per physical block and kv head, owned by the
 *                        caller like the per-channel table)
 *   block_table        : int32 [num_seqs][max_blocks_per_seq]
 *   cu_q_lens          : int32 [num_seqs + 1] prefix of new-token counts, or
 *                        NULL for pure decode (READING: one new token per
 *                        sequence, token b belongs to sequence b; pass 2
 *                        says cu_q_lens may be None in decode)
 *   context_kv_lens    : int32 [num_seqs], tokens already cached per sequence
 *                        (READING: the new tokens go to [ctx, ctx + q))
 * Returns ORC_ERR_BOUNDS (and stops) if a position leaves the block table or
 * a block id leaves the pool.  Sequences are processed in order; the loop
 * over new tokens replaces the pages' per-chunk loop, with the same placement. */
int orc_store(int quant_mode, int num_seqs, int64_t num_tokens, int kv_heads,
              int head_dim, int block_size, int num_blocks,
              int max_blocks_per_seq, const uint16_t *k_states,
              const uint16_t *v_states, int8_t *k_cache, int8_t *v_cache,
              float *k_scale, float *v_scale, const int32_t *block_table,
              const int32_t *cu_q_lens, const int32_t *context_kv_lens)
{
    if (quant_mode < 0 || quant_mode > 2)
        return ORC_ERR_ARG;
    const int64_t row_elems = (int64_t)kv_heads * head_dim;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t first = cu_q_lens ? cu_q_lens[b] : b;
        int64_t count = cu_q_lens ? (int64_t)cu_q_lens[b + 1] - cu_q_lens[b] : 1;
        if (count < 0 || first < 0 || first + count > num_tokens)
            return ORC_ERR_BOUNDS;
        for (int64_t i = 0; i < count; ++i) {
            int64_t tok = first + i;
            int64_t pos = (int64_t)context_kv_lens[b] + i;
            int32_t blk, slot;
            int rc = orc_slot(block_table, max_blocks_per_seq, block_size,
                              num_blocks, b, pos, &blk, &slot);
            if (rc != ORC_OK)
                return rc;
            for (int kv = 0; kv < 2; ++kv) {
                const uint16_t *xs = kv ? v_states : k_states;
                int8_t *cache = kv ? v_cache : k_cache;
                float *scale = kv ? v_scale : k_scale;
                for (int h = 0; h < kv_heads; ++h) {
                    const uint16_t *row = xs + tok * row_elems + (int64_t)h * head_dim;
                    int64_t dst_row = ((int64_t)blk * kv_heads + h) * block_size + slot;
                    int8_t *dst = cache + dst_row * head_dim;
                    if (quant_mode == 0) {
                        float s = orc_row_scale(row, head_dim);
                        scale[dst_row] = s;
                        for (int d = 0; d < head_dim; ++d)
                            dst[d] = orc_quantize_one(orc_bf16_to_f32(row[d]), s);
                    } else if (quant_mode == 1) {
                        for (int d = 0; d < head_dim; ++d)
                            dst[d] = orc_quantize_one(orc_bf16_to_f32(row[d]),
                                                      scale[h * head_dim + d]);
                    } else {
                        float s = scale[(int64_t)blk * kv_heads + h];
                        for (int d = 0; d < head_dim; ++d)
                            dst[d] = orc_quantize_one(orc_bf16_to_f32(row[d]), s);
                    }
                }
            }
        }
    }
    return ORC_OK;
}

/* Exclusive prefix sum of context_lengths: the default context_seq_offset.
 * [PR379] passes 1 and 3 ("Must fix" on context_seq_offset) describe it as a
 * cumsum shifted by one with entry 0 equal to zero. */
void orc_exclusive_cumsum(int num_seqs, const int32_t *lens, int64_t *out)
{
    int64_t acc = 0;
    for (int b = 0; b < num_seqs; ++b) {
        out[b] = acc;
        acc += lens[b];
    }
}

/* The dequant-gather: MojoDequantFromPagedKVCache as the [PR379] reviews
 * describe it.  For each sequence b and each position p < context_lengths[b]
 * the row set [H][D] of logical position p is dequantised into
 *   out[(off_b + p) * tok_stride + h * head_stride + d]      (bf16 bits)
 * with off_b = context_seq_offset[b], or the exclusive prefix sum of
 * context_lengths when that pointer is NULL.  Caller-given offsets may leave
 * padding rows between sequences (the pages' tests use padded offsets); rows
 * that no sequence covers are not touched.  out_rows bounds the row index. */
int orc_dequant_gather(int quant_mode, int num_seqs, int kv_heads,
                       int head_dim, int block_size, int num_blocks,
                       int max_blocks_per_seq, const int8_t *k_cache,
                       const int8_t *v_cache, const float *k_scale,
                       const float *v_scale, const int32_t *block_table,
                       const int32_t *context_lengths,
                       const int64_t *context_seq_offset, uint16_t *k_out,
                       uint16_t *v_out, int64_t out_rows, int64_t tok_stride,
                       int64_t head_stride)
{
    if (quant_mode < 0 || quant_mode > 2)
        return ORC_ERR_ARG;
    int64_t acc = 0;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t off = context_seq_offset ? context_seq_offset[b] : acc;
        acc += context_lengths[b];
        for (int64_t p = 0; p < context_lengths[b]; ++p) {
            int32_t blk, slot;
            int rc = orc_slot(block_table, max_blocks_per_seq, block_size,
                              num_blocks, b, p, &blk, &slot);
            if (rc != ORC_OK)
                return rc;
            if (off + p < 0 || off + p >= out_rows)
                return ORC_ERR_BOUNDS;
            for (int kv = 0; kv < 2; ++kv) {
                const int8_t *cache = kv ? v_cache : k_cache;
                const float *scale = kv ? v_scale : k_scale;
                uint16_t *out = kv ? v_out : k_out;
                for (int h = 0; h < kv_heads; ++h) {
                    int64_t src_row = ((int64_t)blk * kv_heads + h) * block_size + slot;
                    const int8_t *src = cache + src_row * head_dim;
                    uint16_t *dst = out + (off + p) * tok_stride + (int64_t)h * head_stride;
                    for (int d = 0; d < head_dim; ++d) {
                        float s = quant_mode == 0   ? scale[src_row]
                                  : quant_mode == 1 ? scale[h * head_dim + d]
                                                    : scale[(int64_t)blk * kv_heads + h];
                        dst[d] = orc_dequantize_one(src[d], s);
                    }
                }
            }
        }
    }
    return ORC_OK;
}

/* Element-level entry points, so that tests can pin each step on its own. */
int8_t orc_quantize_value(uint16_t x_bf16, float s)
{
    return orc_quantize_one(orc_bf16_to_f32(x_bf16), s);
}

uint16_t orc_dequantize_value(int8_t q, float s)
{
    return orc_dequantize_one(q, s);
}

uint16_t orc_round_to_bf16(float f) { return orc_f32_to_bf16_rne(f); }

float orc_row_scale_bf16(const uint16_t *row, int head_dim)
{
    return orc_row_scale(row, head_dim);
}

/* ---- bf16 paged cache without quantisation ---------------------------------
 * MojoStorePagedKVCache, the int8 store's sibling ("Mojo Opset" README, "Op
 * List"; [PR379] pass 1, "Must fix", on the cu_q_lens check it performs): the
 * same placement as orc_store, with each row copied as is.  Caches are bf16
 * bits [num_blocks][H][block_size][D]. */
int orc_store_bf16(int num_seqs, int64_t num_tokens, int kv_heads, int head_dim,
                   int block_size, int num_blocks, int max_blocks_per_seq,
                   const uint16_t *k_states, const uint16_t *v_states,
                   uint16_t *k_cache, uint16_t *v_cache,
                   const int32_t *block_table, const int32_t *cu_q_lens,
                   const int32_t *context_kv_lens)
{
    const int64_t row_elems = (int64_t)kv_heads * head_dim;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t first = cu_q_lens ? cu_q_lens[b] : b;
        int64_t count = cu_q_lens ? (int64_t)cu_q_lens[b + 1] - cu_q_lens[b] : 1;
        if (count < 0 || first < 0 || first + count > num_tokens)
            return ORC_ERR_BOUNDS;
        for (int64_t i = 0; i < count; ++i) {
            int32_t blk, slot;
            int rc = orc_slot(block_table, max_blocks_per_seq, block_size,
                              num_blocks, b, (int64_t)context_kv_lens[b] + i,
                              &blk, &slot);
            if (rc != ORC_OK)
                return rc;
            for (int kv = 0; kv < 2; ++kv) {
                const uint16_t *xs = kv ? v_states : k_states;
                uint16_t *cache = kv ? v_cache : k_cache;
                for (int h = 0; h < kv_heads; ++h) {
                    const uint16_t *src = xs + (first + i) * row_elems + (int64_t)h * head_dim;
                    uint16_t *dst = cache + (((int64_t)blk * kv_heads + h) * block_size + slot) * head_dim;
                    for (int d = 0; d < head_dim; ++d)
                        dst[d] = src[d];
                }
            }
        }
    }
    return ORC_OK;
}

/* Gather of the bf16 cache: the layout and offsets of orc_dequant_gather,
 * values copied as is. */
int orc_gather_bf16(int num_seqs, int kv_heads, int head_dim, int block_size,
                    int num_blocks, int max_blocks_per_seq, const uint16_t *k_cache,
                    const uint16_t *v_cache, const int32_t *block_table,
                    const int32_t *context_lengths, const int64_t *context_seq_offset,
                    uint16_t *k_out, uint16_t *v_out, int64_t out_rows,
                    int64_t tok_stride, int64_t head_stride)
{
    int64_t acc = 0;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t off = context_seq_offset ? context_seq_offset[b] : acc;
        acc += context_lengths[b];
        for (int64_t p = 0; p < context_lengths[b]; ++p) {
            int32_t blk, slot;
            int rc = orc_slot(block_table, max_blocks_per_seq, block_size,
                              num_blocks, b, p, &blk, &slot);
            if (rc != ORC_OK)
                return rc;
            if (off + p < 0 || off + p >= out_rows)
                return ORC_ERR_BOUNDS;
            for (int kv = 0; kv < 2; ++kv) {
                const uint16_t *cache = kv ? v_cache : k_cache;
                uint16_t *out = kv ? v_out : k_out;
                for (int h = 0; h < kv_heads; ++h) {
                    const uint16_t *src = cache + (((int64_t)blk * kv_heads + h) * block_size + slot) * head_dim;
                    uint16_t *dst = out + (off + p) * tok_stride + (int64_t)h * head_stride;
                    for (int d = 0; d < head_dim; ++d)
                        dst[d] = src[d];
                }
            }
        }
    }
    return ORC_OK;
}

/* ---- paged decode attention over the int8 cache ---------------------------
 * MojoPagedDecodeGQA of the "Mojo Opset" README ("Op List", Attention): one
 * decode query per sequence attends over the paged cache.  The pages give no
 * formula; READING: the standard grouped-query scaled dot-product attention,
 * over the values the dequant-gather produces, i.e. the bf16 rows
 * bf16_rne(float(q) * s) of the cache, so that the fused op equals the
 * dequant-gather followed by attention:
 *   kv head of query head j     h = j / group       (group = Hq / H)
 *   score_p = softmax_scale * sum_d query[b][j][d] * K'[b][p][h][d]
 *   w_p     = exp(score_p - max_p score_p) / sum_p exp(score_p - max)
 *   out[b][j][d] = sum_p w_p * V'[b][p][h][d]        (p < context_lengths[b])
 * computed in fp64 and returned unrounded; an empty context gives 0.
 *   query : bf16 bits [num_seqs][Hq][D], dense;  out : fp64 [num_seqs][Hq][D]. */
int orc_paged_decode_attention(int quant_mode, int num_seqs, int kv_heads, int group,
                               int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_seq, const uint16_t *query,
                               const int8_t *k_cache, const int8_t *v_cache,
                               const float *k_scale, const float *v_scale,
                               const int32_t *block_table, const int32_t *context_lengths,
                               double softmax_scale, double *out)
{
    if (quant_mode < 0 || quant_mode > 2 || group < 1)
        return ORC_ERR_ARG;
    const int hq = kv_heads * group;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t len = context_lengths[b];
        for (int j = 0; j < hq; ++j) {
            int h = j / group;
            const uint16_t *qv = query + ((int64_t)b * hq + j) * head_dim;
            double *o = out + ((int64_t)b * hq + j) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (len <= 0)
                continue;
            /* pass 1: the largest score */
            double mx = -HUGE_VAL;
            for (int64_t p = 0; p < len; ++p) {
                int32_t blk, slot;
                int rc = orc_slot(block_table, max_blocks_per_seq, block_size,
                                  num_blocks, b, p, &blk, &slot);
                if (rc != ORC_OK)
                    return rc;
                int64_t row = ((int64_t)blk * kv_heads + h) * block_size + slot;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) {
                    float s = quant_mode == 0   ? k_scale[row]
                              : quant_mode == 1 ? k_scale[h * head_dim + d]
                                                : k_scale[(int64_t)blk * kv_heads + h];
                    double kd = orc_bf16_to_f32(orc_dequantize_one(k_cache[row * head_dim + d], s));
                    dot += (double)orc_bf16_to_f32(qv[d]) * kd;
                }
                double sc = softmax_scale * dot;
                if (sc > mx)
                    mx = sc;
            }
            /* pass 2: weights and the weighted sum of V' rows */
            double total = 0.0;
            for (int64_t p = 0; p < len; ++p) {
                int32_t blk, slot;
                if (orc_slot(block_table, max_blocks_per_seq, block_size, num_blocks, b, p,
                             &blk, &slot) != ORC_OK)
                    return ORC_ERR_BOUNDS;
                int64_t row = ((int64_t)blk * kv_heads + h) * block_size + slot;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) {
                    float s = quant_mode == 0   ? k_scale[row]
                              : quant_mode == 1 ? k_scale[h * head_dim + d]
                                                : k_scale[(int64_t)blk * kv_heads + h];
                    double kd = orc_bf16_to_f32(orc_dequantize_one(k_cache[row * head_dim + d], s));
                    dot += (double)orc_bf16_to_f32(qv[d]) * kd;
                }
                double w = exp(softmax_scale * dot - mx);
                total += w;
                for (int d = 0; d < head_dim; ++d) {
                    float s = quant_mode == 0   ? v_scale[row]
                              : quant_mode == 1 ? v_scale[h * head_dim + d]
                                                : v_scale[(int64_t)blk * kv_heads + h];
                    o[d] += w * orc_bf16_to_f32(orc_dequantize_one(v_cache[row * head_dim + d], s));
                }
            }
            for (int d = 0; d < head_dim; ++d)
                o[d] /= total;
        }
    }
    return ORC_OK;
}
