/*
 * kvc8.h -- C ABI of libkvc8: the int8 ("C8") paged KV-cache store and
 * dequant-gather on NVIDIA GB300 (sm_103a).
 *
 * Source of the operations (web pages, cited by title and section):
 *   [PR379]  mojo_opset pull request #379, "feat: [MLU] add mlu experimental
 *            ops; fix post norm bug": the Gemini Code Assist review and the
 *            four github-actions review passes, which describe the
 *            torch-native MojoStorePagedKVCacheC8 and
 *            MojoDequantFromPagedKVCache operators, their dequant_from_cache
 *            helper, build_paged_kv_chunk_metadata and the context_seq_offset
 *            default.
 *   [README] "Mojo Opset" README, "Op List" (MojoStorePagedKVCache, the bf16
 *            sibling) and "Backend Implementations / Torch native".
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory on the CUDA device that is current
 *     on the calling thread, unless the argument says "host".  The caller owns
 *     all memory; the library allocates nothing and never synchronises the
 *     stream (except kvc8_get_error, which exists to do so).
 *   - Work is enqueued on `stream` and runs asynchronously.  Arguments that
 *     can be checked on the host are checked before anything is enqueued; a
 *     failed check returns KVC8_ERR_INVALID_ARG or KVC8_ERR_UNSUPPORTED and
 *     enqueues nothing.
 *   - Data-dependent errors (a block id outside the pool, a position beyond the
 *     block table, an output row beyond out_rows, a negative length) can only be
 *     seen on the device.  The kernels skip the offending row and record the
 *     first such error in the optional device word `dev_error` (one int32_t,
 *     0 = no error; the caller zeroes it).  They never trap.  Read it with
 *     kvc8_get_error.
 *   - Launch failures return KVC8_ERR_CUDA.
 *
 * Layouts (row-major, innermost last).  H = kv_heads, D = head_dim,
 * bs = block_size, NB = num_blocks, B = num_seqs, MB = max_blocks_per_seq:
 *   key_cache, value_cache   int8  [NB][H][bs][D]
 *   scale cache (mode 0)     fp32  [NB][H][bs]     one scale per cached row
 *   static scale (mode 1)    fp32  [H][D]          one scale per (head, channel)
 *   block_table              int32 [B][MB]         physical block of each logical block
 *   bf16 K/V tokens          [tokens][H][D] with element strides (tok_stride,
 *                            head_stride, 1); both strides multiples of 8 and
 *                            the base 16-byte aligned.
 * The per-block layout [H][bs][D] follows from the review passes of [PR379]:
 * the store writes key_cache[block, :, offset:offset+len, :] after permuting
 * the new tokens to [heads, len, dim], the dequant helper broadcasts the scale
 * with a token axis inserted before the channel axis, and the gather
 * transposes [heads, tokens, dim] to [tokens, heads, dim].
 *
 * Arithmetic (bit-exact, no fast-math):
 *   quantise     q = clamp(round_half_even(x / s), -127, 127), one IEEE fp32
 *                division (q = 0 when s == 0)
 *   mode 0 scale s = max_d |x_d| / 127 in fp32, per (token, kv head)
 *   dequantise   out = bf16_round_nearest_even(fp32(q) * s), one fp32 multiply
 */
#ifndef KVC8_H
#define KVC8_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvc8_status {
    KVC8_OK = 0,
    KVC8_ERR_INVALID_ARG = 1,   /* null pointer, bad size, stride or alignment */
    KVC8_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle */
    KVC8_ERR_CUDA = 3,          /* a CUDA call or launch failed */
    KVC8_ERR_DEVICE_BOUNDS = 4, /* kvc8_get_error: the device word is set */
    KVC8_ERR_WORKSPACE = 5      /* workspace missing, too small or misaligned */
} kvc8_status;

/* Codes the kernels write into the device error word (first error wins). */
enum {
    KVC8_DEV_OK = 0,
    KVC8_DEV_BAD_BLOCK_ID = 1,     /* block_table entry outside [0, num_blocks) */
    KVC8_DEV_POS_BEYOND_TABLE = 2, /* position >= max_blocks_per_seq * block_size */
    KVC8_DEV_OUT_ROW_RANGE = 3,    /* gather output row outside [0, out_rows) */
    KVC8_DEV_BAD_LENGTH = 4        /* negative length or decreasing cu_q_lens */
};

/* Geometry of one paged cache and one batch.  quant_mode: 0 = dynamic scale
 * per (token, kv head), kept in a scale cache beside the codes; 1 = static
 * scale per (kv head, channel), passed in; 2 = static scale per (physical
 * block, kv head), passed in.  [PR379] (every pass: the store is a symmetric
 * int8 quantisation against a passed-in per-channel scale; the docstring says
 * per_channal) describes the per-channel form; the dynamic form stores its
 * per-row scales where the pass-1 "Must fix" expects per-block scale shapes,
 * and mode 2 is the plain per-block reading of that same passage and of the
 * pass-1 "[CHECK]" note (quant_mode != 0 is per-block), one caller-owned
 * scale for every row of a block. */
typedef struct kvc8_geom {
    int32_t num_seqs;           /* B >= 0 */
    int32_t kv_heads;           /* H >= 1 */
    int32_t head_dim;           /* D: multiple of 16, 16..256 */
    int32_t block_size;         /* bs >= 1 */
    int32_t num_blocks;         /* NB >= 1 */
    int32_t max_blocks_per_seq; /* MB >= 1 */
    int32_t quant_mode;         /* 0, 1 or 2 */
} kvc8_geom;

/* Human-readable name of a status code (static string). */
const char *kvc8_status_str(kvc8_status status);

/* Library version as major * 10000 + minor * 100 + patch. */
int32_t kvc8_version(void);

/*
 * kvc8_store -- quantise new bf16 K and V tokens to int8 and scatter them into
 * the paged cache: MojoStorePagedKVCacheC8 of [PR379].
 *
 * For sequence b (0 <= b < B) the new tokens are rows [cu_q_lens[b],
 * cu_q_lens[b+1]) of key_states / value_states.  The i-th of them goes to
 * logical position pos = context_kv_lens[b] + i, i.e. physical block
 * block_table[b][pos / bs], slot pos % bs, for every kv head: the codes to
 * cache[block][h][slot][0:D], and in mode 0 the row's scale to
 * scale_cache[block][h][slot].  This replaces the pages' per-chunk host loop
 * over build_paged_kv_chunk_metadata (pass-1 and pass-3 "Suggestions" on the
 * Python loop and .tolist()) with per-token slot arithmetic on the device:
 * one launch, no host synchronisation.
 *
 *   g              geometry (host pointer)
 *   num_tokens     rows of key_states/value_states (0 <= N < 2^31); 0 is a no-op
 *   key_states,
 *   value_states   bf16 [N][H][D], strides (x_tok_stride, x_head_stride, 1)
 *                  in elements
 *   key_cache,
 *   value_cache    int8 [NB][H][bs][D], written in place
 *   key_scale,
 *   value_scale    mode 0: fp32 [NB][H][bs] scale caches, written in place;
 *                  mode 1: fp32 [H][D] static scales, read only;
 *                  mode 2: fp32 [NB][H] block scales, read only
 *   block_table    int32 [B][MB]
 *   cu_q_lens      int32 [B+1], cu_q_lens[0] = 0, non-decreasing, last = N;
 *                  or NULL for pure decode: one new token per sequence, token
 *                  b belongs to sequence b, and N must equal B (pass 2, "Must
 *                  fix": cu_q_lens may be None in decode)
 *   context_kv_lens int32 [B], tokens already cached per sequence
 *   dev_error      optional int32 device word (see conventions), or NULL
 *
 * Tokens whose position leaves the block table or whose block id leaves the
 * pool are skipped and reported through dev_error.  Sequences must not share
 * physical blocks for the slots this call writes.
 */
kvc8_status kvc8_store(const kvc8_geom *g, int64_t num_tokens,
                       const void *key_states, const void *value_states,
                       int64_t x_tok_stride, int64_t x_head_stride,
                       int8_t *key_cache, int8_t *value_cache,
                       float *key_scale, float *value_scale,
                       const int32_t *block_table, const int32_t *cu_q_lens,
                       const int32_t *context_kv_lens, int32_t *dev_error,
                       cudaStream_t stream);

/* Bytes of device workspace that kvc8_build_metadata, kvc8_dequant_gather
 * and kvc8_append_gather need for this geometry (depends on num_seqs only;
 * the gathers use the first part, the plan).  Host function. */
size_t kvc8_gather_workspace_bytes(const kvc8_geom *g);

/*
 * kvc8_build_metadata -- the gather plan: per-sequence output offsets and the
 * prefix of logical blocks per sequence, written into `workspace`.
 *
 * The output offsets are context_seq_offset when given, else the exclusive
 * prefix sum of context_lengths: pass 1 and pass 3 ("Must fix" on
 * context_seq_offset) describe the default as a cumsum shifted right by one
 * with entry 0 = 0.  Computed on the device; no .item() and no host sync
 * (pass-3 "Suggestions" on per-iteration .item()).
 *
 *   context_lengths     int32 [B], tokens to gather per sequence (>= 0)
 *   context_seq_offset  int64 [B] caller-given first output row per sequence
 *                       (padding between sequences allowed), or NULL
 *   offsets_out         optional int64 [B]: receives the offsets used
 *   workspace           >= kvc8_gather_workspace_bytes(g) bytes, 256-byte
 *                       aligned; the plan stays valid while context_lengths,
 *                       context_seq_offset and geometry are unchanged
 */
kvc8_status kvc8_build_metadata(const kvc8_geom *g, const int32_t *context_lengths,
                                const int64_t *context_seq_offset,
                                int64_t *offsets_out, void *workspace,
                                size_t workspace_bytes, int32_t *dev_error,
                                cudaStream_t stream);

/*
 * kvc8_dequant_gather -- gather every sequence's pages and dequantise them into
 * contiguous bf16 rows: MojoDequantFromPagedKVCache of [PR379].
 *
 * For each b and p < context_lengths[b], for every kv head h and channel d:
 *   out[(off_b + p) * out_tok_stride + h * out_head_stride + d]
 *       = bf16(fp32(cache[blk][h][slot][d]) * s)
 * with blk = block_table[b][p / bs], slot = p % bs, s = scale_cache[blk][h][slot]
 * (mode 0), static_scale[h][d] (mode 1) or block_scale[blk][h] (mode 2), and
 * off_b as in
 * kvc8_build_metadata.  This is the pages' per-sequence loop (list-comprehension
 * concat of the sequence's blocks, dequant_from_cache, slice to the context,
 * transpose to [tokens, heads, dim], in-place write at the offset) as one
 * pass with no host synchronisation.  Rows not covered by any sequence are not
 * written.  The output may be strided (the pages' tests pass a transposed
 * view); out_tok_stride and out_head_stride are in elements, multiples of 8,
 * and key_out / value_out are 16-byte aligned.
 *
 * Enqueues the plan (kvc8_build_metadata into `workspace`) and the gather; the
 * gather launch overlaps the plan's tail (programmatic dependent launch).
 *
 *   key_cache, value_cache   int8 [NB][H][bs][D]
 *   key_scale, value_scale   mode 0: fp32 [NB][H][bs]; mode 1: fp32 [H][D];
 *                            mode 2: fp32 [NB][H]
 *   block_table              int32 [B][MB]
 *   context_lengths          int32 [B]
 *   context_seq_offset       int64 [B] or NULL (exclusive prefix sum)
 *   key_out, value_out       bf16, rows [0, out_rows)
 *   workspace                as in kvc8_build_metadata; also holds the gather's
 *                            work counter, so calls that overlap on the GPU need
 *                            separate workspaces
 */
kvc8_status kvc8_dequant_gather(const kvc8_geom *g, const int8_t *key_cache,
                                const int8_t *value_cache, const float *key_scale,
                                const float *value_scale, const int32_t *block_table,
                                const int32_t *context_lengths,
                                const int64_t *context_seq_offset, void *key_out,
                                void *value_out, int64_t out_rows,
                                int64_t out_tok_stride, int64_t out_head_stride,
                                void *workspace, size_t workspace_bytes,
                                int32_t *dev_error, cudaStream_t stream);

/*
 * kvc8_dequant_gather_planned -- kvc8_dequant_gather with a plan that an earlier
 * kvc8_build_metadata wrote into `workspace` for the same context lengths,
 * offsets and geometry (e.g. reused across the layers of one model step).
 * One launch (after an 8-byte memset of the plan's work counter: the gather
 * hands out its work through an atomic counter kept in the workspace, so two
 * gathers that overlap on the GPU must not share a workspace).  Arguments as
 * in kvc8_dequant_gather.
 */
kvc8_status kvc8_dequant_gather_planned(const kvc8_geom *g, const int8_t *key_cache,
                                        const int8_t *value_cache,
                                        const float *key_scale, const float *value_scale,
                                        const int32_t *block_table,
                                        const int32_t *context_lengths, void *key_out,
                                        void *value_out, int64_t out_rows,
                                        int64_t out_tok_stride, int64_t out_head_stride,
                                        void *workspace, size_t workspace_bytes,
                                        int32_t *dev_error, cudaStream_t stream);

/*
 * kvc8_append_gather -- kvc8_store followed by kvc8_dequant_gather of every
 * sequence's whole context (cached + new tokens), in one pass over the data.
 * The pages run these as two ops on the decode path (MojoStorePagedKVCacheC8
 * with cu_q_lens NULL "in decode", [PR379] pass 2 "Must fix"; then
 * MojoDequantFromPagedKVCache, every pass "Must fix").  The result is
 * bit-identical to the two calls with context_lengths[b] = context_kv_lens[b]
 * + q_b (q_b = cu_q_lens[b+1] - cu_q_lens[b], or 1 when cu_q_lens is NULL):
 * the same codes and scales land in the cache and the same bf16 rows in the
 * output.  The new tokens' rows are quantised once; their codes and scales go
 * to the cache and their dequantised values straight to output rows
 * offset_b + context_kv_lens[b] + i, while the same launch gathers the cached
 * positions [0, context_kv_lens[b]) from the cache.  Enqueues a plan (into
 * `workspace`) and one fused launch that overlaps the plan's tail.  A long
 * append (more than 16 384 new K and V rows, i.e. a prompt rather than a
 * decode step) runs instead as the store kernel, a plan over the cached and
 * the new positions and the gather, which is faster there; that path keeps
 * per-sequence lengths in the workspace after the plan, so it is taken only
 * when workspace_bytes >= kvc8_gather_workspace_bytes(g).  Same results
 * either way.
 *
 * Arguments: the new tokens, strides, caches, scales, block table, cu_q_lens
 * and context_kv_lens as in kvc8_store (num_tokens == cu_q_lens[B]); the
 * offsets, outputs, strides, workspace and error word as in
 * kvc8_dequant_gather, where context_seq_offset (or, when NULL, the exclusive
 * prefix sum of context_kv_lens + q) places each sequence.  num_tokens == 0
 * is a plain gather of the cached positions.  Errors as in the two calls; an
 * output row outside [0, out_rows) is reported and not written (its codes are
 * still stored).
 */
kvc8_status kvc8_append_gather(const kvc8_geom *g, int64_t num_tokens, const void *key_states,
                               const void *value_states, int64_t x_tok_stride,
                               int64_t x_head_stride, int8_t *key_cache, int8_t *value_cache,
                               float *key_scale, float *value_scale,
                               const int32_t *block_table, const int32_t *cu_q_lens,
                               const int32_t *context_kv_lens,
                               const int64_t *context_seq_offset, void *key_out,
                               void *value_out, int64_t out_rows, int64_t out_tok_stride,
                               int64_t out_head_stride, void *workspace,
                               size_t workspace_bytes, int32_t *dev_error, cudaStream_t stream);

/*
 * kvc8_build_append_metadata -- the plan of kvc8_append_gather alone, written
 * into `workspace` (same size rule as kvc8_build_metadata): tiles over the
 * cached positions context_kv_lens[b], offsets over context_kv_lens[b] + q_b
 * (or the caller's context_seq_offset), optionally copied to offsets_out.
 * Lets the layers of one model step share one plan through
 * kvc8_append_gather_planned.
 */
kvc8_status kvc8_build_append_metadata(const kvc8_geom *g, const int32_t *cu_q_lens,
                                       const int32_t *context_kv_lens,
                                       const int64_t *context_seq_offset, int64_t *offsets_out,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_error, cudaStream_t stream);

/*
 * kvc8_append_gather_planned -- kvc8_append_gather with a plan that an earlier
 * kvc8_build_append_metadata wrote into `workspace` for the same cu_q_lens,
 * context_kv_lens, offsets and geometry.  One fused launch (after an 8-byte
 * memset of the plan's work counter; calls that overlap on the GPU need
 * separate workspaces).  Arguments as in kvc8_append_gather.
 */
kvc8_status kvc8_append_gather_planned(const kvc8_geom *g, int64_t num_tokens,
                                       const void *key_states, const void *value_states,
                                       int64_t x_tok_stride, int64_t x_head_stride,
                                       int8_t *key_cache, int8_t *value_cache, float *key_scale,
                                       float *value_scale, const int32_t *block_table,
                                       const int32_t *cu_q_lens, const int32_t *context_kv_lens,
                                       void *key_out, void *value_out, int64_t out_rows,
                                       int64_t out_tok_stride, int64_t out_head_stride,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_error, cudaStream_t stream);

/* Bytes of device workspace kvc8_paged_decode_attention needs for this
 * geometry and number of query heads (a bound from num_seqs, kv_heads,
 * max_blocks_per_seq * block_size and the group size).  Host function. */
size_t kvc8_attention_workspace_bytes(const kvc8_geom *g, int32_t num_q_heads);

/*
 * kvc8_paged_decode_attention -- one decode query per sequence attends over its
 * context in the int8 paged cache, reading the codes directly: the pages'
 * MojoPagedDecodeGQA ("Mojo Opset" README, "Op List", Attention) on the
 * values MojoDequantFromPagedKVCache ([PR379]) would produce, without writing
 * them out.  The pages give no formula; the reading is grouped-query scaled
 * dot-product attention: query head j (0 <= j < num_q_heads) uses kv head
 * j / (num_q_heads / H), and
 *   out[b][j] = sum_{p < context_lengths[b]} w_p * V'[b][p][h],
 *   w = softmax_p(softmax_scale * <query[b][j], K'[b][p][h]>),
 * with K', V' the bf16 rows kvc8_dequant_gather would write for those
 * positions.  Computed with bf16 tensor-core products, fp32 accumulation,
 * bf16-rounded softmax weights and a bf16 output (round to nearest even); an
 * empty context gives zeros.  Enqueues a split plan, the attention kernel and
 * a merge of the splits (programmatic dependent launches, no host sync).
 *
 *   num_q_heads     H * group with 1 <= group <= 8
 *   query           bf16 [B][num_q_heads][D], element strides (q_seq_stride,
 *                   q_head_stride, 1), multiples of 8, 16-byte aligned
 *   caches, scales, block_table  as in kvc8_dequant_gather (all three modes)
 *   context_lengths int32 [B], positions to attend per sequence
 *   softmax_scale   finite, e.g. 1/sqrt(D)
 *   out             bf16 [B][num_q_heads][D], strides (out_seq_stride,
 *                   out_head_stride, 1)
 *   workspace       >= kvc8_attention_workspace_bytes(g, num_q_heads) bytes,
 *                   256-byte aligned; calls that overlap on the GPU need
 *                   separate workspaces
 * Supported: head_dim 64 or 128 and block_size a multiple of 16, else
 * KVC8_ERR_UNSUPPORTED.  Block ids outside the pool are reported through
 * dev_error and their 16-position pieces left out.
 */
kvc8_status kvc8_paged_decode_attention(const kvc8_geom *g, int32_t num_q_heads,
                                        const void *query, int64_t q_seq_stride,
                                        int64_t q_head_stride, const int8_t *key_cache,
                                        const int8_t *value_cache, const float *key_scale,
                                        const float *value_scale, const int32_t *block_table,
                                        const int32_t *context_lengths, float softmax_scale,
                                        void *out, int64_t out_seq_stride,
                                        int64_t out_head_stride, void *workspace,
                                        size_t workspace_bytes, int32_t *dev_error,
                                        cudaStream_t stream);

/*
 * kvc8_store_bf16 -- the same scatter as kvc8_store for a bf16 paged cache,
 * without quantisation: MojoStorePagedKVCache of the "Mojo Opset" README
 * ("Op List", KVCache), the int8 store's sibling ([PR379] pass 1, "Must fix":
 * the sibling checks cu_q_lens; here a NULL cu_q_lens means decode, as in
 * kvc8_store).  Each new token's K and V rows are copied bit for bit to
 * key_cache/value_cache[block][h][slot][0:D] (bf16 [NB][H][bs][D]), with the
 * slot mapping and the argument and error conventions of kvc8_store;
 * g->quant_mode is ignored.
 */
kvc8_status kvc8_store_bf16(const kvc8_geom *g, int64_t num_tokens,
                            const void *key_states, const void *value_states,
                            int64_t x_tok_stride, int64_t x_head_stride,
                            void *key_cache, void *value_cache,
                            const int32_t *block_table, const int32_t *cu_q_lens,
                            const int32_t *context_kv_lens, int32_t *dev_error,
                            cudaStream_t stream);

/*
 * kvc8_gather_bf16 -- gather a bf16 paged cache into contiguous rows (the
 * layout of kvc8_dequant_gather's output, values copied bit for bit), with the
 * plan, offsets, strides, workspace and error conventions of
 * kvc8_dequant_gather; g->quant_mode is ignored.
 */
kvc8_status kvc8_gather_bf16(const kvc8_geom *g, const void *key_cache,
                             const void *value_cache, const int32_t *block_table,
                             const int32_t *context_lengths,
                             const int64_t *context_seq_offset, void *key_out,
                             void *value_out, int64_t out_rows, int64_t out_tok_stride,
                             int64_t out_head_stride, void *workspace,
                             size_t workspace_bytes, int32_t *dev_error,
                             cudaStream_t stream);

/* Largest num_seqs that kvc8_dequant_gather_noalloc accepts. */
#define KVC8_NOALLOC_MAX_SEQS 4096

/*
 * kvc8_dequant_gather_noalloc -- kvc8_dequant_gather for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry point;
 * it exists for library users.
 *
 * Who needs it: code that runs inside a host runtime owning all device memory
 * and offering its plugins no allocator, or a serving loop that must not
 * allocate once it is running (an allocation can synchronise the device and
 * upsets a memory plan fixed in advance).  Such a caller cannot provide the
 * `workspace` that kvc8_dequant_gather needs.
 *
 * What it does instead: the gather's plan (offsets, tile prefix, work counter,
 * about 50 KB) lives in one fixed device array inside the library, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc or cudaFree, no allocating library call);
 * the caller still passes every input and output.  num_seqs above
 * KVC8_NOALLOC_MAX_SEQS is rejected with KVC8_ERR_UNSUPPORTED before anything
 * is enqueued.
 *
 * Set-up: the first call on a device looks up that device's copy of the array
 * (cudaGetSymbolAddress, with the device current) and remembers it.  With
 * lazy module loading, that lookup is also when the library's device code and
 * globals -- this array included -- are loaded onto the device, which
 * allocates device memory; and each kernel's code is loaded at its first
 * launch.  So make the first call on each device at start-up, before any
 * stream capture and before the phase that must not allocate: a call with
 * g->num_seqs = 0 does the lookup and nothing else, and one call on a small
 * real batch also loads the plan and gather kernels.
 *
 * Sharing: all calls on a device use the one array.  Each call rewrites every
 * field it reads from it (the plan kernel zeroes the work counter), but calls
 * whose work overlaps on the GPU (other streams, other host threads) race on
 * it and must be serialised by the caller.
 *
 * Arguments, checks, layouts and results are those of kvc8_dequant_gather in
 * every quant_mode (0, 1 and 2), without the workspace pair; the same
 * geometries are refused, plus num_seqs above KVC8_NOALLOC_MAX_SEQS.
 */
kvc8_status kvc8_dequant_gather_noalloc(const kvc8_geom *g, const int8_t *key_cache,
                                        const int8_t *value_cache,
                                        const float *key_scale, const float *value_scale,
                                        const int32_t *block_table,
                                        const int32_t *context_lengths,
                                        const int64_t *context_seq_offset, void *key_out,
                                        void *value_out, int64_t out_rows,
                                        int64_t out_tok_stride, int64_t out_head_stride,
                                        int32_t *dev_error, cudaStream_t stream);

/*
 * kvc8_get_error -- synchronise `stream`, copy the device error word to
 * *host_code (host pointer) and return KVC8_ERR_DEVICE_BOUNDS if it is
 * non-zero, KVC8_OK if zero.  With reset != 0 the word is zeroed afterwards.
 */
kvc8_status kvc8_get_error(int32_t *dev_error, int32_t *host_code, int32_t reset,
                           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC8_H */
