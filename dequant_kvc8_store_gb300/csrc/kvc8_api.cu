// kvc8_api.cu -- the extern "C" entry points of libkvc8 (declared in kvc8.h):
// host-side argument checks, then the launches in kvc8_store.cu,
// kvc8_gather.cu, kvc8_bf16.cu and kvc8_attention.cu.  Nothing here allocates device memory or synchronises,
// except kvc8_get_error, whose purpose is to synchronise.
#include <cmath>
#include <cstdint>

#include "kvc8_internal.cuh"

namespace kvc8 {

int sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const bool in_range = dev >= 0 && dev < kMaxDevices;
    if (in_range) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (in_range) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

constexpr int kMaxHeadDim = 256;
// Appended rows (tokens x 2 x kv_heads) up to which the fused append + gather
// beats the store followed by a gather (measured on decode-shaped batches:
// 16 384 rows still won, 65 536 lost).
constexpr int64_t kFusedAppendMaxRows = 16384;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kvc8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVC8_OK : KVC8_ERR_CUDA; }

kvc8_status check_workspace(const kvc8_geom *g, const void *ws, size_t bytes) {
    if (ws == nullptr || !aligned(ws, kAlign)) return KVC8_ERR_WORKSPACE;
    if (bytes < plan_bytes(g->num_seqs)) return KVC8_ERR_WORKSPACE;
    return KVC8_OK;
}

}  // namespace

kvc8_status check_geom(const kvc8_geom *g) {
    if (g == nullptr) return KVC8_ERR_INVALID_ARG;
    if (g->num_seqs < 0 || g->kv_heads < 1 || g->block_size < 1 || g->num_blocks < 1 ||
        g->max_blocks_per_seq < 1 || g->head_dim < 16)
        return KVC8_ERR_INVALID_ARG;
    if (g->quant_mode < 0 || g->quant_mode > 2) return KVC8_ERR_INVALID_ARG;
    if (g->head_dim % 16 != 0) return KVC8_ERR_INVALID_ARG;
    if (g->head_dim > kMaxHeadDim) return KVC8_ERR_UNSUPPORTED;
    // tile and unit counters are 32/64-bit; keep B * MB * 2H well inside int64
    if ((int64_t)g->num_seqs * g->max_blocks_per_seq > (int64_t)INT32_MAX) return KVC8_ERR_UNSUPPORTED;
    return KVC8_OK;
}

kvc8_status check_gather_args(const kvc8_geom *g, const int8_t *kc, const int8_t *vc,
                              const float *ks, const float *vs, const int32_t *bt,
                              const int32_t *lens, const void *ko, const void *vo,
                              int64_t out_rows, int64_t tok_stride, int64_t head_stride) {
    if (kc == nullptr || vc == nullptr || ks == nullptr || vs == nullptr || bt == nullptr ||
        lens == nullptr || ko == nullptr || vo == nullptr)
        return KVC8_ERR_INVALID_ARG;
    if (out_rows < 0 || tok_stride < 0 || head_stride < 0) return KVC8_ERR_INVALID_ARG;
    if (tok_stride % 8 != 0 || head_stride % 8 != 0) return KVC8_ERR_INVALID_ARG;
    if (!aligned(ko, 16) || !aligned(vo, 16) || !aligned(kc, 16) || !aligned(vc, 16))
        return KVC8_ERR_INVALID_ARG;
    if (!aligned(ks, 16) || !aligned(vs, 16)) return KVC8_ERR_INVALID_ARG;
    return KVC8_OK;
}

}  // namespace kvc8

using namespace kvc8;

extern "C" {

const char *kvc8_status_str(kvc8_status s) {
    switch (s) {
        case KVC8_OK: return "ok";
        case KVC8_ERR_INVALID_ARG: return "invalid argument";
        case KVC8_ERR_UNSUPPORTED: return "unsupported geometry";
        case KVC8_ERR_CUDA: return "CUDA error";
        case KVC8_ERR_DEVICE_BOUNDS: return "device-side bounds error";
        case KVC8_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    }
    return "unknown status";
}

int32_t kvc8_version(void) { return 10000; }

kvc8_status kvc8_store(const kvc8_geom *g, int64_t num_tokens, const void *key_states,
                       const void *value_states, int64_t x_tok_stride, int64_t x_head_stride,
                       int8_t *key_cache, int8_t *value_cache, float *key_scale,
                       float *value_scale, const int32_t *block_table, const int32_t *cu_q_lens,
                       const int32_t *context_kv_lens, int32_t *dev_error, cudaStream_t stream) {
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (num_tokens < 0) return KVC8_ERR_INVALID_ARG;
    if (num_tokens > INT32_MAX) return KVC8_ERR_UNSUPPORTED;  // token indices are 32-bit
    if (cu_q_lens == nullptr && num_tokens != g->num_seqs) return KVC8_ERR_INVALID_ARG;
    if (num_tokens == 0 || g->num_seqs == 0) return num_tokens == 0 ? KVC8_OK : KVC8_ERR_INVALID_ARG;
    if (key_states == nullptr || value_states == nullptr || key_cache == nullptr ||
        value_cache == nullptr || key_scale == nullptr || value_scale == nullptr ||
        block_table == nullptr || context_kv_lens == nullptr)
        return KVC8_ERR_INVALID_ARG;
    if (x_tok_stride < 0 || x_head_stride < 0 || x_tok_stride % 8 != 0 || x_head_stride % 8 != 0)
        return KVC8_ERR_INVALID_ARG;
    if (!aligned(key_states, 16) || !aligned(value_states, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16))
        return KVC8_ERR_INVALID_ARG;
    if (!aligned(key_scale, 16) || !aligned(value_scale, 16)) return KVC8_ERR_INVALID_ARG;
    StoreArgs a;
    a.g = *g;
    a.num_tokens = num_tokens;
    a.k_states = static_cast<const uint16_t *>(key_states);
    a.v_states = static_cast<const uint16_t *>(value_states);
    a.x_tok_stride = x_tok_stride;
    a.x_head_stride = x_head_stride;
    a.k_cache = key_cache;
    a.v_cache = value_cache;
    a.k_scale = key_scale;
    a.v_scale = value_scale;
    a.block_table = block_table;
    a.cu_q_lens = cu_q_lens;
    a.context_kv_lens = context_kv_lens;
    a.dev_error = dev_error;
    a.bs_magic = g->block_size >= 2 ? ~0ull / (unsigned long long)g->block_size + 1ull : 0ull;
    return cuda_status(launch_store(a, stream));
}

// The plan, then room for one int32 per sequence (the spans of a long
// append, which kvc8_append_gather gathers in a second pass).
size_t kvc8_gather_workspace_bytes(const kvc8_geom *g) {
    if (g == nullptr || g->num_seqs < 0) return 0;
    return plan_bytes(g->num_seqs) +
           align_up(sizeof(int32_t) * (size_t)(g->num_seqs > 0 ? g->num_seqs : 1), kAlign);
}

kvc8_status kvc8_build_metadata(const kvc8_geom *g, const int32_t *context_lengths,
                                const int64_t *context_seq_offset, int64_t *offsets_out,
                                void *workspace, size_t workspace_bytes, int32_t *dev_error,
                                cudaStream_t stream) {
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (context_lengths == nullptr && g->num_seqs > 0) return KVC8_ERR_INVALID_ARG;
    st = check_workspace(g, workspace, workspace_bytes);
    if (st != KVC8_OK) return st;
    return cuda_status(launch_plan(*g, context_lengths, context_seq_offset, offsets_out,
                                   workspace, dev_error, stream));
}

kvc8_status kvc8_dequant_gather(const kvc8_geom *g, const int8_t *key_cache,
                                const int8_t *value_cache, const float *key_scale,
                                const float *value_scale, const int32_t *block_table,
                                const int32_t *context_lengths,
                                const int64_t *context_seq_offset, void *key_out,
                                void *value_out, int64_t out_rows, int64_t out_tok_stride,
                                int64_t out_head_stride, void *workspace,
                                size_t workspace_bytes, int32_t *dev_error,
                                cudaStream_t stream) {
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (g->num_seqs == 0) return KVC8_OK;
    st = check_gather_args(g, key_cache, value_cache, key_scale, value_scale, block_table,
                           context_lengths, key_out, value_out, out_rows, out_tok_stride,
                           out_head_stride);
    if (st != KVC8_OK) return st;
    st = check_workspace(g, workspace, workspace_bytes);
    if (st != KVC8_OK) return st;
    cudaError_t e = launch_plan(*g, context_lengths, context_seq_offset, nullptr, workspace,
                                dev_error, stream);
    if (e != cudaSuccess) return KVC8_ERR_CUDA;
    GatherArgs a;
    a.g = *g;
    a.k_cache = key_cache;
    a.v_cache = value_cache;
    a.k_scale = key_scale;
    a.v_scale = value_scale;
    a.block_table = block_table;
    a.context_lengths = context_lengths;
    a.k_out = static_cast<uint16_t *>(key_out);
    a.v_out = static_cast<uint16_t *>(value_out);
    a.out_rows = out_rows;
    a.out_tok_stride = out_tok_stride;
    a.out_head_stride = out_head_stride;
    a.plan = workspace;
    a.dev_error = dev_error;
    return cuda_status(launch_gather(a, /*use_pdl=*/true, stream));
}

kvc8_status kvc8_dequant_gather_planned(const kvc8_geom *g, const int8_t *key_cache,
                                        const int8_t *value_cache, const float *key_scale,
                                        const float *value_scale, const int32_t *block_table,
                                        const int32_t *context_lengths, void *key_out,
                                        void *value_out, int64_t out_rows,
                                        int64_t out_tok_stride, int64_t out_head_stride,
                                        void *workspace, size_t workspace_bytes,
                                        int32_t *dev_error, cudaStream_t stream) {
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (g->num_seqs == 0) return KVC8_OK;
    st = check_gather_args(g, key_cache, value_cache, key_scale, value_scale, block_table,
                           context_lengths, key_out, value_out, out_rows, out_tok_stride,
                           out_head_stride);
    if (st != KVC8_OK) return st;
    st = check_workspace(g, workspace, workspace_bytes);
    if (st != KVC8_OK) return st;
    GatherArgs a;
    a.g = *g;
    a.k_cache = key_cache;
    a.v_cache = value_cache;
    a.k_scale = key_scale;
    a.v_scale = value_scale;
    a.block_table = block_table;
    a.context_lengths = context_lengths;
    a.k_out = static_cast<uint16_t *>(key_out);
    a.v_out = static_cast<uint16_t *>(value_out);
    a.out_rows = out_rows;
    a.out_tok_stride = out_tok_stride;
    a.out_head_stride = out_head_stride;
    a.plan = workspace;
    a.dev_error = dev_error;
    if (reset_plan_counter(workspace, stream) != cudaSuccess) return KVC8_ERR_CUDA;
    return cuda_status(launch_gather(a, /*use_pdl=*/false, stream));
}

// Shared checks and argument packing of the append + gather entry points.
static kvc8_status append_args(const kvc8_geom *g, int64_t num_tokens, const void *key_states,
                               const void *value_states, int64_t x_tok_stride,
                               int64_t x_head_stride, int8_t *key_cache, int8_t *value_cache,
                               float *key_scale, float *value_scale,
                               const int32_t *block_table, const int32_t *cu_q_lens,
                               const int32_t *context_kv_lens, void *key_out, void *value_out,
                               int64_t out_rows, int64_t out_tok_stride,
                               int64_t out_head_stride, void *workspace,
                               size_t workspace_bytes, int32_t *dev_error, GatherArgs *a,
                               AppendArgs *p) {
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (num_tokens < 0) return KVC8_ERR_INVALID_ARG;
    if (num_tokens > INT32_MAX) return KVC8_ERR_UNSUPPORTED;  // token indices are 32-bit
    if (cu_q_lens == nullptr && num_tokens != g->num_seqs) return KVC8_ERR_INVALID_ARG;
    // the fused kernel indexes its work items and appended rows in 32 bits
    if ((int64_t)g->num_seqs * g->max_blocks_per_seq * g->kv_heads > (int64_t)INT32_MAX ||
        num_tokens * 2 * g->kv_heads > (int64_t)INT32_MAX)
        return KVC8_ERR_UNSUPPORTED;
    st = check_gather_args(g, key_cache, value_cache, key_scale, value_scale, block_table,
                           context_kv_lens, key_out, value_out, out_rows, out_tok_stride,
                           out_head_stride);
    if (st != KVC8_OK) return st;
    if (num_tokens > 0) {
        if (key_states == nullptr || value_states == nullptr) return KVC8_ERR_INVALID_ARG;
        if (x_tok_stride < 0 || x_head_stride < 0 || x_tok_stride % 8 != 0 ||
            x_head_stride % 8 != 0)
            return KVC8_ERR_INVALID_ARG;
        if (!aligned(key_states, 16) || !aligned(value_states, 16)) return KVC8_ERR_INVALID_ARG;
    }
    st = check_workspace(g, workspace, workspace_bytes);
    if (st != KVC8_OK) return st;
    a->g = *g;
    a->k_cache = key_cache;
    a->v_cache = value_cache;
    a->k_scale = key_scale;
    a->v_scale = value_scale;
    a->block_table = block_table;
    a->context_lengths = context_kv_lens;  // the gather part reads the cached positions
    a->k_out = static_cast<uint16_t *>(key_out);
    a->v_out = static_cast<uint16_t *>(value_out);
    a->out_rows = out_rows;
    a->out_tok_stride = out_tok_stride;
    a->out_head_stride = out_head_stride;
    a->plan = workspace;
    a->dev_error = dev_error;
    p->num_tokens = num_tokens;
    const int64_t rows = num_tokens * 2 * g->kv_heads;
    p->items = (rows + kAppendRowsPerItem - 1) / kAppendRowsPerItem;
    p->k_states = static_cast<const uint16_t *>(key_states);
    p->v_states = static_cast<const uint16_t *>(value_states);
    p->x_tok_stride = x_tok_stride;
    p->x_head_stride = x_head_stride;
    p->k_cache = key_cache;
    p->v_cache = value_cache;
    p->k_scale = key_scale;
    p->v_scale = value_scale;
    p->cu_q_lens = cu_q_lens;
    p->context_kv_lens = context_kv_lens;
    return KVC8_OK;
}

kvc8_status kvc8_append_gather(const kvc8_geom *g, int64_t num_tokens, const void *key_states,
                               const void *value_states, int64_t x_tok_stride,
                               int64_t x_head_stride, int8_t *key_cache, int8_t *value_cache,
                               float *key_scale, float *value_scale,
                               const int32_t *block_table, const int32_t *cu_q_lens,
                               const int32_t *context_kv_lens,
                               const int64_t *context_seq_offset, void *key_out,
                               void *value_out, int64_t out_rows, int64_t out_tok_stride,
                               int64_t out_head_stride, void *workspace,
                               size_t workspace_bytes, int32_t *dev_error, cudaStream_t stream) {
    if (g != nullptr && g->num_seqs == 0 && check_geom(g) == KVC8_OK)
        return num_tokens == 0 ? KVC8_OK : KVC8_ERR_INVALID_ARG;
    GatherArgs a;
    AppendArgs p;
    kvc8_status st = append_args(g, num_tokens, key_states, value_states, x_tok_stride,
                                 x_head_stride, key_cache, value_cache, key_scale, value_scale,
                                 block_table, cu_q_lens, context_kv_lens, key_out, value_out,
                                 out_rows, out_tok_stride, out_head_stride, workspace,
                                 workspace_bytes, dev_error, &a, &p);
    if (st != KVC8_OK) return st;
    // A long append (a prompt rather than a decode step) is faster as the
    // store kernel followed by a gather of every position: the fused kernel's
    // append rows follow the definition with one division per value.
    const size_t span_at = plan_bytes(g->num_seqs);
    const bool long_append =
        num_tokens * 2 * g->kv_heads > kFusedAppendMaxRows &&
        workspace_bytes >= span_at + sizeof(int32_t) * (size_t)g->num_seqs;
    if (long_append) {
        StoreArgs s;
        s.g = *g;
        s.num_tokens = num_tokens;
        s.k_states = p.k_states;
        s.v_states = p.v_states;
        s.x_tok_stride = x_tok_stride;
        s.x_head_stride = x_head_stride;
        s.k_cache = key_cache;
        s.v_cache = value_cache;
        s.k_scale = key_scale;
        s.v_scale = value_scale;
        s.block_table = block_table;
        s.cu_q_lens = cu_q_lens;
        s.context_kv_lens = context_kv_lens;
        s.dev_error = dev_error;
        s.bs_magic = g->block_size >= 2 ? ~0ull / (unsigned long long)g->block_size + 1ull : 0ull;
        if (launch_store(s, stream) != cudaSuccess) return KVC8_ERR_CUDA;
        int32_t *spans = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + span_at);
        if (launch_plan_span(*g, context_kv_lens, cu_q_lens, context_seq_offset, workspace, spans,
                             dev_error, stream) != cudaSuccess)
            return KVC8_ERR_CUDA;
        a.context_lengths = spans;
        return cuda_status(launch_gather(a, /*use_pdl=*/true, stream));
    }
    if (launch_plan_append(*g, context_kv_lens, cu_q_lens, context_seq_offset, nullptr,
                           workspace, dev_error, stream) != cudaSuccess)
        return KVC8_ERR_CUDA;
    return cuda_status(launch_append_gather(a, p, /*use_pdl=*/true, stream));
}

kvc8_status kvc8_build_append_metadata(const kvc8_geom *g, const int32_t *cu_q_lens,
                                       const int32_t *context_kv_lens,
                                       const int64_t *context_seq_offset, int64_t *offsets_out,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_error, cudaStream_t stream) {
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (context_kv_lens == nullptr && g->num_seqs > 0) return KVC8_ERR_INVALID_ARG;
    st = check_workspace(g, workspace, workspace_bytes);
    if (st != KVC8_OK) return st;
    return cuda_status(launch_plan_append(*g, context_kv_lens, cu_q_lens, context_seq_offset,
                                          offsets_out, workspace, dev_error, stream));
}

kvc8_status kvc8_append_gather_planned(const kvc8_geom *g, int64_t num_tokens,
                                       const void *key_states, const void *value_states,
                                       int64_t x_tok_stride, int64_t x_head_stride,
                                       int8_t *key_cache, int8_t *value_cache, float *key_scale,
                                       float *value_scale, const int32_t *block_table,
                                       const int32_t *cu_q_lens, const int32_t *context_kv_lens,
                                       void *key_out, void *value_out, int64_t out_rows,
                                       int64_t out_tok_stride, int64_t out_head_stride,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_error, cudaStream_t stream) {
    if (g != nullptr && g->num_seqs == 0 && check_geom(g) == KVC8_OK)
        return num_tokens == 0 ? KVC8_OK : KVC8_ERR_INVALID_ARG;
    GatherArgs a;
    AppendArgs p;
    kvc8_status st = append_args(g, num_tokens, key_states, value_states, x_tok_stride,
                                 x_head_stride, key_cache, value_cache, key_scale, value_scale,
                                 block_table, cu_q_lens, context_kv_lens, key_out, value_out,
                                 out_rows, out_tok_stride, out_head_stride, workspace,
                                 workspace_bytes, dev_error, &a, &p);
    if (st != KVC8_OK) return st;
    if (reset_plan_counter(workspace, stream) != cudaSuccess) return KVC8_ERR_CUDA;
    return cuda_status(launch_append_gather(a, p, /*use_pdl=*/false, stream));
}

size_t kvc8_attention_workspace_bytes(const kvc8_geom *g, int32_t num_q_heads) {
    if (g == nullptr || g->num_seqs < 0 || g->kv_heads < 1 || num_q_heads < g->kv_heads) return 0;
    return attention_workspace_bytes(*g, num_q_heads / g->kv_heads);
}

kvc8_status kvc8_paged_decode_attention(const kvc8_geom *g, int32_t num_q_heads,
                                        const void *query, int64_t q_seq_stride,
                                        int64_t q_head_stride, const int8_t *key_cache,
                                        const int8_t *value_cache, const float *key_scale,
                                        const float *value_scale, const int32_t *block_table,
                                        const int32_t *context_lengths, float softmax_scale,
                                        void *out, int64_t out_seq_stride,
                                        int64_t out_head_stride, void *workspace,
                                        size_t workspace_bytes, int32_t *dev_error,
                                        cudaStream_t stream) {
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (num_q_heads < 1 || num_q_heads % g->kv_heads != 0) return KVC8_ERR_INVALID_ARG;
    const int group = num_q_heads / g->kv_heads;
    if (group > 8 || (g->head_dim != 64 && g->head_dim != 128) || g->block_size % 16 != 0)
        return KVC8_ERR_UNSUPPORTED;
    if (!std::isfinite(softmax_scale)) return KVC8_ERR_INVALID_ARG;
    const int64_t splits =
        ((int64_t)g->max_blocks_per_seq * g->block_size + kAttnChunk - 1) / kAttnChunk;
    if ((int64_t)g->num_seqs * g->kv_heads * splits > (int64_t)INT32_MAX) return KVC8_ERR_UNSUPPORTED;
    if (g->num_seqs == 0) return KVC8_OK;
    if (query == nullptr || key_cache == nullptr || value_cache == nullptr ||
        key_scale == nullptr || value_scale == nullptr || block_table == nullptr ||
        context_lengths == nullptr || out == nullptr)
        return KVC8_ERR_INVALID_ARG;
    if (q_seq_stride < 0 || q_head_stride < 0 || q_seq_stride % 8 != 0 || q_head_stride % 8 != 0 ||
        out_seq_stride < 0 || out_head_stride < 0)
        return KVC8_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(key_scale, 16) || !aligned(value_scale, 16) || !aligned(out, 2))
        return KVC8_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned(workspace, kAlign) ||
        workspace_bytes < attention_workspace_bytes(*g, group))
        return KVC8_ERR_WORKSPACE;
    AttnArgs a = {};
    a.g = *g;
    a.group = group;
    a.q = static_cast<const uint16_t *>(query);
    a.q_seq_stride = q_seq_stride;
    a.q_head_stride = q_head_stride;
    a.k_cache = key_cache;
    a.v_cache = value_cache;
    a.k_scale = key_scale;
    a.v_scale = value_scale;
    a.block_table = block_table;
    a.context_lengths = context_lengths;
    a.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);  // log2(e)
    a.out = static_cast<uint16_t *>(out);
    a.out_seq_stride = out_seq_stride;
    a.out_head_stride = out_head_stride;
    a.dev_error = dev_error;
    return cuda_status(launch_attention(a, workspace, stream));
}

// Geometry checks for the bf16 cache (quant_mode is not used there).
static kvc8_status check_geom_bf16(const kvc8_geom *g) {
    if (g == nullptr) return KVC8_ERR_INVALID_ARG;
    kvc8_geom q = *g;
    q.quant_mode = 0;
    return check_geom(&q);
}

kvc8_status kvc8_store_bf16(const kvc8_geom *g, int64_t num_tokens, const void *key_states,
                            const void *value_states, int64_t x_tok_stride, int64_t x_head_stride,
                            void *key_cache, void *value_cache, const int32_t *block_table,
                            const int32_t *cu_q_lens, const int32_t *context_kv_lens,
                            int32_t *dev_error, cudaStream_t stream) {
    kvc8_status st = check_geom_bf16(g);
    if (st != KVC8_OK) return st;
    if (num_tokens < 0) return KVC8_ERR_INVALID_ARG;
    if (num_tokens > INT32_MAX) return KVC8_ERR_UNSUPPORTED;
    if (cu_q_lens == nullptr && num_tokens != g->num_seqs) return KVC8_ERR_INVALID_ARG;
    if (num_tokens == 0 || g->num_seqs == 0) return num_tokens == 0 ? KVC8_OK : KVC8_ERR_INVALID_ARG;
    if (key_states == nullptr || value_states == nullptr || key_cache == nullptr ||
        value_cache == nullptr || block_table == nullptr || context_kv_lens == nullptr)
        return KVC8_ERR_INVALID_ARG;
    if (x_tok_stride < 0 || x_head_stride < 0 || x_tok_stride % 8 != 0 || x_head_stride % 8 != 0)
        return KVC8_ERR_INVALID_ARG;
    if (!aligned(key_states, 16) || !aligned(value_states, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16))
        return KVC8_ERR_INVALID_ARG;
    StoreBf16Args a;
    a.g = *g;
    a.num_tokens = num_tokens;
    a.k_states = static_cast<const uint16_t *>(key_states);
    a.v_states = static_cast<const uint16_t *>(value_states);
    a.x_tok_stride = x_tok_stride;
    a.x_head_stride = x_head_stride;
    a.k_cache = static_cast<uint16_t *>(key_cache);
    a.v_cache = static_cast<uint16_t *>(value_cache);
    a.block_table = block_table;
    a.cu_q_lens = cu_q_lens;
    a.context_kv_lens = context_kv_lens;
    a.dev_error = dev_error;
    return cuda_status(launch_store_bf16(a, stream));
}

kvc8_status kvc8_gather_bf16(const kvc8_geom *g, const void *key_cache, const void *value_cache,
                             const int32_t *block_table, const int32_t *context_lengths,
                             const int64_t *context_seq_offset, void *key_out, void *value_out,
                             int64_t out_rows, int64_t out_tok_stride, int64_t out_head_stride,
                             void *workspace, size_t workspace_bytes, int32_t *dev_error,
                             cudaStream_t stream) {
    kvc8_status st = check_geom_bf16(g);
    if (st != KVC8_OK) return st;
    if (g->num_seqs == 0) return KVC8_OK;
    if (key_cache == nullptr || value_cache == nullptr || block_table == nullptr ||
        context_lengths == nullptr || key_out == nullptr || value_out == nullptr)
        return KVC8_ERR_INVALID_ARG;
    if (out_rows < 0 || out_tok_stride < 0 || out_head_stride < 0 || out_tok_stride % 8 != 0 ||
        out_head_stride % 8 != 0)
        return KVC8_ERR_INVALID_ARG;
    if (!aligned(key_out, 16) || !aligned(value_out, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16))
        return KVC8_ERR_INVALID_ARG;
    kvc8_geom q = *g;
    q.quant_mode = 0;
    st = check_workspace(&q, workspace, workspace_bytes);
    if (st != KVC8_OK) return st;
    if (launch_plan(q, context_lengths, context_seq_offset, nullptr, workspace, dev_error,
                    stream) != cudaSuccess)
        return KVC8_ERR_CUDA;
    GatherBf16Args a;
    a.g = q;
    a.k_cache = static_cast<const uint16_t *>(key_cache);
    a.v_cache = static_cast<const uint16_t *>(value_cache);
    a.block_table = block_table;
    a.context_lengths = context_lengths;
    a.k_out = static_cast<uint16_t *>(key_out);
    a.v_out = static_cast<uint16_t *>(value_out);
    a.out_rows = out_rows;
    a.out_tok_stride = out_tok_stride;
    a.out_head_stride = out_head_stride;
    a.plan = workspace;
    a.dev_error = dev_error;
    return cuda_status(launch_gather_bf16(a, /*use_pdl=*/true, stream));
}

kvc8_status kvc8_get_error(int32_t *dev_error, int32_t *host_code, int32_t reset,
                           cudaStream_t stream) {
    if (dev_error == nullptr || host_code == nullptr) return KVC8_ERR_INVALID_ARG;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, dev_error, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return KVC8_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KVC8_ERR_CUDA;
    *host_code = v;
    if (reset) {
        if (cudaMemsetAsync(dev_error, 0, sizeof(int32_t), stream) != cudaSuccess)
            return KVC8_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return KVC8_ERR_CUDA;
    }
    return v == 0 ? KVC8_OK : KVC8_ERR_DEVICE_BOUNDS;
}

}  // extern "C"
