// kvc8_internal.cuh -- device helpers and launcher declarations shared by the
// libkvc8 translation units (store, gather, C ABI).  Not part of the ABI.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "kvc8.h"

namespace kvc8 {

// ---------------------------------------------------------------------------
// Memory access helpers (inline PTX).

// 16-byte read-once load: bypass L1 allocation, data is streamed.
__device__ __forceinline__ uint4 ld_stream_16(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 4-byte read-only load through the non-coherent path (metadata, scales).
__device__ __forceinline__ float ld_nc_f32(const float *p) {
    float v;
    asm("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int32_t ld_nc_s32(const int32_t *p) {
    int32_t v;
    asm("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// 8-byte store with default (write-back) caching: the cache pages are read
// again by the consumer of the cache.
__device__ __forceinline__ void st_8(void *p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// 16-byte streaming store (evict-first): write-once output.
__device__ __forceinline__ void st_stream_16(void *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

// 32-byte streaming store (sm_100+ 256-bit vector store).
__device__ __forceinline__ void st_stream_32(void *p, uint4 lo, uint4 hi) {
    asm volatile("st.global.cs.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                 "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z),
                 "r"(hi.w)
                 : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// First device error wins; later ones are dropped.
__device__ __forceinline__ void report(int32_t *dev_error, int32_t code) {
    if (dev_error != nullptr) atomicCAS(dev_error, 0, code);
}

// Sequence b of new token t with cu[b], cu[b+1] and ctx[b], in as few
// dependent loads as the search allows: coarse ballot rounds narrow [lo, hi)
// to at most 32 sequences, then lane j loads cu[lo+j], cu[lo+j+1] and
// ctx[lo+j] at once and the answer's three values come back by shuffles.
// All lanes get the same result; if t lies past cu[hi], b = hi - 1 and
// [first, next) does not contain t (the caller reports it).
struct TokenSeq {
    int b;
    int64_t first, next, ctx;
};

// The search in two halves, so that a caller can issue the loads of one token
// and consume them later: seq_probe_begin runs the coarse rounds and issues the
// final round's loads, seq_probe_end consumes them.
struct SeqProbe {
    int lo, hi;
    int32_t c0, c1, cx;  // this lane's cu[lo+lane], cu[lo+lane+1], ctx[lo+lane]
};

__device__ __forceinline__ SeqProbe seq_probe_begin(const int32_t *cu, const int32_t *ctx, int B,
                                                    int64_t t, int lane) {
    SeqProbe p;
    int lo = 0, hi = B;  // cu[lo] <= t < cu[hi]
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) >> 5;
        const int idx = lo + step * (lane + 1);
        const bool le = idx < hi && (int64_t)ld_nc_s32(cu + idx) <= t;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, le);
        if (m != 0u) lo += step * (32 - __clz(m));
        hi = min(hi, lo + step);
    }
    p.lo = lo;
    p.hi = hi;
    p.c0 = 0;
    p.c1 = 0x7FFFFFFF;
    p.cx = 0;
    const int j = lo + lane;
    if (j < hi) {
        p.c0 = ld_nc_s32(cu + j);
        p.c1 = ld_nc_s32(cu + j + 1);
        p.cx = ld_nc_s32(ctx + j);
    }
    return p;
}

__device__ __forceinline__ TokenSeq seq_probe_end(const SeqProbe &p, int64_t t, int lane) {
    const int j = p.lo + lane;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, j < p.hi && (int64_t)p.c1 <= t);
    const int k = min(__popc(m), p.hi - p.lo - 1);
    TokenSeq r;
    r.b = p.lo + k;
    r.first = __shfl_sync(0xFFFFFFFFu, p.c0, k);
    r.next = __shfl_sync(0xFFFFFFFFu, p.c1, k);
    r.ctx = __shfl_sync(0xFFFFFFFFu, p.cx, k);
    return r;
}

__device__ __forceinline__ TokenSeq seq_ctx_of_token(const int32_t *cu, const int32_t *ctx, int B,
                                                     int64_t t, int lane) {
    return seq_probe_end(seq_probe_begin(cu, ctx, B, t, lane), t, lane);
}

// ---------------------------------------------------------------------------
// Gather plan, written by the plan kernel into the caller's workspace.
//   header.total_tiles : number of (sequence, logical block) tiles
//   header.work_counter: next work item of the gather (reset by the plan)
//   offsets[B]         : first output row of each sequence (int64)
//   tile_start[B + 1]  : exclusive prefix of ceil(len_b / bs), tile_start[B] = total
struct PlanHeader {
    int64_t total_tiles;
    int64_t work_counter;  // gather work items handed out so far (atomic)
    int64_t pad[2];
};

constexpr size_t kAlign = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t plan_offsets_at(int32_t) { return align_up(sizeof(PlanHeader), kAlign); }
__host__ __device__ inline size_t plan_tile_start_at(int32_t num_seqs) {
    return plan_offsets_at(num_seqs) + align_up(sizeof(int64_t) * (size_t)(num_seqs > 0 ? num_seqs : 1), kAlign);
}
__host__ __device__ inline size_t plan_bytes(int32_t num_seqs) {
    return plan_tile_start_at(num_seqs) + align_up(sizeof(int32_t) * ((size_t)num_seqs + 1), kAlign);
}

// ---------------------------------------------------------------------------
// Launchers (host).  Arguments are validated by the C ABI before these run.

struct StoreArgs {
    kvc8_geom g;
    int64_t num_tokens;
    const uint16_t *k_states;
    const uint16_t *v_states;
    int64_t x_tok_stride;
    int64_t x_head_stride;
    int8_t *k_cache;
    int8_t *v_cache;
    float *k_scale;
    float *v_scale;
    const int32_t *block_table;
    const int32_t *cu_q_lens;
    const int32_t *context_kv_lens;
    int32_t *dev_error;
    unsigned long long bs_magic;  // ceil(2^64 / block_size) for block_size >= 2
};

struct GatherArgs {
    kvc8_geom g;
    const int8_t *k_cache;
    const int8_t *v_cache;
    const float *k_scale;
    const float *v_scale;
    const int32_t *block_table;
    const int32_t *context_lengths;
    uint16_t *k_out;
    uint16_t *v_out;
    int64_t out_rows;
    int64_t out_tok_stride;
    int64_t out_head_stride;
    const void *plan;
    int32_t *dev_error;
};

// bf16 paged cache (no quantisation): caches are uint16_t (bf16 bits).
struct StoreBf16Args {
    kvc8_geom g;
    int64_t num_tokens;
    const uint16_t *k_states;
    const uint16_t *v_states;
    int64_t x_tok_stride;
    int64_t x_head_stride;
    uint16_t *k_cache;
    uint16_t *v_cache;
    const int32_t *block_table;
    const int32_t *cu_q_lens;
    const int32_t *context_kv_lens;
    int32_t *dev_error;
};

struct GatherBf16Args {
    kvc8_geom g;
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    const int32_t *block_table;
    const int32_t *context_lengths;
    uint16_t *k_out;
    uint16_t *v_out;
    int64_t out_rows;
    int64_t out_tok_stride;
    int64_t out_head_stride;
    const void *plan;
    int32_t *dev_error;
};

// Fused append + gather: the new tokens' rows, quantised and written to the
// cache, and their dequantised values written straight to the output rows
// after each sequence's cached positions.  The gather part of the same launch
// reads only the cached positions (GatherArgs.context_lengths = the cached
// lengths), so the two parts touch disjoint cache bytes.
struct AppendArgs {
    int64_t num_tokens;
    int64_t items;  // append work items (kAppendRowsPerItem rows each), first in the item order
    const uint16_t *k_states;
    const uint16_t *v_states;
    int64_t x_tok_stride;
    int64_t x_head_stride;
    int8_t *k_cache;
    int8_t *v_cache;
    float *k_scale;  // mode 0: the scale caches (written); mode 1: the static scales
    float *v_scale;
    const int32_t *cu_q_lens;  // NULL: one new token per sequence
    const int32_t *context_kv_lens;
};

constexpr int kAppendRowsPerItem = 8;  // one (token, K|V, head) row per warp of a CTA

// Paged decode attention over the int8 cache (kvc8_attention.cu).
struct AttnArgs {
    kvc8_geom g;
    int32_t group;      // query heads per kv head (1..8)
    int32_t chunk;      // positions per split (a multiple of 16)
    const uint16_t *q;  // bf16 [B][H * group][D], strides below
    int64_t q_seq_stride;
    int64_t q_head_stride;
    const int8_t *k_cache;
    const int8_t *v_cache;
    const float *k_scale;
    const float *v_scale;
    const int32_t *block_table;
    const int32_t *context_lengths;
    float scale_log2;  // softmax scale * log2(e)
    uint16_t *out;     // bf16 [B][H * group][D], strides below
    int64_t out_seq_stride;
    int64_t out_head_stride;
    const void *plan;  // the split plan (plan kernel with block_size = chunk)
    float *part_o;     // [items][group][D] unnormalised partial outputs
    float *part_m;     // [items][group] running maxima (log2 domain)
    float *part_l;     // [items][group] running sums
    int32_t *dev_error;
};

constexpr int kAttnChunk = 2048;  // positions per split of a sequence

// Workspace of the attention: the split plan, then the partials.
size_t attention_workspace_bytes(const kvc8_geom &g, int group);
cudaError_t launch_attention(AttnArgs a, void *workspace, cudaStream_t stream);

cudaError_t launch_store(const StoreArgs &a, cudaStream_t stream);
cudaError_t launch_store_bf16(const StoreBf16Args &a, cudaStream_t stream);
cudaError_t launch_gather_bf16(const GatherBf16Args &a, bool use_pdl, cudaStream_t stream);
cudaError_t launch_plan(const kvc8_geom &g, const int32_t *context_lengths,
                        const int64_t *context_seq_offset, int64_t *offsets_out, void *plan,
                        int32_t *dev_error, cudaStream_t stream);
// Plan of an append + gather: tiles cover the cached lengths, offsets the
// lengths after the append (cached + new tokens, new = cu_q_lens[b+1] -
// cu_q_lens[b], or 1 each when cu_q_lens is NULL).
cudaError_t launch_plan_append(const kvc8_geom &g, const int32_t *context_kv_lens,
                               const int32_t *cu_q_lens, const int64_t *context_seq_offset,
                               int64_t *offsets_out, void *plan, int32_t *dev_error,
                               cudaStream_t stream);
// Plan of a gather over the cached and the newly stored positions
// (tiles and offsets over context_kv_lens + new), the spans written to
// spans_out[B] for the gather to read as its lengths.
cudaError_t launch_plan_span(const kvc8_geom &g, const int32_t *context_kv_lens,
                             const int32_t *cu_q_lens, const int64_t *context_seq_offset,
                             void *plan, int32_t *spans_out, int32_t *dev_error,
                             cudaStream_t stream);
// The fused append + gather launch (a programmatic dependent of the plan when use_pdl).
cudaError_t launch_append_gather(const GatherArgs &a, const AppendArgs &p, bool use_pdl,
                                 cudaStream_t stream);
// use_pdl: launch as a programmatic dependent of the previous kernel (the plan).
cudaError_t launch_gather(const GatherArgs &a, bool use_pdl, cudaStream_t stream);
// Zero the gather's work counter in a plan built earlier (for planned gathers).
cudaError_t reset_plan_counter(void *plan, cudaStream_t stream);

// Per-device SM count (cached).
int sm_count();

// Host-side caches of per-device launch facts.  Each is one atomic word per
// device, so host threads that launch at the same time -- on one device or on
// several -- read either a complete entry or none (and then query again).
constexpr int kMaxDevices = 64;

struct OccupancySlots {
    std::atomic<uint64_t> word[kMaxDevices];  // ((smem + 1) << 8) | CTAs per SM; 0 = unknown
};

// Resident CTAs per SM of `kern` with `threads` threads and `smem` bytes of
// dynamic shared memory on the current device, cached in `slots` (one
// OccupancySlots per kernel variant).
template <typename Kernel>
cudaError_t occupancy(OccupancySlots &slots, Kernel kern, int threads, size_t smem, int *occ) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    const uint64_t key = ((uint64_t)smem + 1) << 8;
    if (cached) {
        const uint64_t w = slots.word[dev].load(std::memory_order_relaxed);
        if ((w & ~(uint64_t)0xFF) == key) {
            *occ = (int)(w & 0xFF);
            return cudaSuccess;
        }
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem);
    if (e != cudaSuccess) return e;
    n = n < 1 ? 1 : (n > 255 ? 255 : n);
    if (cached) slots.word[dev].store(key | (uint64_t)n, std::memory_order_relaxed);
    *occ = n;
    return cudaSuccess;
}

// Host-side argument checks shared by the entry points (kvc8_api.cu).
kvc8_status check_geom(const kvc8_geom *g);
kvc8_status check_gather_args(const kvc8_geom *g, const int8_t *kc, const int8_t *vc,
                              const float *ks, const float *vs, const int32_t *bt,
                              const int32_t *lens, const void *ko, const void *vo,
                              int64_t out_rows, int64_t tok_stride, int64_t head_stride);

}  // namespace kvc8
