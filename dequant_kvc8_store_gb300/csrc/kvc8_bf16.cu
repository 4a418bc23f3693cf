// kvc8_bf16.cu -- the bf16 paged KV cache without quantisation: store new
// tokens into pages and gather pages back into contiguous rows.  This is the
// int8 path's sibling MojoStorePagedKVCache ("Mojo Opset" README, "Op List",
// KVCache rows; mojo_opset pull request #379, "feat: [MLU] add mlu
// experimental ops; fix post norm bug", first review pass, "Must fix" on the
// cu_q_lens check that this sibling performs).  Same layout and slot mapping as
// the int8 path, with bf16 rows [NB][H][bs][D] and no codec: both kernels are
// pure data movement.
#include "kvc8_internal.cuh"

namespace kvc8 {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kGatherThreads = 256;

// Slot of new token t (warp-uniform): physical block and in-block slot, or a
// device error code.
struct Slot {
    int32_t blk;
    int64_t slot;
    int32_t err;
};

__device__ __forceinline__ Slot token_slot(const StoreBf16Args &a, int64_t t, int lane) {
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int bs = a.g.block_size;
    Slot r{0, 0, 0};
    int b;
    int64_t i_in_seq, ctx;
    bool bad_len = false;
    if (a.cu_q_lens != nullptr) {
        const TokenSeq ts = seq_ctx_of_token(a.cu_q_lens, a.context_kv_lens, B, t, lane);
        b = ts.b;
        ctx = ts.ctx;
        i_in_seq = t - ts.first;
        bad_len = !(ts.first <= t && t < ts.next);
    } else {
        b = (int)t;
        i_in_seq = 0;
        ctx = ld_nc_s32(a.context_kv_lens + b);
    }
    const int64_t pos = ctx + i_in_seq;
    const int64_t lb = pos / bs;
    if (bad_len || ctx < 0) {
        r.err = KVC8_DEV_BAD_LENGTH;
    } else if (lb >= MB) {
        r.err = KVC8_DEV_POS_BEYOND_TABLE;
    } else {
        r.blk = ld_nc_s32(a.block_table + (int64_t)b * MB + lb);
        if (r.blk < 0 || r.blk >= NB) r.err = KVC8_DEV_BAD_BLOCK_ID;
    }
    r.slot = pos - lb * bs;
    return r;
}

// One warp per token: the lanes move the token's 2H rows of D bf16 values in
// chunks requested before the slot lookup, so that the loads overlap it.  WIDE
// (inputs and caches 32-byte aligned, input strides multiples of 16 values):
// 32-byte chunks, one 256-bit load and store each, 4 in flight per lane;
// otherwise 16-byte chunks, 8 in flight per lane.
template <bool WIDE>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
store_bf16_kernel(const StoreBf16Args a) {
    constexpr int CW = WIDE ? 16 : 8;   // values per chunk
    constexpr int K = WIDE ? 4 : 8;     // chunks in flight per lane
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int CPR = D / CW;             // chunks per row
    const int nch = 2 * H * CPR;        // chunks per token
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
    for (int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); t < a.num_tokens;
         t += nwarps) {
        Slot sl{0, 0, 0};
        for (int c0 = 0; c0 < nch; c0 += 32 * K) {
            uint4 v[K][WIDE ? 2 : 1];
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int c = c0 + k * 32 + lane;
                if (c < nch) {
                    const int row = c / CPR, col = c - row * CPR;
                    const int kv = row >= H, h = row - kv * H;
                    const uint16_t *src = (kv ? a.v_states : a.k_states) + t * a.x_tok_stride +
                                          (int64_t)h * a.x_head_stride + col * CW;
                    if (WIDE) {
                        asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                            : "=r"(v[k][0].x), "=r"(v[k][0].y), "=r"(v[k][0].z), "=r"(v[k][0].w),
                              "=r"(v[k][WIDE ? 1 : 0].x), "=r"(v[k][WIDE ? 1 : 0].y),
                              "=r"(v[k][WIDE ? 1 : 0].z), "=r"(v[k][WIDE ? 1 : 0].w)
                            : "l"(src));
                    } else {
                        v[k][0] = ld_stream_16(src);
                    }
                }
            }
            if (c0 == 0) {
                sl = token_slot(a, t, lane);
                if (sl.err != 0 && lane == 0) report(a.dev_error, sl.err);
            }
            if (sl.err != 0) break;  // warp-uniform: skip the token
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int c = c0 + k * 32 + lane;
                if (c < nch) {
                    const int row = c / CPR, col = c - row * CPR;
                    const int kv = row >= H, h = row - kv * H;
                    uint16_t *dst = (kv ? a.v_cache : a.k_cache) +
                                    ((((int64_t)sl.blk * H + h) * bs + sl.slot) * D + col * CW);
                    if (WIDE) {
                        asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst),
                                     "r"(v[k][0].x), "r"(v[k][0].y), "r"(v[k][0].z), "r"(v[k][0].w),
                                     "r"(v[k][WIDE ? 1 : 0].x), "r"(v[k][WIDE ? 1 : 0].y),
                                     "r"(v[k][WIDE ? 1 : 0].z), "r"(v[k][WIDE ? 1 : 0].w)
                                     : "memory");
                    } else {
                        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(v[k][0].x),
                                     "r"(v[k][0].y), "r"(v[k][0].z), "r"(v[k][0].w)
                                     : "memory");
                    }
                }
            }
        }
    }
}

// Largest b in [0, B] with ts[b] <= tile.
__device__ __forceinline__ int seq_of_tile(const int32_t *ts, int B, int64_t tile) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((int64_t)ts[mid] <= tile) lo = mid; else hi = mid;
    }
    return lo;
}

// 32 bytes from the cache, streamed past L1: one 256-bit load when WIDE
// (32-byte aligned), else two 128-bit loads.
template <bool WIDE>
__device__ __forceinline__ void load_chunk32(const uint16_t *p, uint4 &lo, uint4 &hi) {
    if (WIDE) {
        asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
              "=r"(hi.z), "=r"(hi.w)
            : "l"(p));
    } else {
        lo = ld_stream_16(p);
        hi = ld_stream_16(p + 8);
    }
}

// Work item: one tile (sequence, logical block) and a pair of its (K|V, head)
// slabs, handed out by the plan's atomic counter, as in the int8 gather.  Each
// thread moves one 32-byte chunk (16 values) per slab per round: one 256-bit
// load and store each when the cache, the outputs and their strides are
// 32-byte aligned (WIDE), else two 128-bit ones.
template <bool WIDE>
__global__ void __launch_bounds__(kGatherThreads)
gather_bf16_kernel(const GatherBf16Args a) {
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int CPR = D >> 4;  // 16-value chunks per row
    __shared__ long long s_item;

    pdl_wait_prior_grid();
    const char *plan = static_cast<const char *>(a.plan);
    const PlanHeader *hdr = reinterpret_cast<const PlanHeader *>(plan);
    const int64_t *off = reinterpret_cast<const int64_t *>(plan + plan_offsets_at(B));
    const int32_t *ts = reinterpret_cast<const int32_t *>(plan + plan_tile_start_at(B));
    unsigned long long *counter =
        reinterpret_cast<unsigned long long *>(const_cast<int64_t *>(&hdr->work_counter));
    const int64_t items = hdr->total_tiles * H;

    int64_t item = blockIdx.x;
    while (item < items) {
        long long next = 0;
        if (threadIdx.x == 0) next = (long long)atomicAdd(counter, 1ull) + gridDim.x;
        const int64_t tile = item / H;
        const int r2 = (int)(item - tile * H);
        const int b = seq_of_tile(ts, B, tile);
        const int64_t j = tile - ts[b];
        const int64_t len = ld_nc_s32(a.context_lengths + b);
        const int nvalid = (int)min((int64_t)bs, len - j * bs);
        const int32_t blk = ld_nc_s32(a.block_table + (int64_t)b * MB + j);
        const int64_t row0 = off[b] + j * bs;
        bool ok = true;
        if (blk < 0 || blk >= NB) {
            if (threadIdx.x == 0) report(a.dev_error, KVC8_DEV_BAD_BLOCK_ID);
            ok = false;
        } else if (row0 < 0 || row0 + nvalid > a.out_rows) {
            if (threadIdx.x == 0) report(a.dev_error, KVC8_DEV_OUT_ROW_RANGE);
            ok = false;
        }
        if (ok) {
            const int nch = nvalid * CPR;
            for (int c0 = 0; c0 < nch; c0 += kGatherThreads) {
                const int c = c0 + threadIdx.x;
                uint4 lo[2], hi[2];
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int u = 2 * r2 + sl;
                    const int kv = u >= H, h = u - kv * H;
                    if (c < nch) {
                        const uint16_t *src = (kv ? a.v_cache : a.k_cache) +
                                              (((int64_t)blk * H + h) * bs * D + (int64_t)c * 16);
                        load_chunk32<WIDE>(src, lo[sl], hi[sl]);
                    }
                }
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int u = 2 * r2 + sl;
                    const int kv = u >= H, h = u - kv * H;
                    if (c < nch) {
                        const int row = c / CPR, col = c - row * CPR;
                        uint16_t *dst = (kv ? a.v_out : a.k_out) + (row0 + row) * a.out_tok_stride +
                                        (int64_t)h * a.out_head_stride + col * 16;
                        if (WIDE) {
                            st_stream_32(dst, lo[sl], hi[sl]);
                        } else {
                            st_stream_16(dst, lo[sl].x, lo[sl].y, lo[sl].z, lo[sl].w);
                            st_stream_16(dst + 8, hi[sl].x, hi[sl].y, hi[sl].z, hi[sl].w);
                        }
                    }
                }
            }
        }
        if (threadIdx.x == 0) s_item = next;
        __syncthreads();
        item = s_item;
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_store_bf16(const StoreBf16Args &a, cudaStream_t stream) {
    if (a.num_tokens <= 0) return cudaSuccess;
    auto a32 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; };
    const bool wide = a32(a.k_states) && a32(a.v_states) && a32(a.k_cache) && a32(a.v_cache) &&
                      a.x_tok_stride % 16 == 0 && a.x_head_stride % 16 == 0;
    auto kern = wide ? store_bf16_kernel<true> : store_bf16_kernel<false>;
    static OccupancySlots slots[2];
    int occ = 0;
    const cudaError_t e = occupancy(slots[wide], kern, kWarpsPerCta * 32, 0, &occ);
    if (e != cudaSuccess) return e;
    const int64_t need = (a.num_tokens + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = (int64_t)sm_count() * occ;
    kern<<<(int)(need < cap ? need : cap), kWarpsPerCta * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gather_bf16(const GatherBf16Args &a, bool use_pdl, cudaStream_t stream) {
    auto a32 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; };
    const bool wide = a32(a.k_cache) && a32(a.v_cache) && a32(a.k_out) && a32(a.v_out) &&
                      a.out_tok_stride % 16 == 0 && a.out_head_stride % 16 == 0;
    auto kern = wide ? gather_bf16_kernel<true> : gather_bf16_kernel<false>;
    static OccupancySlots slots[2];
    int occ = 0;
    const cudaError_t e = occupancy(slots[wide], kern, kGatherThreads, 0, &occ);
    if (e != cudaSuccess) return e;
    const int64_t max_items = (int64_t)a.g.num_seqs * a.g.max_blocks_per_seq * a.g.kv_heads;
    const int64_t cap = (int64_t)sm_count() * occ;
    const int grid = (int)(max_items < cap ? max_items : cap);
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGatherThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace kvc8
