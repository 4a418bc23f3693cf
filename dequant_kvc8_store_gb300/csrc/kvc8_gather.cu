// kvc8_gather.cu -- gather each sequence's pages and dequantise them into
// contiguous bf16 rows (MojoDequantFromPagedKVCache in mojo_opset pull request
// #379, "feat: [MLU] add mlu experimental ops; fix post norm bug"), plus the
// plan kernel that replaces the pages' host-side offset cumsum and per-batch
// .item() loop.
//
// Work decomposition.  A tile is one logical block j of one sequence b; a unit
// is one (tile, K|V, kv head): bs rows of D int8 codes, contiguous in the
// cache ([blk][h][0:bs][0:D]), that land as bs rows of D bf16 values at
// out[(off_b + j*bs + slot)][h][:] -- a 2*D-byte contiguous segment per row.
// Units are numbered tile-major and dealt round-robin to a persistent grid, so
// every CTA streams equal-sized units regardless of how ragged the sequence
// lengths are.  Inside a unit each thread moves 16-byte chunks (16 codes ->
// 32 bytes of bf16), four chunks in flight per thread.  Source reads and
// destination writes are both fully coalesced without a shared-memory
// transpose, because the transpose [heads, tokens, dim] -> [tokens, heads, dim]
// only permutes whole D-element rows.
//
// Arithmetic per element: c = int8 code, exactly recovered as float by the
// bias trick (0x4B000000 | (c + 128)) - (2^23 + 128); v = c * s in one IEEE
// fp32 multiply; bf16 by cvt.rn (round to nearest even).
#include "kvc8_internal.cuh"

namespace kvc8 {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kGatherThreads = 256;
constexpr int kUnroll = 4;

// ---------------------------------------------------------------------------
// Plan: one CTA scans context_lengths (int64 running sum for the offsets and an
// int32 running count of tiles).

template <typename T>
__device__ T block_inclusive_scan(T v, T *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        T t = lane < nw ? warp_tot[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T n = __shfl_up_sync(0xFFFFFFFFu, t, o);
            if (lane >= o) t += n;
        }
        if (lane < nw) warp_tot[lane] = t;  // inclusive prefix of warp totals
    }
    __syncthreads();
    if (warp > 0) v += warp_tot[warp - 1];
    return v;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const kvc8_geom g, const int32_t *__restrict__ lens,
            const int64_t *__restrict__ given_off, int64_t *__restrict__ offsets_out,
            char *__restrict__ plan, int32_t *__restrict__ dev_error) {
    // The gather may start launching now; it waits for this grid to finish
    // (griddepcontrol.wait) before it reads the plan.
    pdl_launch_dependents();
    __shared__ int64_t tot64[32];
    __shared__ int32_t tot32[32];
    __shared__ int64_t carry_len_s;
    __shared__ int32_t carry_tiles_s;
    const int B = g.num_seqs, bs = g.block_size, MB = g.max_blocks_per_seq;
    int64_t *off = reinterpret_cast<int64_t *>(plan + plan_offsets_at(B));
    int32_t *ts = reinterpret_cast<int32_t *>(plan + plan_tile_start_at(B));
    if (threadIdx.x == 0) {
        carry_len_s = 0;
        carry_tiles_s = 0;
    }
    __syncthreads();
    for (int base = 0; base < B; base += kPlanThreads) {
        const int i = base + threadIdx.x;
        int64_t len = 0;
        int32_t tiles = 0;
        if (i < B) {
            len = lens[i];
            if (len < 0) {
                report(dev_error, KVC8_DEV_BAD_LENGTH);
                len = 0;
            }
            int64_t t64 = (len + bs - 1) / bs;
            if (t64 > MB) {
                report(dev_error, KVC8_DEV_POS_BEYOND_TABLE);
                t64 = MB;
            }
            tiles = (int32_t)t64;
        }
        const int64_t carry_len = carry_len_s;
        const int32_t carry_tiles = carry_tiles_s;
        const int64_t inc_len = block_inclusive_scan<int64_t>(len, tot64);
        const int32_t inc_tiles = block_inclusive_scan<int32_t>(tiles, tot32);
        if (i < B) {
            const int64_t o = given_off != nullptr ? given_off[i] : carry_len + inc_len - len;
            off[i] = o;
            ts[i] = carry_tiles + inc_tiles - tiles;
            if (offsets_out != nullptr) offsets_out[i] = o;
        }
        __syncthreads();
        if (threadIdx.x == kPlanThreads - 1) {
            carry_len_s = carry_len + inc_len;
            carry_tiles_s = carry_tiles + inc_tiles;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        ts[B] = carry_tiles_s;
        reinterpret_cast<PlanHeader *>(plan)->total_tiles = carry_tiles_s;
    }
}

// ---------------------------------------------------------------------------
// Gather.

// Largest b in [0, B] with ts[b] <= tile (ts[0] = 0 <= tile).
__device__ __forceinline__ int seq_of_tile(const int32_t *ts, int B, int64_t tile) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((int64_t)ts[mid] <= tile) lo = mid; else hi = mid;
    }
    return lo;
}

// Four int8 codes -> four exact floats.
__device__ __forceinline__ void codes_to_f32(uint32_t w, float f[4]) {
    const uint32_t wb = w ^ 0x80808080u;  // c + 128 per byte
    const float bias = 8388736.0f;        // 2^23 + 128
    f[0] = __fsub_rn(__uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7440)), bias);
    f[1] = __fsub_rn(__uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7441)), bias);
    f[2] = __fsub_rn(__uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7442)), bias);
    f[3] = __fsub_rn(__uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7443)), bias);
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 16 codes with one scale each (sc[e] for element e) -> 8 packed bf16 pairs.
__device__ __forceinline__ void dequant16(const uint4 v, const float *sc, uint32_t out[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float f[4];
        codes_to_f32(w[j], f);
        const float p0 = __fmul_rn(f[0], sc[4 * j + 0]);
        const float p1 = __fmul_rn(f[1], sc[4 * j + 1]);
        const float p2 = __fmul_rn(f[2], sc[4 * j + 2]);
        const float p3 = __fmul_rn(f[3], sc[4 * j + 3]);
        out[2 * j] = bf16x2_rn(p0, p1);
        out[2 * j + 1] = bf16x2_rn(p2, p3);
    }
}

template <int MODE, bool WIDE>
__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(const GatherArgs a) {
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int CPR = D >> 4;  // 16-code chunks per row
    const bool col_fixed = (kGatherThreads % CPR) == 0;

    pdl_wait_prior_grid();
    const char *plan = static_cast<const char *>(a.plan);
    const int64_t *off = reinterpret_cast<const int64_t *>(plan + plan_offsets_at(B));
    const int32_t *ts = reinterpret_cast<const int32_t *>(plan + plan_tile_start_at(B));
    const int64_t total_tiles = reinterpret_cast<const PlanHeader *>(plan)->total_tiles;
    const int64_t units = total_tiles * 2 * H;

    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t tile = u / (2 * H);
        const int r = (int)(u - tile * 2 * H);
        const int kv = r >= H;
        const int h = r - kv * H;
        const int b = seq_of_tile(ts, B, tile);
        const int64_t j = tile - ts[b];
        int64_t len = ld_nc_s32(a.context_lengths + b);
        const int nvalid = (int)min((int64_t)bs, len - j * bs);
        const int32_t blk = ld_nc_s32(a.block_table + (int64_t)b * MB + j);
        const int64_t row0 = off[b] + j * bs;
        if (blk < 0 || blk >= NB) {
            if (threadIdx.x == 0) report(a.dev_error, KVC8_DEV_BAD_BLOCK_ID);
            continue;
        }
        if (row0 < 0 || row0 + nvalid > a.out_rows) {
            if (threadIdx.x == 0) report(a.dev_error, KVC8_DEV_OUT_ROW_RANGE);
            continue;
        }
        const int8_t *src = (kv ? a.v_cache : a.k_cache) + ((int64_t)blk * H + h) * bs * D;
        const float *scl = kv ? a.v_scale : a.k_scale;
        uint16_t *dst = (kv ? a.v_out : a.k_out) + row0 * a.out_tok_stride +
                        (int64_t)h * a.out_head_stride;
        const float *row_scale = scl + ((int64_t)blk * H + h) * bs;  // mode 0
        const float *chan_scale = scl + (int64_t)h * D;               // mode 1

        float fixed_sc[16];
        if (MODE == 1 && col_fixed) {
            const int col = threadIdx.x % CPR;
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 s4 = __ldg(reinterpret_cast<const float4 *>(chan_scale + col * 16 + e));
                fixed_sc[e] = s4.x; fixed_sc[e + 1] = s4.y; fixed_sc[e + 2] = s4.z; fixed_sc[e + 3] = s4.w;
            }
        }

        const int nchunks = nvalid * CPR;
        for (int c0 = 0; c0 < nchunks; c0 += kGatherThreads * kUnroll) {
            uint4 v[kUnroll];
            float s[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int c = c0 + k * kGatherThreads + threadIdx.x;
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                s[k] = 0.0f;
                if (c < nchunks) {
                    v[k] = ld_stream_16(src + (int64_t)c * 16);
                    if (MODE == 0) s[k] = ld_nc_f32(row_scale + c / CPR);
                }
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int c = c0 + k * kGatherThreads + threadIdx.x;
                if (c >= nchunks) continue;
                const int row = c / CPR;
                const int col = c - row * CPR;
                float sc[16];
                if (MODE == 0) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) sc[e] = s[k];
                } else if (col_fixed) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) sc[e] = fixed_sc[e];
                } else {
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const float4 s4 = __ldg(reinterpret_cast<const float4 *>(chan_scale + col * 16 + e));
                        sc[e] = s4.x; sc[e + 1] = s4.y; sc[e + 2] = s4.z; sc[e + 3] = s4.w;
                    }
                }
                uint32_t o[8];
                dequant16(v[k], sc, o);
                uint16_t *p = dst + (int64_t)row * a.out_tok_stride + col * 16;
                if (WIDE) {
                    st_stream_32(p, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
                } else {
                    st_stream_16(p, o[0], o[1], o[2], o[3]);
                    st_stream_16(p + 8, o[4], o[5], o[6], o[7]);
                }
            }
        }
    }
}

template <int MODE, bool WIDE>
cudaError_t launch_gather_variant(const GatherArgs &a, bool use_pdl, cudaStream_t stream) {
    auto kern = gather_kernel<MODE, WIDE>;
    static int occ_cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int occ = dev < 64 ? occ_cached[dev] : 0;
    if (occ == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kGatherThreads, 0);
        if (e != cudaSuccess) return e;
        if (occ < 1) occ = 1;
        if (dev < 64) occ_cached[dev] = occ;
    }
    const int64_t max_units = (int64_t)a.g.num_seqs * a.g.max_blocks_per_seq * 2 * a.g.kv_heads;
    const int64_t cap = (int64_t)sm_count() * occ;
    const int grid = (int)(max_units < cap ? max_units : cap);
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGatherThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t launch_plan(const kvc8_geom &g, const int32_t *context_lengths,
                        const int64_t *context_seq_offset, int64_t *offsets_out, void *plan,
                        int32_t *dev_error, cudaStream_t stream) {
    plan_kernel<<<1, kPlanThreads, 0, stream>>>(g, context_lengths, context_seq_offset,
                                                offsets_out, static_cast<char *>(plan), dev_error);
    return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs &a, bool use_pdl, cudaStream_t stream) {
    const uintptr_t k = reinterpret_cast<uintptr_t>(a.k_out);
    const uintptr_t v = reinterpret_cast<uintptr_t>(a.v_out);
    const bool wide = (k % 32 == 0) && (v % 32 == 0) && (a.out_tok_stride % 16 == 0) &&
                      (a.out_head_stride % 16 == 0);
    if (a.g.quant_mode == 0)
        return wide ? launch_gather_variant<0, true>(a, use_pdl, stream)
                    : launch_gather_variant<0, false>(a, use_pdl, stream);
    return wide ? launch_gather_variant<1, true>(a, use_pdl, stream)
                : launch_gather_variant<1, false>(a, use_pdl, stream);
}

}  // namespace kvc8
