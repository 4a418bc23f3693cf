// kvc8_gather.cu -- gather each sequence's pages and dequantise them into
// contiguous bf16 rows (MojoDequantFromPagedKVCache in mojo_opset pull request
// #379, "feat: [MLU] add mlu experimental ops; fix post norm bug"), plus the
// plan kernel that replaces the pages' host-side offset cumsum and per-batch
// .item() loop.
//
// Work decomposition.  A tile is one logical block j of one sequence b; a slab
// is one (tile, K|V, kv head): bs rows of D int8 codes, contiguous in the
// cache ([blk][h][0:bs][0:D]), that land as bs rows of D bf16 values at
// out[(off_b + j*bs + slot)][h][:] -- a 2*D-byte contiguous segment per row.
// A work item is a tile and a pair of its slabs; items are numbered tile-major
// and handed to a persistent grid through an atomic counter, so every CTA keeps
// streaming equal-sized items however ragged the sequence lengths are.  Inside
// an item each thread moves chunks of 32 codes (256-bit loads; 16 when D is not
// a multiple of 32) -> 64 bytes of bf16, one chunk per slab per round, so two
// loads are in flight per thread and the low register count keeps many CTAs
// resident.  Source reads and destination writes
// are both fully coalesced without a shared-memory transpose, because the
// transpose [heads, tokens, dim] -> [tokens, heads, dim] only permutes whole
// D-element rows.
//
// Arithmetic per element: c = int8 code, exactly recovered as float by the
// bias trick (0x4B000000 | (c + 128)) - (2^23 + 128); v = c * s in one IEEE
// fp32 multiply; bf16 by cvt.rn (round to nearest even).
#include "kvc8_internal.cuh"

namespace kvc8 {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kGatherThreads = 256;

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
            char *__restrict__ plan, int32_t *__restrict__ dev_error,
            const int32_t *__restrict__ cu_q, int q_mode, int32_t *__restrict__ spans_out) {
    // lens: the positions cached per sequence.  q_mode 0: the output rows of
    // a sequence are exactly those; 1: an append adds cu_q[b+1] - cu_q[b]
    // rows after them (the fused append computes them, so tiles cover only
    // lens); 2: as 1 with one row; 3 and 4: as 1 and 2 with the new tokens
    // already in the cache, so tiles cover lens + new.  spans_out, if given,
    // receives lens + new per sequence.
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
    for (int base = 0; base < B; base += blockDim.x) {
        const int i = base + threadIdx.x;
        int64_t len = 0, span = 0;  // span: output rows of the sequence
        int32_t tiles = 0;
        if (i < B) {
            len = lens[i];
            if (len < 0) {
                report(dev_error, KVC8_DEV_BAD_LENGTH);
                len = 0;
            }
            int64_t q = 0;
            if (q_mode == 1 || q_mode == 3) {
                q = (int64_t)cu_q[i + 1] - cu_q[i];
                if (q < 0) {
                    report(dev_error, KVC8_DEV_BAD_LENGTH);
                    q = 0;
                }
            } else if (q_mode == 2 || q_mode == 4) {
                q = 1;
            }
            span = len + q;
            if (spans_out != nullptr) spans_out[i] = (int32_t)min(span, (int64_t)INT32_MAX);
            if (q_mode >= 3) len = span;  // the gather reads every position
            int64_t t64 = (len + bs - 1) / bs;
            if (t64 > MB) {
                report(dev_error, KVC8_DEV_POS_BEYOND_TABLE);
                t64 = MB;
            }
            tiles = (int32_t)t64;
        }
        const int64_t carry_len = carry_len_s;
        const int32_t carry_tiles = carry_tiles_s;
        const int64_t inc_len = block_inclusive_scan<int64_t>(span, tot64);
        const int32_t inc_tiles = block_inclusive_scan<int32_t>(tiles, tot32);
        if (i < B) {
            const int64_t o = given_off != nullptr ? given_off[i] : carry_len + inc_len - span;
            off[i] = o;
            ts[i] = carry_tiles + inc_tiles - tiles;
            if (offsets_out != nullptr) offsets_out[i] = o;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) {
            carry_len_s = carry_len + inc_len;
            carry_tiles_s = carry_tiles + inc_tiles;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        ts[B] = carry_tiles_s;
        PlanHeader *hdr = reinterpret_cast<PlanHeader *>(plan);
        hdr->total_tiles = carry_tiles_s;
        hdr->work_counter = 0;  // the gather's work distribution starts afresh
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

// Four int8 codes -> four exact floats: (0x4B000000 | (c + 128)) - (2^23 + 128).
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

// One chunk of CH codes (CH/4 words) -> CH/2 packed bf16 pairs.  Modes 0 and
// 2: one scale for the chunk (the row's, or the block's); mode 1: per-channel
// scales sc[0..CH).
template <int CH, int MODE>
__device__ __forceinline__ void dequant_chunk(const uint32_t *w, float s, const float *sc,
                                              uint32_t *o) {
#pragma unroll
    for (int j = 0; j < CH / 4; ++j) {
        float f[4];
        codes_to_f32(w[j], f);
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = __fmul_rn(f[e], MODE != 1 ? s : sc[4 * j + e]);
        o[2 * j] = bf16x2_rn(p[0], p[1]);
        o[2 * j + 1] = bf16x2_rn(p[2], p[3]);
    }
}

template <int CH>
__device__ __forceinline__ void load_chunk(const int8_t *p, uint32_t *w) {
    if (CH == 32) {
        asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
              "=r"(w[6]), "=r"(w[7])
            : "l"(p));
    } else {
        const uint4 v = ld_stream_16(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
}

template <int CH, bool WIDE>
__device__ __forceinline__ void store_chunk(uint16_t *p, const uint32_t *o) {
#pragma unroll
    for (int q = 0; q < CH / 16; ++q) {
        if (WIDE) {
            st_stream_32(p + 16 * q, make_uint4(o[8 * q], o[8 * q + 1], o[8 * q + 2], o[8 * q + 3]),
                         make_uint4(o[8 * q + 4], o[8 * q + 5], o[8 * q + 6], o[8 * q + 7]));
        } else {
            st_stream_16(p + 16 * q, o[8 * q], o[8 * q + 1], o[8 * q + 2], o[8 * q + 3]);
            st_stream_16(p + 16 * q + 8, o[8 * q + 4], o[8 * q + 5], o[8 * q + 6], o[8 * q + 7]);
        }
    }
}

// Append part of the fused append + gather: row r = (token t, K|V, head h) of
// the new tokens, one per warp.  Lane l holds values [4l, 4l + 4) of each
// 128-value chunk of the row (two chunks when D = 256).  The codes follow the
// definition directly -- s = fl(amax / 127) (mode 0) or the static scale
// (per channel, mode 1; per block, mode 2),
// q = clamp(rne(fl(x / s)), -127, 127), 0 when s = 0 -- because an append is a
// handful of rows per sequence and its time is latency.  The output values are
// formed exactly as the gather forms them from the cache: fl(float(q) * s),
// rounded to bf16 (RNE).
template <int MODE, int CH>
__device__ __forceinline__ void append_row(const GatherArgs &a, const AppendArgs &p, int64_t r,
                                           const int64_t *off, const float *s_tab) {
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int lane = threadIdx.x & 31;
    if (r >= p.num_tokens * 2 * H) return;  // warp-uniform
    const int64_t t = (int64_t)((uint32_t)r / (uint32_t)(2 * H));  // r < 2^31
    const int u = (int)(r - t * 2 * H);
    const int kv = u >= H, h = u - kv * H;
    const uint16_t *src = (kv ? p.v_states : p.k_states) + t * p.x_tok_stride +
                          (int64_t)h * p.x_head_stride;
    uint32_t x[2][2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int d0 = c * 128 + lane * 4;
        x[c][0] = x[c][1] = 0u;
        if (d0 < D)
            asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                : "=r"(x[c][0]), "=r"(x[c][1])
                : "l"(src + d0));
    }

    // slot of token t (warp-uniform)
    int b;
    int64_t i_in_seq, ctx;
    bool bad_len = false;
    if (p.cu_q_lens != nullptr) {
        const TokenSeq ts = seq_ctx_of_token(p.cu_q_lens, p.context_kv_lens, B, t, lane);
        b = ts.b;
        ctx = ts.ctx;
        i_in_seq = t - ts.first;
        bad_len = !(ts.first <= t && t < ts.next);
    } else {
        b = (int)t;
        i_in_seq = 0;
        ctx = ld_nc_s32(p.context_kv_lens + b);
    }
    const int64_t pos = ctx + i_in_seq;
    // pos < 2^32: a 32-bit division (ctx and the token index are below 2^31)
    const int64_t lb = pos >= 0 ? (int64_t)((uint32_t)pos / (uint32_t)bs) : -1;
    int32_t err = 0, blk = 0;
    if (bad_len || ctx < 0) {
        err = KVC8_DEV_BAD_LENGTH;
    } else if (lb >= MB) {
        err = KVC8_DEV_POS_BEYOND_TABLE;
    } else {
        blk = ld_nc_s32(a.block_table + (int64_t)b * MB + lb);
        if (blk < 0 || blk >= NB) err = KVC8_DEV_BAD_BLOCK_ID;
    }
    if (err != 0) {
        if (lane == 0) report(a.dev_error, err);
        return;
    }
    const int64_t row = ((int64_t)blk * H + h) * bs + (pos - lb * bs);
    const int64_t orow = off[b] + pos;
    const bool out_ok = orow >= 0 && orow < a.out_rows;
    if (!out_ok && lane == 0) report(a.dev_error, KVC8_DEV_OUT_ROW_RANGE);

    float s = 0.0f;  // modes 0 and 2: the row scale
    if (MODE == 2) s = ld_nc_f32((kv ? p.v_scale : p.k_scale) + (int64_t)blk * H + h);
    if (MODE == 0) {
        uint32_t m = 0u;  // |x| as bf16 bits: integer order = magnitude order
#pragma unroll
        for (int c = 0; c < 2; ++c)
            m = max(m, max(max(x[c][0] & 0x7FFFu, (x[c][0] >> 16) & 0x7FFFu),
                           max(x[c][1] & 0x7FFFu, (x[c][1] >> 16) & 0x7FFFu)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        s = __fdiv_rn(__uint_as_float(m << 16), 127.0f);
        if (lane == 0) (kv ? p.v_scale : p.k_scale)[row] = s;
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int d0 = c * 128 + lane * 4;
        if (d0 >= D) continue;
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (MODE != 1) {
                sc[e] = s;
            } else {
                constexpr int SPAD = CH + 4;
                const int d = d0 + e;
                sc[e] = s_tab[((kv * H + h) * (D / CH) + d / CH) * SPAD + d % CH];
            }
        }
        int q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t w = x[c][e >> 1];
            const float v = __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
            q[e] = sc[e] == 0.0f ? 0 : min(127, max(-127, __float2int_rn(__fdiv_rn(v, sc[e]))));
        }
        const uint32_t codes = __byte_perm(__byte_perm((uint32_t)q[0], (uint32_t)q[1], 0x0040),
                                           __byte_perm((uint32_t)q[2], (uint32_t)q[3], 0x0040),
                                           0x5410);
        asm volatile("st.global.u32 [%0], %1;" ::"l"((kv ? p.v_cache : p.k_cache) + row * D + d0),
                     "r"(codes)
                     : "memory");
        if (out_ok) {
            const uint32_t o0 = bf16x2_rn(__fmul_rn((float)q[0], sc[0]), __fmul_rn((float)q[1], sc[1]));
            const uint32_t o1 = bf16x2_rn(__fmul_rn((float)q[2], sc[2]), __fmul_rn((float)q[3], sc[3]));
            asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(
                             (kv ? a.v_out : a.k_out) + orow * a.out_tok_stride +
                             (int64_t)h * a.out_head_stride + d0),
                         "r"(o0), "r"(o1)
                         : "memory");
        }
    }
}

// A work item is one tile (sequence b, logical block j) and a pair of (K|V,
// head) slabs: units 2r and 2r+1 of the tile's 2H units, so both slabs share
// the tile's metadata.  Items are handed out by an atomic counter in the plan.
// APPEND: the fused append + gather; items [0, p.items) are append items
// (kAppendRowsPerItem rows each), the gather items follow.
template <int MODE, int CH, bool WIDE, bool APPEND>
__global__ void __launch_bounds__(kGatherThreads, APPEND ? (MODE == 1 ? 4 : 6) : 0)
gather_kernel(const GatherArgs a, const AppendArgs p) {
    constexpr int W = CH / 4;  // words per chunk
    constexpr int PER = 1;     // chunks per slab per thread per round
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int CPR = D / CH;  // chunks per row

    // Mode 1: static scales [2][H][D] as chunks of CH values padded by 4
    // floats, so the chunk columns of a warp fall in different banks.
    constexpr int SPAD = CH + 4;
    extern __shared__ float s_tab[];
    if (MODE == 1) {
        for (int i = threadIdx.x; i < 2 * H * D; i += blockDim.x) {
            const int row = i / D, d = i - row * D;
            s_tab[(row * CPR + d / CH) * SPAD + d % CH] =
                i < H * D ? ld_nc_f32(a.k_scale + i) : ld_nc_f32(a.v_scale + (i - H * D));
        }
        __syncthreads();
    }
    __shared__ long long s_item;

    pdl_wait_prior_grid();  // the plan (and its counter reset) is complete
    const char *plan = static_cast<const char *>(a.plan);
    const PlanHeader *hdr = reinterpret_cast<const PlanHeader *>(plan);
    const int64_t *off = reinterpret_cast<const int64_t *>(plan + plan_offsets_at(B));
    const int32_t *ts_g = reinterpret_cast<const int32_t *>(plan + plan_tile_start_at(B));
    // tile_start in shared memory when it fits: each item's sequence is then
    // found without a chain of dependent global loads
    constexpr int kTsShared = 1024;
    __shared__ int32_t s_ts[kTsShared];
    const int32_t *ts = ts_g;
    if (B + 1 <= kTsShared) {
        for (int i = threadIdx.x; i <= B; i += blockDim.x) s_ts[i] = ts_g[i];
        __syncthreads();
        ts = s_ts;
    }
    unsigned long long *counter =
        reinterpret_cast<unsigned long long *>(const_cast<int64_t *>(&hdr->work_counter));
    const int64_t items = hdr->total_tiles * H + (APPEND ? p.items : 0);

    int64_t item = blockIdx.x;
    if (APPEND) {
        // Items come in increasing order, so once a CTA draws a gather item it
        // never draws an append item again: the append loop runs first.
        while (item < p.items) {
            long long next = 0;
            if (threadIdx.x == 0) next = (long long)atomicAdd(counter, 1ull) + gridDim.x;
            append_row<MODE, CH>(a, p, item * kAppendRowsPerItem + (threadIdx.x >> 5), off, s_tab);
            if (threadIdx.x == 0) s_item = next;
            __syncthreads();
            item = s_item;
            __syncthreads();
        }
    }
    const int64_t first_gather = APPEND ? p.items : 0;
    while (item < items) {
        long long next = 0;
        if (threadIdx.x == 0) next = (long long)atomicAdd(counter, 1ull) + gridDim.x;
        const int64_t gitem = item - first_gather;

        // 32-bit division in append mode (the host keeps its item counts below
        // 2^31); a 64-bit division there raised the kernel's register count
        const int64_t tile = APPEND ? (int64_t)((uint32_t)gitem / (uint32_t)H) : gitem / H;
        const int r2 = (int)(gitem - tile * H);
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
            const int8_t *src[2];
            const float *rsc[2];
            const float *csc[2];
            uint16_t *dst[2];
            float sblk[2];  // mode 2: the slab's block scale
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                const int u = 2 * r2 + sl;
                const int kv = u >= H;
                const int h = u - kv * H;
                src[sl] = (kv ? a.v_cache : a.k_cache) + ((int64_t)blk * H + h) * bs * D;
                rsc[sl] = (kv ? a.v_scale : a.k_scale) + ((int64_t)blk * H + h) * bs;
                sblk[sl] = MODE == 2 ? ld_nc_f32((kv ? a.v_scale : a.k_scale) + (int64_t)blk * H + h)
                                     : 0.0f;
                csc[sl] = s_tab + (kv * H + h) * CPR * SPAD;
                dst[sl] = (kv ? a.v_out : a.k_out) + row0 * a.out_tok_stride +
                          (int64_t)h * a.out_head_stride;
            }
            const int nch = nvalid * CPR;  // chunks per slab
            for (int c0 = 0; c0 < nch; c0 += kGatherThreads * PER) {
                uint32_t w[2][PER][W];
                float s[2][PER];
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
#pragma unroll
                    for (int k = 0; k < PER; ++k) {
                        const int c = c0 + k * kGatherThreads + threadIdx.x;
#pragma unroll
                        for (int i = 0; i < W; ++i) w[sl][k][i] = 0u;
                        s[sl][k] = 0.0f;
                        if (c < nch) {
                            load_chunk<CH>(src[sl] + (int64_t)c * CH, w[sl][k]);
                            if (MODE == 0) s[sl][k] = ld_nc_f32(rsc[sl] + c / CPR);
                            if (MODE == 2) s[sl][k] = sblk[sl];
                        }
                    }
                }
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
#pragma unroll
                    for (int k = 0; k < PER; ++k) {
                        const int c = c0 + k * kGatherThreads + threadIdx.x;
                        if (c >= nch) continue;
                        const int row = c / CPR;
                        const int col = c - row * CPR;
                        uint32_t o[CH / 2];
                        dequant_chunk<CH, MODE>(w[sl][k], s[sl][k], csc[sl] + col * SPAD, o);
                        store_chunk<CH, WIDE>(dst[sl] + (int64_t)row * a.out_tok_stride + col * CH, o);
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

template <int MODE, int CH, bool WIDE, bool APPEND>
cudaError_t launch_gather_variant(const GatherArgs &a, const AppendArgs &p, bool use_pdl,
                                  cudaStream_t stream) {
    auto kern = gather_kernel<MODE, CH, WIDE, APPEND>;
    const size_t smem = MODE == 1 ? sizeof(float) * 2 * a.g.kv_heads * (a.g.head_dim / CH) * (CH + 4) : 0;
    static OccupancySlots slots;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = occupancy(slots, kern, kGatherThreads, smem, &occ);
    if (e != cudaSuccess) return e;
    const int64_t max_items = (int64_t)a.g.num_seqs * a.g.max_blocks_per_seq * a.g.kv_heads +
                              (APPEND ? p.items : 0);
    const int64_t cap = (int64_t)sm_count() * occ;
    const int grid = (int)(max_items < cap ? max_items : cap);
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGatherThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a, p);
}

template <int MODE, bool WIDE, bool APPEND>
cudaError_t launch_gather_mode(const GatherArgs &a, const AppendArgs &p, bool use_pdl,
                               cudaStream_t stream) {
    if (a.g.head_dim % 32 == 0)
        return launch_gather_variant<MODE, 32, WIDE, APPEND>(a, p, use_pdl, stream);
    return launch_gather_variant<MODE, 16, WIDE, APPEND>(a, p, use_pdl, stream);
}

template <bool APPEND>
cudaError_t launch_gather_any(const GatherArgs &a, const AppendArgs &p, bool use_pdl,
                              cudaStream_t stream) {
    const uintptr_t k = reinterpret_cast<uintptr_t>(a.k_out);
    const uintptr_t v = reinterpret_cast<uintptr_t>(a.v_out);
    const bool wide = (k % 32 == 0) && (v % 32 == 0) && (a.out_tok_stride % 16 == 0) &&
                      (a.out_head_stride % 16 == 0);
    if (a.g.quant_mode == 0)
        return wide ? launch_gather_mode<0, true, APPEND>(a, p, use_pdl, stream)
                    : launch_gather_mode<0, false, APPEND>(a, p, use_pdl, stream);
    if (a.g.quant_mode == 1)
        return wide ? launch_gather_mode<1, true, APPEND>(a, p, use_pdl, stream)
                    : launch_gather_mode<1, false, APPEND>(a, p, use_pdl, stream);
    return wide ? launch_gather_mode<2, true, APPEND>(a, p, use_pdl, stream)
                : launch_gather_mode<2, false, APPEND>(a, p, use_pdl, stream);
}

// Threads of the plan's one CTA: a warp per 32 sequences, up to 1024.
int plan_threads(int32_t num_seqs) {
    const int w = (num_seqs + 31) / 32;
    return 32 * (w < 1 ? 1 : (w > kPlanThreads / 32 ? kPlanThreads / 32 : w));
}

}  // namespace

cudaError_t launch_plan(const kvc8_geom &g, const int32_t *context_lengths,
                        const int64_t *context_seq_offset, int64_t *offsets_out, void *plan,
                        int32_t *dev_error, cudaStream_t stream) {
    plan_kernel<<<1, plan_threads(g.num_seqs), 0, stream>>>(g, context_lengths, context_seq_offset,
                                                offsets_out, static_cast<char *>(plan), dev_error,
                                                nullptr, 0, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_plan_span(const kvc8_geom &g, const int32_t *context_kv_lens,
                             const int32_t *cu_q_lens, const int64_t *context_seq_offset,
                             void *plan, int32_t *spans_out, int32_t *dev_error,
                             cudaStream_t stream) {
    plan_kernel<<<1, plan_threads(g.num_seqs), 0, stream>>>(g, context_kv_lens, context_seq_offset, nullptr,
                                                static_cast<char *>(plan), dev_error, cu_q_lens,
                                                cu_q_lens != nullptr ? 3 : 4, spans_out);
    return cudaGetLastError();
}

cudaError_t launch_plan_append(const kvc8_geom &g, const int32_t *context_kv_lens,
                               const int32_t *cu_q_lens, const int64_t *context_seq_offset,
                               int64_t *offsets_out, void *plan, int32_t *dev_error,
                               cudaStream_t stream) {
    plan_kernel<<<1, plan_threads(g.num_seqs), 0, stream>>>(g, context_kv_lens, context_seq_offset,
                                                offsets_out, static_cast<char *>(plan), dev_error,
                                                cu_q_lens, cu_q_lens != nullptr ? 1 : 2, nullptr);
    return cudaGetLastError();
}

cudaError_t reset_plan_counter(void *plan, cudaStream_t stream) {
    return cudaMemsetAsync(static_cast<char *>(plan) + offsetof(PlanHeader, work_counter), 0,
                           sizeof(int64_t), stream);
}

cudaError_t launch_gather(const GatherArgs &a, bool use_pdl, cudaStream_t stream) {
    return launch_gather_any<false>(a, AppendArgs{}, use_pdl, stream);
}

cudaError_t launch_append_gather(const GatherArgs &a, const AppendArgs &p, bool use_pdl,
                                 cudaStream_t stream) {
    return launch_gather_any<true>(a, p, use_pdl, stream);
}

}  // namespace kvc8
