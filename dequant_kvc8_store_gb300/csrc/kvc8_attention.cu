// kvc8_attention.cu -- paged decode attention that reads the int8 cache
// directly: MojoPagedDecodeGQA of the "Mojo Opset" README ("Op List",
// Attention) over the values MojoDequantFromPagedKVCache (mojo_opset pull
// request #379) would materialise, without materialising them.
//
// Definition (the pages give no formula; this is grouped-query scaled
// dot-product attention of one query per sequence): query head j of sequence
// b uses kv head h = j / group, K'[p] and V'[p] are the cache rows dequantised
// exactly as the gather does (bf16(fl(float(code) * s))), and
//   out[b][j] = sum_p softmax_p(scale * <q[b][j], K'[p]>) * V'[p],  p < len_b,
// rounded to bf16; an empty context gives zeros.
//
// Work decomposition (split-K "flash decoding"): a sequence's context is cut
// into splits of kAttnChunk positions; a work item is (split, kv head) and is
// handed to a persistent grid through the plan's atomic counter.  A CTA of 4
// warps takes an item; each warp walks sub-tiles of 16 positions (a sub-tile
// never straddles a block: block_size is a multiple of 16) and keeps an online
// softmax state for the group's query heads.  The warps then merge through
// shared memory; a sequence with one split writes its output directly, longer
// ones leave a partial (m, l, O) per split for the merge kernel.
//
// Tensor cores: per sub-tile, S^T = K' Q^T and O^T += V'^T P^T are
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate) with the 16 positions -- or 16
// channels -- on M and the group's query heads (<= 8) on N, so nothing is
// padded when group = 8.  Each thread's fragment elements are assigned to
// channels so that it loads contiguous bytes: for QK, the k index
// kappa = 2t + j (+8) of k-step kk is channel t*D/4 + 4kk + j (+2); for PV,
// the row r (r + 8) of m-tile i is channel g*D/8 + 2i (+1).  P^T for the
// second mma is the first mma's accumulator, rounded to bf16 and transposed
// in registers (movmatrix).  The row sums use the rounded weights, so the
// normaliser matches the weights the second mma applies.
//
// The op is bound by HBM (the int8 rows are read once); the dequantisation of
// K and V runs on the CUDA cores beside the mma.
#include <cmath>

#include "kvc8_internal.cuh"

namespace kvc8 {
namespace {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kSub = 16;     // positions per warp step
constexpr int kMaxGroup = 8;  // query heads per kv head (mma N)
constexpr int kMergeThreads = 128;

__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// bf16x2 of (lo, hi), each rounded to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Codes e0 and e1 of a word, times s0 and s1: two exact conversions and two
// IEEE products, as packed fp32x2 operations.
__device__ __forceinline__ float2 dequant2(uint32_t w, int e0, int e1, float s0, float s1) {
    const uint32_t wb = w ^ 0x80808080u;
    float2 x = make_float2(__uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7440 + e0)),
                           __uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7440 + e1)));
    x = __fadd2_rn(x, make_float2(-8388736.0f, -8388736.0f));  // exact: c
    return __fmul2_rn(x, make_float2(s0, s1));
}

// 2^x by the hardware approximation (relative error far below the bf16
// rounding the weights get next); -inf gives 0.
__device__ __forceinline__ float ex2_fast(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Largest b in [0, B) with ts[b] <= tile.
__device__ __forceinline__ int seq_of_split(const int32_t *ts, int B, int64_t tile) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)ts[mid] <= tile) lo = mid; else hi = mid;
    }
    return lo;
}

template <int N>
__device__ __forceinline__ void load_bytes(const void *p, uint32_t *w) {
    if (N == 32) {
        const uint4 x = ld_stream_16(p), y = ld_stream_16(static_cast<const char *>(p) + 16);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        w[4] = y.x; w[5] = y.y; w[6] = y.z; w[7] = y.w;
    } else if (N == 16) {
        const uint4 x = ld_stream_16(p);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else {  // 8
        asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
    }
}

// The codes, scales and masks of one 16-position sub-tile, as one thread of
// the warp holds them.
template <int D>
struct Tile {
    uint32_t k0[D / 16], k1[D / 16];  // K codes: positions gid, gid + 8; bytes [tig*D/4, +D/4)
    uint32_t v[4][D / 32];            // V codes: positions 2tig, 2tig+1, 2tig+8, 2tig+9
    float sk0, sk1, sv[4];            // modes 0 and 2: the rows' (or block's) scales
    int32_t valid;                    // positions of the sub-tile before the context end
    bool ok;                          // the block id is inside the pool
};

template <int MODE, int D>
__device__ __forceinline__ void load_tile(const AttnArgs &a, int b, int h, int64_t p0,
                                          int64_t p_end, int gid, int tig, int lane,
                                          Tile<D> &t) {
    constexpr int KB = D / 4, VB = D / 8;
    const int H = a.g.kv_heads, bs = a.g.block_size, MB = a.g.max_blocks_per_seq;
    const int64_t lb = (int64_t)((uint32_t)p0 / (uint32_t)bs);
    const int32_t blk = ld_nc_s32(a.block_table + (int64_t)b * MB + lb);
    t.ok = blk >= 0 && blk < a.g.num_blocks;
    t.valid = (int32_t)min((int64_t)kSub, p_end - p0);
    if (!t.ok) {
        if (lane == 0) report(a.dev_error, KVC8_DEV_BAD_BLOCK_ID);
        return;
    }
    const int64_t row0 = ((int64_t)blk * H + h) * bs + (p0 - lb * bs);
    const int8_t *kp = a.k_cache + (row0 + gid) * D + tig * KB;
    load_bytes<KB>(kp, t.k0);
    load_bytes<KB>(kp + 8 * D, t.k1);
    const int8_t *vp = a.v_cache + (row0 + 2 * tig) * D + gid * VB;
    load_bytes<VB>(vp, t.v[0]);
    load_bytes<VB>(vp + D, t.v[1]);
    load_bytes<VB>(vp + 8 * D, t.v[2]);
    load_bytes<VB>(vp + 9 * D, t.v[3]);
    if (MODE == 0) {
        t.sk0 = ld_nc_f32(a.k_scale + row0 + gid);
        t.sk1 = ld_nc_f32(a.k_scale + row0 + gid + 8);
        t.sv[0] = ld_nc_f32(a.v_scale + row0 + 2 * tig);
        t.sv[1] = ld_nc_f32(a.v_scale + row0 + 2 * tig + 1);
        t.sv[2] = ld_nc_f32(a.v_scale + row0 + 2 * tig + 8);
        t.sv[3] = ld_nc_f32(a.v_scale + row0 + 2 * tig + 9);
    } else if (MODE == 2) {
        t.sk0 = t.sk1 = ld_nc_f32(a.k_scale + (int64_t)blk * H + h);
        t.sv[0] = t.sv[1] = t.sv[2] = t.sv[3] = ld_nc_f32(a.v_scale + (int64_t)blk * H + h);
    }
}

// O^T += V'^T P^T for one sub-tile; MASK zeroes V' rows at or past `valid`.
template <int MODE, int D, bool MASK>
__device__ __forceinline__ void pv_tile(const float *s_tab_v, const Tile<D> &t, int gid, int tig,
                                        uint32_t pb0, uint32_t pb1, float (*o)[4]) {
    constexpr int VB = D / 8, KS = D / 16;
    bool vv[4] = {true, true, true, true};
    if (MASK) {
        vv[0] = 2 * tig < t.valid;
        vv[1] = 2 * tig + 1 < t.valid;
        vv[2] = 2 * tig + 8 < t.valid;
        vv[3] = 2 * tig + 9 < t.valid;
    }
#pragma unroll
    for (int i = 0; i < KS; ++i) {
        float sd0 = 0.0f, sd1 = 0.0f;
        if (MODE == 1) {
            const float2 t2 = *reinterpret_cast<const float2 *>(s_tab_v + gid * (VB + 2) + 2 * i);
            sd0 = t2.x;
            sd1 = t2.y;
        }
        float f[4][2];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = dequant2(t.v[e][(2 * i) >> 2], (2 * i) & 3, (2 * i + 1) & 3,
                                      MODE == 1 ? sd0 : t.sv[e], MODE == 1 ? sd1 : t.sv[e]);
            f[e][0] = x.x;
            f[e][1] = x.y;
            if (MASK && !vv[e]) f[e][0] = f[e][1] = 0.0f;
        }
        mma_bf16(o[i], pack_bf16(f[0][0], f[1][0]), pack_bf16(f[0][1], f[1][1]),
                 pack_bf16(f[2][0], f[3][0]), pack_bf16(f[2][1], f[3][1]), pb0, pb1);
    }
}

template <int MODE, int D>
__device__ __forceinline__ void compute_tile(const AttnArgs &a, int h, const float *s_tab,
                                             const uint32_t *qf, int gid, int tig,
                                             const Tile<D> &t, float &m0, float &m1, float &l0,
                                             float &l1, float (*o)[4]) {
    constexpr int KB = D / 4, KS = D / 16;
    const int H = a.g.kv_heads;
    // S^T = K' Q^T
    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (MODE == 1) {
            const float4 t4 =
                *reinterpret_cast<const float4 *>(s_tab + h * (D + 16) + tig * (KB + 4) + 4 * kk);
            s4[0] = t4.x; s4[1] = t4.y; s4[2] = t4.z; s4[3] = t4.w;
        }
        const float2 a01 = dequant2(t.k0[kk], 0, 1, MODE == 1 ? s4[0] : t.sk0, MODE == 1 ? s4[1] : t.sk0);
        const float2 a23 = dequant2(t.k0[kk], 2, 3, MODE == 1 ? s4[2] : t.sk0, MODE == 1 ? s4[3] : t.sk0);
        const float2 b01 = dequant2(t.k1[kk], 0, 1, MODE == 1 ? s4[0] : t.sk1, MODE == 1 ? s4[1] : t.sk1);
        const float2 b23 = dequant2(t.k1[kk], 2, 3, MODE == 1 ? s4[2] : t.sk1, MODE == 1 ? s4[3] : t.sk1);
        mma_bf16(c, pack_bf16(a01.x, a01.y), pack_bf16(b01.x, b01.y), pack_bf16(a23.x, a23.y),
                 pack_bf16(b23.x, b23.y), qf[2 * kk], qf[2 * kk + 1]);
    }
    // scale into the log2 domain, mask positions past the context
    const bool va = gid < t.valid, vb8 = gid + 8 < t.valid;
    c[0] = va ? c[0] * a.scale_log2 : -INFINITY;
    c[1] = va ? c[1] * a.scale_log2 : -INFINITY;
    c[2] = vb8 ? c[2] * a.scale_log2 : -INFINITY;
    c[3] = vb8 ? c[3] * a.scale_log2 : -INFINITY;
    // online softmax per query head (a column: lanes with the same tig)
    float x0 = fmaxf(c[0], c[2]), x1 = fmaxf(c[1], c[3]);
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xFFFFFFFFu, x0, sh));
        x1 = fmaxf(x1, __shfl_xor_sync(0xFFFFFFFFu, x1, sh));
    }
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);  // finite: valid >= 1
    const float corr0 = ex2_fast(m0 - n0), corr1 = ex2_fast(m1 - n1);
    m0 = n0;
    m1 = n1;
    const uint32_t plo = pack_bf16(ex2_fast(c[0] - n0), ex2_fast(c[1] - n1));  // position gid
    const uint32_t phi = pack_bf16(ex2_fast(c[2] - n0), ex2_fast(c[3] - n1));  // position gid+8
    l0 = l0 * corr0 + (bf16_lo(plo) + bf16_lo(phi));
    l1 = l1 * corr1 + (bf16_hi(plo) + bf16_hi(phi));
#pragma unroll
    for (int i = 0; i < KS; ++i) {
        o[i][0] *= corr0; o[i][2] *= corr0;
        o[i][1] *= corr1; o[i][3] *= corr1;
    }
    const uint32_t pb0 = transpose8x8(plo), pb1 = transpose8x8(phi);
    const float *s_tab_v = s_tab + (H + h) * (D + 16);
    if (t.valid == kSub) pv_tile<MODE, D, false>(s_tab_v, t, gid, tig, pb0, pb1, o);
    else pv_tile<MODE, D, true>(s_tab_v, t, gid, tig, pb0, pb1, o);
}

// One work item = (split j of sequence b, kv head h).  Mode 1 is held to four
// CTAs per SM (its scale-table reads otherwise push it past 128 registers).
template <int MODE, int D>
__global__ void __launch_bounds__(kAttnThreads, MODE == 1 ? 4 : 0)
attention_kernel(const AttnArgs a) {
    constexpr int KB = D / 4;   // K code bytes per thread per position
    constexpr int VB = D / 8;   // V code bytes per thread per position
    constexpr int KS = D / 16;  // QK k-steps = PV m-tiles
    const int H = a.g.kv_heads, bs = a.g.block_size, B = a.g.num_seqs;
    const int MB = a.g.max_blocks_per_seq;
    const int G = a.group;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, tig = lane & 3;

    extern __shared__ float smem[];
    // Mode 1: the static scales [2][H][D], each row cut into the pieces one
    // thread reads (K: four of D/4, V: eight of D/8) and each piece padded so
    // that the pieces of a warp's threads fall in different banks.
    float *s_tab = smem;
    float *s_o = smem + (MODE == 1 ? 2 * H * (D + 16) : 0);  // [warps][8][D]
    float *s_m = s_o + kAttnWarps * kMaxGroup * D;         // [warps][8]
    float *s_l = s_m + kAttnWarps * kMaxGroup;             // [warps][8]
    __shared__ long long s_item;

    if (MODE == 1) {
        for (int i = threadIdx.x; i < 2 * H * D; i += blockDim.x) {
            const int row = i / D, d = i - row * D;
            if (row < H)
                s_tab[row * (D + 16) + (d / KB) * (KB + 4) + d % KB] = ld_nc_f32(a.k_scale + i);
            else
                s_tab[row * (D + 16) + (d / VB) * (VB + 2) + d % VB] = ld_nc_f32(a.v_scale + (i - H * D));
        }
        __syncthreads();
    }
    pdl_launch_dependents();  // the merge grid may launch; it waits for this one
    pdl_wait_prior_grid();    // the split plan is complete

    const char *plan = static_cast<const char *>(a.plan);
    const PlanHeader *hdr = reinterpret_cast<const PlanHeader *>(plan);
    const int32_t *ts = reinterpret_cast<const int32_t *>(plan + plan_tile_start_at(B));
    unsigned long long *counter =
        reinterpret_cast<unsigned long long *>(const_cast<int64_t *>(&hdr->work_counter));
    const int64_t items = hdr->total_tiles * H;
    const int64_t cap = (int64_t)MB * bs;

    int64_t item = blockIdx.x;
    while (item < items) {
        long long next = 0;
        if (threadIdx.x == 0) next = (long long)atomicAdd(counter, 1ull) + gridDim.x;
        const int64_t tile = (int64_t)((uint32_t)item / (uint32_t)H);  // items < 2^31
        const int h = (int)(item - tile * H);
        const int b = seq_of_split(ts, B, tile);
        const int64_t j = tile - ts[b];
        const int nsplit = ts[b + 1] - ts[b];
        const int64_t raw_len = ld_nc_s32(a.context_lengths + b);
        if (raw_len > cap && j == 0 && h == 0 && threadIdx.x == 0)
            report(a.dev_error, KVC8_DEV_POS_BEYOND_TABLE);
        const int64_t len = min(raw_len, cap);
        const int64_t p_begin = j * a.chunk;
        const int64_t p_end = min(len, p_begin + a.chunk);

        // Q^T fragments (mma B operand): query head gid of the group, its
        // channels [tig*KB, tig*KB + KB) as bf16 pairs
        uint32_t qf[KB / 2];
        if (gid < G) {
            const uint16_t *qp = a.q + (int64_t)b * a.q_seq_stride +
                                 (int64_t)(h * G + gid) * a.q_head_stride + tig * KB;
            load_bytes<KB * 2 >= 32 ? 32 : 16>(qp, qf);
            if (KB * 2 > 32) load_bytes<32>(qp + 16, qf + 8);
        } else {
#pragma unroll
            for (int i = 0; i < KB / 2; ++i) qf[i] = 0u;
        }

        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // heads 2tig, 2tig+1
        float o[KS][4];
#pragma unroll
        for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;

        // One sub-tile at a time: requesting the next one before computing the
        // current (a register double buffer) measured slower, the extra
        // registers costing more occupancy than the overlap gained.
        constexpr int64_t kStride = kAttnWarps * kSub;
        for (int64_t p0 = p_begin + warp * kSub; p0 < p_end; p0 += kStride) {
            Tile<D> t;
            load_tile<MODE, D>(a, b, h, p0, p_end, gid, tig, lane, t);
            if (t.ok) compute_tile<MODE, D>(a, h, s_tab, qf, gid, tig, t, m0, m1, l0, l1, o);
        }
        // row sums over the warp's positions
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, sh);
            l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, sh);
        }
        // warp partials -> shared memory: heads 2tig, 2tig+1; channels gid*VB + 2i (+1)
        float *so0 = s_o + (warp * kMaxGroup + 2 * tig) * D + gid * VB;
        float *so1 = so0 + D;
#pragma unroll
        for (int i = 0; i < KS; ++i) {
            so0[2 * i] = o[i][0];
            so0[2 * i + 1] = o[i][2];
            so1[2 * i] = o[i][1];
            so1[2 * i + 1] = o[i][3];
        }
        if (gid == 0) {
            s_m[warp * kMaxGroup + 2 * tig] = m0;
            s_m[warp * kMaxGroup + 2 * tig + 1] = m1;
            s_l[warp * kMaxGroup + 2 * tig] = l0;
            s_l[warp * kMaxGroup + 2 * tig + 1] = l1;
        }
        __syncthreads();
        // merge the warps; warp 0 always saw a position, so M is finite
        for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
            const int hd = idx / D, d = idx - hd * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w * kMaxGroup + hd]);
            float L = 0.0f, O = 0.0f;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) {
                const float f = exp2f(s_m[w * kMaxGroup + hd] - M);
                L += s_l[w * kMaxGroup + hd] * f;
                O += s_o[(w * kMaxGroup + hd) * D + d] * f;
            }
            if (nsplit == 1) {
                a.out[(int64_t)b * a.out_seq_stride + (int64_t)(h * G + hd) * a.out_head_stride + d] =
                    (uint16_t)(pack_bf16(O / L, 0.0f) & 0xFFFFu);
            } else {
                a.part_o[(item * G + hd) * D + d] = O;
                if (d == 0) {
                    a.part_m[item * G + hd] = M;
                    a.part_l[item * G + hd] = L;
                }
            }
        }
        if (threadIdx.x == 0) s_item = next;
        __syncthreads();
        item = s_item;
        __syncthreads();
    }
}

// Sequences with more than one split: combine the splits' partials; empty
// sequences: zeros.  One CTA per (sequence, kv head); a warp per query head,
// the lanes over channels (D/32 each), the split weights computed 32 at a
// time and broadcast by shuffles.
__global__ void __launch_bounds__(kMergeThreads)
attention_merge_kernel(const AttnArgs a) {
    pdl_wait_prior_grid();  // all partials are written
    const int H = a.g.kv_heads, B = a.g.num_seqs, D = a.g.head_dim, G = a.group;
    const int b = blockIdx.x / H, h = blockIdx.x - b * H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t *ts = reinterpret_cast<const int32_t *>(static_cast<const char *>(a.plan) +
                                                          plan_tile_start_at(B));
    const int first = ts[b], nsplit = ts[b + 1] - ts[b];
    if (nsplit == 1) return;
    const int per = D / 32;  // channels per lane: 2 or 4
    for (int hd = warp; hd < G; hd += kMergeThreads / 32) {
        uint16_t *dst = a.out + (int64_t)b * a.out_seq_stride +
                        (int64_t)(h * G + hd) * a.out_head_stride + lane * per;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (nsplit > 1) {
            float M = -INFINITY;
            for (int j = lane; j < nsplit; j += 32)
                M = fmaxf(M, a.part_m[((int64_t)(first + j) * H + h) * G + hd]);
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, sh));
            float L = 0.0f;
            for (int j0 = 0; j0 < nsplit; j0 += 32) {
                const int j = j0 + lane;
                float f = 0.0f;
                if (j < nsplit) {
                    const int64_t it = ((int64_t)(first + j) * H + h) * G + hd;
                    f = exp2f(a.part_m[it] - M);
                    L += a.part_l[it] * f;
                }
                const int n = min(32, nsplit - j0);
                for (int k = 0; k < n; ++k) {
                    const float fk = __shfl_sync(0xFFFFFFFFu, f, k);
                    const float *po = a.part_o + (((int64_t)(first + j0 + k) * H + h) * G + hd) * D +
                                      lane * per;
                    if (per == 4) {
                        const float4 v = *reinterpret_cast<const float4 *>(po);
                        acc[0] += fk * v.x; acc[1] += fk * v.y; acc[2] += fk * v.z; acc[3] += fk * v.w;
                    } else {
                        const float2 v = *reinterpret_cast<const float2 *>(po);
                        acc[0] += fk * v.x; acc[1] += fk * v.y;
                    }
                }
            }
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, sh);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] /= L;
        }
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            if (e < per) {
                const uint32_t pr = pack_bf16(acc[e], acc[e + 1]);
                dst[e] = (uint16_t)(pr & 0xFFFFu);
                dst[e + 1] = (uint16_t)(pr >> 16);
            }
        }
    }
}

size_t part_elems(const kvc8_geom &g) {
    const int64_t splits = ((int64_t)g.max_blocks_per_seq * g.block_size + kAttnChunk - 1) / kAttnChunk;
    return (size_t)g.num_seqs * g.kv_heads * splits;  // items
}

template <int MODE, int D>
cudaError_t launch_attention_variant(const AttnArgs &a, cudaStream_t stream) {
    auto kern = attention_kernel<MODE, D>;
    const size_t smem = sizeof(float) * ((MODE == 1 ? 2 * a.g.kv_heads * (D + 16) : 0) +
                                         kAttnWarps * kMaxGroup * (D + 2));
    static OccupancySlots slots;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = occupancy(slots, kern, kAttnThreads, smem, &occ);
    if (e != cudaSuccess) return e;
    const int64_t max_items = (int64_t)part_elems(a.g);
    const int64_t cap = (int64_t)sm_count() * occ;
    const int grid = (int)(max_items < cap ? max_items : cap);
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int MODE>
cudaError_t launch_attention_mode(const AttnArgs &a, cudaStream_t stream) {
    if (a.g.head_dim == 64) return launch_attention_variant<MODE, 64>(a, stream);
    return launch_attention_variant<MODE, 128>(a, stream);
}

}  // namespace

size_t attention_workspace_bytes(const kvc8_geom &g, int group) {
    const size_t items = part_elems(g);
    return plan_bytes(g.num_seqs) + align_up(sizeof(float) * items * group * g.head_dim, kAlign) +
           2 * align_up(sizeof(float) * items * group, kAlign);
}

cudaError_t launch_attention(AttnArgs a, void *workspace, cudaStream_t stream) {
    // the split plan: the gather's plan with splits of kAttnChunk positions
    kvc8_geom gs = a.g;
    gs.block_size = kAttnChunk;
    gs.max_blocks_per_seq =
        (int32_t)(((int64_t)a.g.max_blocks_per_seq * a.g.block_size + kAttnChunk - 1) / kAttnChunk);
    cudaError_t e = launch_plan(gs, a.context_lengths, nullptr, nullptr, workspace, a.dev_error,
                                stream);
    if (e != cudaSuccess) return e;
    const size_t items = part_elems(a.g);
    char *base = static_cast<char *>(workspace) + plan_bytes(a.g.num_seqs);
    a.plan = workspace;
    a.chunk = kAttnChunk;
    a.part_o = reinterpret_cast<float *>(base);
    base += align_up(sizeof(float) * items * a.group * a.g.head_dim, kAlign);
    a.part_m = reinterpret_cast<float *>(base);
    base += align_up(sizeof(float) * items * a.group, kAlign);
    a.part_l = reinterpret_cast<float *>(base);
    if (a.g.quant_mode == 0) e = launch_attention_mode<0>(a, stream);
    else if (a.g.quant_mode == 1) e = launch_attention_mode<1>(a, stream);
    else e = launch_attention_mode<2>(a, stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.g.num_seqs * a.g.kv_heads));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attention_merge_kernel, a);
}

}  // namespace kvc8
