// kvc8_store.cu -- quantise new bf16 K/V tokens to int8 and scatter them into
// the paged cache (MojoStorePagedKVCacheC8 in mojo_opset pull request #379,
// "feat: [MLU] add mlu experimental ops; fix post norm bug").
//
// Work decomposition: each lane owns 16 consecutive channels (32 bytes of
// input, 16 bytes of codes) of one row, and keeps that row and those channels
// for every token it handles.  A token carries 2*H rows (K heads, then V
// heads); L = D/16 lanes (rounded up to a power of two) cover a row, so a warp
// covers 32/L rows of a token and NW = 2H*L/32 warps (rounded up) cover it.
// The warps form S streams of NW warps, one warp per row set, and stream s
// takes tokens s, s + S, s + 2S, ..., so that all streams together sweep a
// window of S consecutive tokens through the batch (the streams' token counts
// differ by at most one).
// - Each warp keeps its next tokens' rows in flight in a ring of shared-memory
//   slots filled by cp.async (each lane copies and later reads back only its
//   own 32 bytes, so no barrier is needed): the loads run ahead of the
//   arithmetic without holding registers.
// - The slots of a stream's next 32 tokens are looked up at once, one token
//   per lane, and handed to the row lanes by shuffles.
// - Because a lane's channels never change, the static per-channel mode keeps
//   its per-channel bracket ends and clamp bounds in registers for the whole
//   launch (computed while the first rows are on their way).
// The per-value work is a few packed fp32x2 operations (see below); the
// kernel sits between the issue and the memory limits.
//
// Rounding is bit-exact with the definition q = clamp(rne(x / s), -127, 127)
// (one IEEE fp32 division), without dividing in the common case.
//
// Dynamic mode (s = fl(amax/127), r = fl(1/s), both exact from 128-entry tables
// indexed by the bf16 mantissa of amax): every value fl(x/s) can take lies
// between x * r_lo and x * r_hi, with r_lo = fl(r (1 - 2^-21)) <= r (1 - 2^-23)
// and r_hi >= r (1 + 2^-23), because r and fl(x/s) are each within a relative
// 2^-24 of 1/s and x/s.  One fused multiply-add per end gives
// 1.5*2^23 + rne(x r_lo) and 1.5*2^23 + rne(x r_hi) from the exact products
// (|x r| <= 127.0001, so adding 1.5*2^23 rounds to an integer, ties to even,
// and the low byte of the result is the code).  If the two agree, rne is
// monotone, so rne(fl(x/s)) is that same integer.  If they differ (a value
// within about 2^-21 relative of a half-integer, in practice almost always an
// exact tie x/s = n + 1/2; about 2 values in 10^4 of bf16 data), the group of
// four values is recomputed in registers by code_exact, which decides the
// rounding from one exact remainder |x| - (n + 1/2) s instead of a division.
//
// Static modes (s per channel, quant_mode 1, held by each lane in registers
// for its channels; or s per block and kv head, quant_mode 2, read once per
// row and token) use the same bracket after clamping |x| to the bound
// bf16(fl(127 s)) (bf16_bound below).  Their flagged groups are redone after
// the store by fix_codes: mode 1 divides; mode 2 takes quant_one, where
// y = fl(x * fl(1/s)) clamped to [-127, 127] has a relative error against
// t = x/s of at most 2^-23 + 2^-48, so |y - t| < 1.55e-5 for |t| <= 130 and
// fl(t) is within half an ulp of t (<= 7.7e-6 below 256).  If y lies more
// than 2^-15 from every half-integer, t and fl(t) lie strictly inside the
// same interval between half-integers as y and rne(y) = rne(fl(t));
// otherwise the value takes one division.  |y| >= 127 means
// |t| >= 126.99998, whose code is +-127 either way.
//
// Scales whose reciprocal could leave the normal range (and zero scales)
// always take the exact path.
#include <type_traits>

#include "kvc8_internal.cuh"

namespace kvc8 {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr float kMagic = 12582912.0f;            // 1.5 * 2^23
constexpr float kNearTie = 0.499969482421875f;   // 0.5 - 2^-15
constexpr float kSatClamp = 127.0f;   // |y| >= 127 gives +-127 on both paths
constexpr float kRecipLo = 0.99999952316284180f;  // 1 - 2^-21
constexpr float kRecipHi = 1.00000047683715820f;  // 1 + 2^-21

// The clamp bound of a static scale s (recip_ok(s)): B = bf16_rne(fl(127 s)).
// B / s lies within a relative 2^-8 + 2^-24 of 127, i.e. in (126.5, 127.5),
// so rne(fl(B / s)) = 127, and by monotonicity every |x| >= B has a code of
// at least 127 in magnitude: clamping |x| to B leaves clamp(code(x)) unchanged.
__device__ __forceinline__ uint32_t bf16_bound(float s) {
    unsigned short b;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b) : "f"(__fmul_rn(127.0f, s)));
    return b;
}

// Reciprocal fast path needs s and 1/s normal and finite.
__device__ __forceinline__ bool recip_ok(float s) {
    return s >= 0x1p-120f && s <= 0x1p+120f;
}

// The definition: one IEEE division, round half to even, clamp; 0 when s == 0.
__device__ __noinline__ int quant_exact(float x, float s) {
    if (s == 0.0f) return 0;
    int q = __float2int_rn(__fdiv_rn(x, s));
    return min(127, max(-127, q));
}

// Code of one value on the fast path (r != 0), or the exact path when the
// value is near a tie, r == 0 marks an out-of-range scale, or force is set.
__device__ __forceinline__ int quant_one(float x, float s, float r) {
    if (r == 0.0f) return quant_exact(x, s);
    float y = fminf(fmaxf(__fmul_rn(x, r), -kSatClamp), kSatClamp);
    float m = __fadd_rn(y, kMagic);
    float d = __fsub_rn(y, __fsub_rn(m, kMagic));
    if (fabsf(d) >= kNearTie) return quant_exact(x, s);
    return __float_as_int(m) - 0x4B400000;
}

// Lower bound on the scales for which code_exact below is exact (all of its
// intermediate quantities stay normal).
constexpr float kExactMinScale = 0x1p-100f;

// rne(fl(x / s)) clamped to [-127, 127], for a bf16 value x, a scale
// 2^-100 <= s <= 2^120 and r = fl(1/s), without dividing.  With t = |x|/s
// and y = fl(|x| r) (|y - t| <= 2^-23 y), let n = floor(y) and h = n + 1/2.
// d = |x| - h s is a multiple of 2^(e_s - 24) (e_s the exponent of s) because
// |x| has 8 significant bits and |x| >= h s / 2; so wherever
// |t - h| < 2^-13, |d| < 2^12 of those units and the fma computes d exactly;
// elsewhere its sign is still exact and |d| is far above the bounds below.
// fl(t) equals h exactly when t lies within half the spacing of floats
// around h (closed interval: h has an even significand, so the midpoints
// round to it), i.e. when -s u_lo <= d <= s u_hi with u_hi = ulp(h)/2 and
// u_lo = u_hi except u_lo = u_hi/2 at h = 1/2, the one power of two among
// the half-integers.  Then rne picks the even neighbour; otherwise fl(t) lies
// on the same side of h as t, and the code is n or n + 1 by the sign of d.
__device__ __forceinline__ int code_exact(float x, float s, float r) {
    const float ax = fabsf(x);
    const float y = __fmul_rn(ax, r);
    int q = 127;  // y >= 127 means t >= 126.99998, which rounds to 127 or more
    if (y < 127.0f) {
        const float n = floorf(y);
        const float h = __fadd_rn(n, 0.5f);
        const float d = __fmaf_rn(-h, s, ax);
        const float u_hi = __int_as_float((__float_as_int(h) & 0x7F800000) - (24 << 23));
        const float u_lo = h == 0.5f ? __fmul_rn(u_hi, 0.5f) : u_hi;
        const int ni = (int)n;
        const bool on_h = d <= __fmul_rn(s, u_hi) && d >= -__fmul_rn(s, u_lo);
        q = on_h ? ni + (ni & 1) : (d > 0.0f ? ni + 1 : ni);
        q = min(q, 127);
    }
    return x < 0.0f ? -q : q;
}

__device__ __forceinline__ uint32_t pack_lo_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// The groups of four codes flagged in `fix` (bit q: codes 4q..4q+3 of a
// lane's run), recomputed from the source values one by one with the exact
// fallback and stored over the fast codes at dst.  Mode 1 divides by each
// value's scale; modes 0 and 2 use the row's scale and reciprocal.
template <int MODE>
__device__ __noinline__ void fix_codes(const uint16_t *src, int8_t *dst, uint32_t fix, float s_row,
                                       float r_row, const float *st) {
    while (fix != 0u) {
        const int q = __ffs(fix) - 1;
        fix &= fix - 1u;
        uint32_t c4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 4 * q + e;
            const float x = __uint_as_float((uint32_t)src[j] << 16);
            const int code = MODE == 1 ? quant_exact(x, ld_nc_f32(st + j)) : quant_one(x, s_row, r_row);
            c4[e] = (uint32_t)code;
        }
        *reinterpret_cast<uint32_t *>(dst + 4 * q) = pack_lo_bytes(c4[0], c4[1], c4[2], c4[3]);
    }
}

__device__ __forceinline__ void store_codes16(int8_t *p, const uint32_t c[4]) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(c[0]), "r"(c[1]),
                 "r"(c[2]), "r"(c[3])
                 : "memory");
}


constexpr int kChunk = 32;  // tokens whose slots one lookup round finds (one per lane)

// cp.async: 16 bytes global -> shared (L2 only), committed in groups and
// waited for by the issuing thread, which alone reads them back.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// tokens per warp in the shared-memory ring (one fewer in flight): the
// static per-channel mode, held to two CTAs per SM by its register tables,
// goes deeper
constexpr int kStagesDyn = 4;
constexpr int kStagesStatic = 8;
template <int MODE>
constexpr int ring_stages() { return MODE == 1 ? kStagesStatic : kStagesDyn; }

// L lanes per row (a power of two, 32 / L rows per warp), MODE 0 dynamic /
// 1 static per channel / 2 static per block.
template <int L, int MODE, bool R32>
__global__ void __launch_bounds__(kWarpsPerCta * 32, MODE == 1 ? 2 : 4)
store_kernel(const StoreArgs a) {
    // cache row indices: 32-bit when the pool has fewer than 2^31 rows
    using Row = typename std::conditional<R32, int32_t, int64_t>::type;
    constexpr int RW = 32 / L;  // rows per warp
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int C = D / 16;  // active lanes per row
    const int rows = 2 * H;
    const int NW = (rows + RW - 1) / RW;  // warps per token
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * kWarpsPerCta + warp;
    const int S = (gridDim.x * kWarpsPerCta) / NW;  // streams
    const int j = gw % NW, s = gw / NW;
    constexpr int kStages = ring_stages<MODE>();
    static_assert((kStages & (kStages - 1)) == 0, "ring slots wrap by masking");

    // Dynamic mode: for a bf16 row maximum amax = (1 + m/128) * 2^E,
    // s = fl(amax / 127) = fl((1 + m/128) / 127) * 2^E and 1/s rounds to
    // fl(1 / that) * 2^-E exactly, as long as both stay normal; the tables
    // hold the two fl() values for the 128 mantissas.  Then each warp's ring
    // of kStages token slots, 32 bytes per lane each.
    extern __shared__ __align__(16) float smem[];
    float *s_tab = smem, *r_tab = smem + 128;
    uint8_t *ring = reinterpret_cast<uint8_t *>(smem + (MODE == 0 ? 256 : 0));
    if (MODE == 0) {
        for (int m = threadIdx.x; m < 128; m += blockDim.x) {
            const float sm = __fdiv_rn(__uint_as_float(0x3F800000u | ((uint32_t)m << 16)), 127.0f);
            s_tab[m] = sm;
            r_tab[m] = __frcp_rn(sm);
        }
        __syncthreads();
    }
    if (s >= S) return;  // warps beyond the last whole stream

    const int rl = lane / L, c = lane % L;
    const int row = j * RW + rl;
    const bool on = row < rows && c < C;
    const int kv = row >= H ? 1 : 0;
    const int h = on ? row - kv * H : 0;
    const uint16_t *xs = (kv ? a.v_states : a.k_states) + (int64_t)h * a.x_head_stride + c * 16;
    int8_t *cache = (kv ? a.v_cache : a.k_cache) + c * 16;
    float *scl = kv ? a.v_scale : a.k_scale;
    const Row hoff = (Row)h * bs;  // cache row of head h in a block, slot 0
    const uint32_t my = smem_u32(ring) + ((uint32_t)warp * kStages * 32 + lane) * 32;

    // this stream's tokens: s, s + S, s + 2S, ... (all streams together
    // sweep a window of S consecutive tokens through the batch); the rows of
    // its m-th token go to ring slot m % kStages, kStages - 1 tokens ahead
    const int mine = s < a.num_tokens ? (int)((a.num_tokens - 1 - s) / S) + 1 : 0;  // tokens < 2^31
    const int64_t pf_step = (int64_t)S * a.x_tok_stride;
    const uint16_t *pf_src = xs + (int64_t)s * a.x_tok_stride;  // next token to request
    int pf_left = on ? mine : 0;                                  // tokens left to request
    uint32_t pf_slot = 0;                                         // its ring slot (bytes)
    constexpr uint32_t kRingMask = kStages * 32 * 32 - 1;
    auto prefetch = [&]() {
        if (pf_left > 0) {
            cp_async16(my + pf_slot, pf_src);
            cp_async16(my + pf_slot + 16, pf_src + 8);
        }
        cp_async_commit();
        --pf_left;
        pf_src += pf_step;
        pf_slot = (pf_slot + 32 * 32) & kRingMask;
    };
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) prefetch();
    // Lanes off the rows feed only the dynamic mode's row maximum, as zeros:
    // no copy ever lands in their ring slots, so zero those once.
    if (MODE == 0 && !on) {
#pragma unroll
        for (int k = 0; k < 2 * kStages; ++k)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(my + 16 * (k & 1) + 32 * 32 * (k >> 1)), "r"(0u)
                         : "memory");
    }

    // Static per-channel mode: this lane's bracket ends r_lo, r_hi of
    // r = fl(1/s) and clamp bounds bf16(fl(127 s)) for its 16 channels, held
    // for the whole launch (computed while the first rows are on their way).
    // A scale outside the reciprocal range sends the lane's values to the
    // exact path.
    float2 rlo1[8], rhi1[8];
    uint32_t bnd1[8];
    bool lane_fast = true;
    if (MODE == 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            rlo1[i] = make_float2(0.0f, 0.0f);
            rhi1[i] = rlo1[i];
            bnd1[i] = 0u;
        }
        if (on) {
            const float *sp = scl + (int64_t)h * D + c * 16;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float s0 = ld_nc_f32(sp + 2 * i), s1 = ld_nc_f32(sp + 2 * i + 1);
                const bool f0 = recip_ok(s0), f1 = recip_ok(s1);
                const float r0 = f0 ? __frcp_rn(s0) : 0.0f, r1 = f1 ? __frcp_rn(s1) : 0.0f;
                rlo1[i] = make_float2(__fmul_rn(r0, kRecipLo), __fmul_rn(r1, kRecipLo));
                rhi1[i] = make_float2(__fmul_rn(r0, kRecipHi), __fmul_rn(r1, kRecipHi));
                bnd1[i] = bf16_bound(s0) | (bf16_bound(s1) << 16);
                lane_fast = lane_fast && f0 && f1;
            }
        }
    }

    const float2 magic2 = make_float2(kMagic, kMagic);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    Row row0 = -1;  // lane i: cache row of (block, head 0, slot) of token 32q + i; -1: skip
    int32_t blk = 0;
    uint32_t rd_slot = 0;  // ring slot of token m (bytes)

    for (int m = 0; m < mine; ++m) {
        const int i = (int)(m & (kChunk - 1));
        if (i == 0) {
            // ---- slots of this stream's next kChunk tokens, one per lane ----
            row0 = -1;
            blk = 0;
            if (m + lane < mine) {
                const int64_t t = s + (int64_t)(m + lane) * S;
                int64_t first = t, next = t + 1, ctx;
                int b;
                if (a.cu_q_lens != nullptr) {
                    // the last sequence whose first new token is at or before t
                    int lo = 0;
                    for (int step = 1 << (31 - __clz(max(B - 1, 1))); step > 0; step >>= 1)
                        if (lo + step < B && (int64_t)ld_nc_s32(a.cu_q_lens + lo + step) <= t) lo += step;
                    b = lo;
                    first = ld_nc_s32(a.cu_q_lens + b);
                    next = ld_nc_s32(a.cu_q_lens + b + 1);
                } else {
                    b = (int)t;
                }
                ctx = ld_nc_s32(a.context_kv_lens + b);
                const int64_t pos = ctx + (t - first);
                // pos < 2^32 always (ctx and the token index are below 2^31):
                // floor(pos / bs) is the high word of pos * ceil(2^64 / bs)
                int64_t lb;
                if (pos >= 0 && pos <= 0xFFFFFFFFll) {
                    lb = bs == 1 ? pos : (int64_t)__umul64hi(a.bs_magic, (unsigned long long)pos);
                } else {
                    lb = pos / bs;
                }
                int32_t err = 0;
                if (!(first <= t && t < next) || ctx < 0) {
                    err = KVC8_DEV_BAD_LENGTH;
                } else if (lb >= MB) {
                    err = KVC8_DEV_POS_BEYOND_TABLE;
                } else {
                    blk = ld_nc_s32(a.block_table + (int64_t)b * MB + lb);
                    if (blk < 0 || blk >= NB) err = KVC8_DEV_BAD_BLOCK_ID;
                }
                if (err == 0) {
                    row0 = (Row)((int64_t)blk * H * bs + (pos - lb * bs));
                } else {
                    blk = 0;  // never used as an index
                    if (j == 0) report(a.dev_error, err);
                }
            }
        }

        // ---- this token's rows from the ring; the next one requested ----
        cp_async_wait<kStages - 2>();
        uint32_t w[8];
        {
            const uint32_t src = my + rd_slot;
            rd_slot = (rd_slot + 32 * 32) & kRingMask;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(src));
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "r"(src + 16));
        }
        prefetch();

        const Row r0 = __shfl_sync(0xFFFFFFFFu, row0, i);
        if (r0 < 0) continue;  // warp-uniform: the token is skipped
        const Row drow = r0 + hoff;

        float s_row = 0.0f, r_row = 0.0f;
        if (MODE == 0) {
            // |x| maximum: max(|a|, |b|) per bf16 half (the sign of the
            // result is garbage and masked off before comparing words)
            // (a tree: each level takes |.| of the previous maxima again)
            uint32_t m4[4], m2[2], m1;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m4[k]) : "r"(w[2 * k]), "r"(w[2 * k + 1]));
#pragma unroll
            for (int k = 0; k < 2; ++k)
                asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2[k]) : "r"(m4[2 * k]), "r"(m4[2 * k + 1]));
            asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m1) : "r"(m2[0]), "r"(m2[1]));
            m1 &= 0x7FFF7FFFu;
            uint32_t mag = max(m1 & 0xFFFFu, m1 >> 16);
#pragma unroll
            for (int o = 1; o < L; o <<= 1)
                mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, o));
            const uint32_t ef = mag >> 7;  // bf16 exponent field of amax
            if (ef >= 14 && ef <= 253) {   // s and 1/s normal and within recip_ok
                const int sh = ((int)ef - 127) << 23;
                s_row = __int_as_float(__float_as_int(s_tab[mag & 127]) + sh);
                r_row = __int_as_float(__float_as_int(r_tab[mag & 127]) - sh);
            } else {
                s_row = __fdiv_rn(__uint_as_float(mag << 16), 127.0f);
                r_row = 0.0f;  // exact path for the whole row
            }
        } else if (MODE == 2) {
            // the row's block scale; a zero reciprocal sends the row to the
            // exact path
            const int32_t bg = __shfl_sync(0xFFFFFFFFu, blk, i);
            s_row = on ? ld_nc_f32(scl + (int64_t)bg * H + h) : 0.0f;
            r_row = recip_ok(s_row) ? __frcp_rn(s_row) : 0.0f;
        }

        uint32_t cw[4];      // packed codes, four per word
        uint32_t fix = 0u;   // bit q: codes 4q..4q+3 need the exact path
        const bool force_exact = (MODE == 1) ? !lane_fast : (r_row == 0.0f);
        // r_lo <= r (1 - 2^-23) and r_hi >= r (1 + 2^-23) bracket every
        // value fl(x / s) can take, so when x r_lo and x r_hi round to the
        // same integer, so does fl(x / s).  Modes 0 and 2: the row's pair;
        // mode 1: each channel's.
        const float2 rlo2 = make_float2(__fmul_rn(r_row, kRecipLo), __fmul_rn(r_row, kRecipLo));
        const float2 rhi2 = make_float2(__fmul_rn(r_row, kRecipHi), __fmul_rn(r_row, kRecipHi));
        // Modes 1 and 2 clamp x to +-bf16(fl(127 s)) before the bracket (one
        // min.xorsign.abs per pair): that bound's code is +-127 and every
        // larger |x| saturates, so the clamp gives clamp(code(x)) and keeps
        // |x r| below 127.5.
        const uint32_t brow = MODE == 2 ? bf16_bound(s_row) * 0x10001u : 0u;
        // Group q of four values adds its bracket gap (0 to 4, the squared
        // differences of the ends) times 8^q to flagsf: an exact base-8
        // record of the flagged groups, kept on the FMA pipe.
        float flagsf = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            uint32_t mbits[4];
            float2 dacc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                uint32_t wi = w[k + e];
                const float2 rlo = MODE == 1 ? rlo1[k + e] : rlo2;
                const float2 rhi = MODE == 1 ? rhi1[k + e] : rhi2;
                if (MODE != 0) {
                    const uint32_t bnd = MODE == 1 ? bnd1[k + e] : brow;
                    asm("min.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(wi) : "r"(wi), "r"(bnd));
                }
                const float2 x2 = make_float2(__uint_as_float(wi << 16), __uint_as_float(wi & 0xFFFF0000u));
                const float2 m2 = __ffma2_rn(x2, rlo, magic2);
                const float2 h2 = __ffma2_rn(x2, rhi, magic2);
                // the two ends differ by one or not at all; their squared
                // differences add up exactly, on the FMA pipe rather than
                // the busier ALU pipe
                const float2 dd = __ffma2_rn(m2, neg1, h2);  // h2 - m2, exact
                dacc = __ffma2_rn(dd, dd, dacc);
                mbits[2 * e] = __float_as_uint(m2.x);  // low byte = code
                mbits[2 * e + 1] = __float_as_uint(m2.y);
            }
            cw[k / 2] = pack_lo_bytes(mbits[0], mbits[1], mbits[2], mbits[3]);
            flagsf = __fmaf_rn(__fadd_rn(dacc.x, dacc.y), (float)(1u << (3 * (k / 2))), flagsf);
        }
        if (flagsf != 0.0f) {  // rare: which groups
            const uint32_t u = (uint32_t)flagsf;
#pragma unroll
            for (int q = 0; q < 4; ++q) fix |= ((u >> (3 * q)) & 7u) ? (1u << q) : 0u;
        }
        // Dynamic mode: the flagged groups (nearly all exact ties,
        // x/s = n + 1/2) are recomputed in registers by code_exact before the
        // store.  The static modes take the out-of-line pass after the store.
        bool slow = force_exact || (MODE == 0 && fix != 0u && !(s_row >= kExactMinScale));
        if (MODE == 0 && !slow && fix != 0u) {
            uint32_t f = fix;
            do {
                const int q = __ffs(f) - 1;
                f &= f - 1u;
                uint32_t w0 = w[0], w1 = w[1];
#pragma unroll
                for (int k = 1; k < 4; ++k)
                    if (q == k) {
                        w0 = w[2 * k];
                        w1 = w[2 * k + 1];
                    }
                const uint32_t cq = pack_lo_bytes(
                    (uint32_t)code_exact(__uint_as_float(w0 << 16), s_row, r_row),
                    (uint32_t)code_exact(__uint_as_float(w0 & 0xFFFF0000u), s_row, r_row),
                    (uint32_t)code_exact(__uint_as_float(w1 << 16), s_row, r_row),
                    (uint32_t)code_exact(__uint_as_float(w1 & 0xFFFF0000u), s_row, r_row));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (q == k) cw[k] = cq;
            } while (f != 0u);
            fix = 0u;
        }
        if (slow) fix = 0xFu;
        if (on) {
            int8_t *dst = cache + (int64_t)drow * D;
            store_codes16(dst, cw);
            if (MODE == 0 && c == 0) scl[drow] = s_row;
            if (fix != 0u) {
                // rare: the flagged groups of four codes again, one by one,
                // with one division where needed, over the codes just stored
                fix_codes<MODE>(xs + (s + (int64_t)m * S) * a.x_tok_stride, dst, fix, s_row, r_row,
                                scl + (int64_t)h * D + c * 16);
            }
        }
    }
    cp_async_wait<0>();
}

template <int L, int MODE, bool R32>
cudaError_t launch_variant(const StoreArgs &a, cudaStream_t stream) {
    auto kern = store_kernel<L, MODE, R32>;
    const size_t smem = (MODE == 0 ? sizeof(float) * 256 : 0) + (size_t)kWarpsPerCta * ring_stages<MODE>() * 32 * 32;
    static OccupancySlots slots;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = occupancy(slots, kern, kWarpsPerCta * 32, smem, &occ);
    if (e != cudaSuccess) return e;
    const int64_t nw = (2 * (int64_t)a.g.kv_heads * L + 31) / 32;  // warps per token
    const int64_t min_grid = (nw + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t need = (a.num_tokens * nw + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = (int64_t)sm_count() * occ;
    int64_t grid = need < cap ? need : cap;
    if (grid < min_grid) grid = min_grid;
    kern<<<(unsigned)grid, kWarpsPerCta * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int MODE, bool R32>
cudaError_t launch_mode_rows(const StoreArgs &a, cudaStream_t stream) {
    const int C = a.g.head_dim / 16;  // 1..16
    if (C <= 1) return launch_variant<1, MODE, R32>(a, stream);
    if (C <= 2) return launch_variant<2, MODE, R32>(a, stream);
    if (C <= 4) return launch_variant<4, MODE, R32>(a, stream);
    if (C <= 8) return launch_variant<8, MODE, R32>(a, stream);
    return launch_variant<16, MODE, R32>(a, stream);
}

template <int MODE>
cudaError_t launch_mode(const StoreArgs &a, cudaStream_t stream) {
    const bool r32 = (int64_t)a.g.num_blocks * a.g.kv_heads * a.g.block_size <= (int64_t)INT32_MAX;
    return r32 ? launch_mode_rows<MODE, true>(a, stream) : launch_mode_rows<MODE, false>(a, stream);
}

}  // namespace

cudaError_t launch_store(const StoreArgs &a, cudaStream_t stream) {
    if (a.num_tokens <= 0) return cudaSuccess;
    if (a.g.quant_mode == 0) return launch_mode<0>(a, stream);
    if (a.g.quant_mode == 1) return launch_mode<1>(a, stream);
    return launch_mode<2>(a, stream);
}

}  // namespace kvc8
