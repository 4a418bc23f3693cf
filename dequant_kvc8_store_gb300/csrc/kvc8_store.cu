// kvc8_store.cu -- quantise new bf16 K/V tokens to int8 and scatter them into
// the paged cache (MojoStorePagedKVCacheC8 in mojo_opset pull request #379,
// "feat: [MLU] add mlu experimental ops; fix post norm bug").
//
// Work decomposition: one warp per token.  A token carries 2*H rows (K heads,
// then V heads) of D bf16 values.  Each lane owns E consecutive values of a row
// (E = 32 when D is a multiple of 32, else 16), so LANES = D/E lanes (rounded
// up to a power of two) cover a row and a warp pass covers 32/LANES rows.  The
// row data of a token is requested before its slot is computed, so the
// metadata lookups overlap the loads.  The grid is persistent (a multiple of
// the SM count) and warps stride over tokens.  The kernel is bound by issue
// slots rather than by HBM, so the per-value work is kept to a few packed
// fp32x2 operations (see below).
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
// Static modes (s per channel, quant_mode 1, from a shared-memory table; or s
// per block and kv head, quant_mode 2, read once per row; y = fl(x * fl(1/s))
// clamped to [-127, 127]):
// the relative error of y against t = x/s is at most 2^-23 + 2^-48, so
// |y - t| < 1.55e-5 for |t| <= 130 and fl(t) is within half an ulp of t
// (<= 7.7e-6 below 256).  If y lies more than 2^-15 from every half-integer,
// t and fl(t) lie strictly inside the same interval between half-integers as
// y and rne(y) = rne(fl(t)); otherwise the group takes the exact path.
// |y| >= 127 means |t| >= 126.99998, whose code is +-127 either way.
//
// Scales whose reciprocal could leave the normal range (and zero scales)
// always take the exact path.
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

template <bool V32>
__device__ __forceinline__ void load32(const uint16_t *p, uint32_t w[8]) {
    if (V32) {
        asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
              "=r"(w[6]), "=r"(w[7])
            : "l"(p));
    } else {
        const uint4 a = ld_stream_16(p), b = ld_stream_16(p + 8);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
}

template <bool V32>
__device__ __forceinline__ void store_codes32(int8_t *p, const uint32_t c[8]) {
    if (V32) {
        asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                     "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(c[5]), "r"(c[6]),
                     "r"(c[7])
                     : "memory");
    } else {
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(c[0]), "r"(c[1]),
                     "r"(c[2]), "r"(c[3])
                     : "memory");
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p + 16), "r"(c[4]),
                     "r"(c[5]), "r"(c[6]), "r"(c[7])
                     : "memory");
    }
}

__device__ __forceinline__ void store_codes16(int8_t *p, const uint32_t c[4]) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(c[0]), "r"(c[1]),
                 "r"(c[2]), "r"(c[3])
                 : "memory");
}

// E values per lane (16 or 32), LANES lanes per row, MODE 0 dynamic / 1 static
// per channel / 2 static per block,
// V32: 32-byte aligned rows (256-bit loads and stores).
template <int E, int LANES, int MODE, bool V32>
__global__ void __launch_bounds__(kWarpsPerCta * 32, MODE == 0 ? 3 : 4)
store_kernel(const StoreArgs a) {
    constexpr int W = E / 2;                  // bf16x2 words per lane per row
    constexpr int RPP = 32 / LANES;           // rows per warp pass
    constexpr int G = (E == 32) ? 2 : 4;      // passes loaded ahead
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int C = D / E;  // active lanes per row
    const int lane = threadIdx.x & 31;
    const int sub = lane / LANES;
    const int c = lane % LANES;
    const bool lane_on = c < C;

    // Shared tables.  Dynamic mode: for a bf16 row maximum amax = (1 + m/128)
    // * 2^E, s = fl(amax / 127) = fl((1 + m/128) / 127) * 2^E and
    // 1/s rounds to fl(1 / that) * 2^-E exactly, as long as both stay normal;
    // the tables hold the two fl() values for the 128 mantissas.  Static
    // per-channel mode: for each (K|V, head, channel) the bracket ends r_lo,
    // r_hi of r = fl(1/s) (as float4 {r_lo, r_lo', r_hi, r_hi'} per pair of
    // channels, one chunk of E channels per lane and row, padded by 4 floats)
    // and the clamp bound bf16(fl(127 s)) (a chunk of E bf16 per lane and row,
    // padded by 8), laid out so that the 8 lanes of each shared-memory
    // wavefront read different banks.  A scale outside the reciprocal range
    // sends the whole launch to the exact path.
    extern __shared__ float smem[];
    float *s_tab = smem;                           // dynamic mode only
    float *r_tab = smem + (MODE == 0 ? 128 : 0);
    constexpr int RCH = 2 * E + 4;                 // floats per (row, lane) chunk, static mode
    constexpr int BCH = E + 8;                     // bf16 per (row, lane) chunk, static mode
    uint16_t *b_tab = reinterpret_cast<uint16_t *>(smem + 2 * H * C * RCH);
    bool all_fast = true;
    if (MODE == 0) {
        for (int m = threadIdx.x; m < 128; m += blockDim.x) {
            const float sm = __fdiv_rn(__uint_as_float(0x3F800000u | ((uint32_t)m << 16)), 127.0f);
            s_tab[m] = sm;
            r_tab[m] = __frcp_rn(sm);
        }
        __syncthreads();
    } else if (MODE == 1) {
        int ok = 1;
        for (int idx = threadIdx.x; idx < 2 * H * D; idx += blockDim.x) {
            const float sc = idx < H * D ? ld_nc_f32(a.k_scale + idx) : ld_nc_f32(a.v_scale + (idx - H * D));
            const bool f = recip_ok(sc);
            const float r = f ? __frcp_rn(sc) : 0.0f;
            const int row = idx / D, d = idx - row * D;
            const int chunk = row * C + d / E, e = d % E;
            float *rp = r_tab + chunk * RCH + (e >> 1) * 4 + (e & 1);
            rp[0] = __fmul_rn(r, kRecipLo);
            rp[2] = __fmul_rn(r, kRecipHi);
            b_tab[chunk * BCH + e] = bf16_bound(sc);
            ok &= f;
        }
        all_fast = __syncthreads_and(ok) != 0;
    }

    const int rows = 2 * H;
    const int passes = (rows + RPP - 1) / RPP;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
    const float2 magic2 = make_float2(kMagic, kMagic);
    const float2 nmagic2 = make_float2(-kMagic, -kMagic);
    const float2 neg1 = make_float2(-1.0f, -1.0f);

    for (int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); t < a.num_tokens;
         t += nwarps) {
        for (int p0 = 0; p0 < passes; p0 += G) {
            // ---- request this group's rows ----
            uint32_t w[G][W];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                const int row = (p0 + k) * RPP + sub;
#pragma unroll
                for (int i = 0; i < W; ++i) w[k][i] = 0u;
                if (p0 + k < passes && row < rows && lane_on) {
                    const int kv = row >= H;
                    const int h = row - kv * H;
                    const uint16_t *src = (kv ? a.v_states : a.k_states) + t * a.x_tok_stride +
                                          (int64_t)h * a.x_head_stride + c * E;
                    load32<V32>(src, w[k]);
                    if (E == 32) load32<V32>(src + 16, w[k] + 8);
                }
            }
            // ---- slot of token t (warp-uniform), overlapping the loads ----
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
            // pos < 2^32 always (ctx and the token index are below 2^31):
            // floor(pos / bs) is the high word of pos * ceil(2^64 / bs)
            int64_t lb;
            if (pos >= 0 && pos <= 0xFFFFFFFFll) {
                lb = bs == 1 ? pos : (int64_t)__umul64hi(a.bs_magic, (unsigned long long)pos);
            } else {
                lb = pos / bs;
            }
            int32_t err = 0;
            int32_t blk = 0;
            if (bad_len || ctx < 0) {
                err = KVC8_DEV_BAD_LENGTH;
            } else if (lb >= MB) {
                err = KVC8_DEV_POS_BEYOND_TABLE;
            } else {
                blk = ld_nc_s32(a.block_table + (int64_t)b * MB + lb);
                if (blk < 0 || blk >= NB) err = KVC8_DEV_BAD_BLOCK_ID;
            }
            if (err != 0) {
                if (lane == 0 && p0 == 0) report(a.dev_error, err);
                break;  // warp-uniform: skip the token
            }
            const int64_t slot = pos - lb * bs;

            // ---- row scales of every pass first (independent chains) ----
            float s_rows[G], r_rows[G];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                s_rows[k] = 0.0f;
                r_rows[k] = 0.0f;
                if (MODE == 0 && p0 + k < passes) {
                    // |x| maximum: max(|a|, |b|) per bf16 half (the sign of the
                    // result is garbage and masked off before comparing words)
                    uint32_t m4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int i = 0; i < W; ++i)
                        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m4[i & 3]) : "r"(m4[i & 3]), "r"(w[k][i]));
                    const uint32_t m2 = __vmaxu2(__vmaxu2(m4[0] & 0x7FFF7FFFu, m4[1] & 0x7FFF7FFFu),
                                                 __vmaxu2(m4[2] & 0x7FFF7FFFu, m4[3] & 0x7FFF7FFFu));
                    uint32_t mag = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
                    for (int o = 1; o < LANES; o <<= 1)
                        mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, o));
                    const uint32_t ef = mag >> 7;  // bf16 exponent field of amax
                    if (ef >= 14 && ef <= 253) {   // s and 1/s normal and within recip_ok
                        const int sh = ((int)ef - 127) << 23;
                        s_rows[k] = __int_as_float(__float_as_int(s_tab[mag & 127]) + sh);
                        r_rows[k] = __int_as_float(__float_as_int(r_tab[mag & 127]) - sh);
                    } else {
                        s_rows[k] = __fdiv_rn(__uint_as_float(mag << 16), 127.0f);
                        r_rows[k] = 0.0f;  // exact path for the whole row
                    }
                } else if (MODE == 2 && p0 + k < passes) {
                    // the row's block scale; a zero reciprocal sends the row
                    // to the exact path
                    const int row = (p0 + k) * RPP + sub;
                    if (row < rows) {
                        const int kv = row >= H;
                        const int h = row - kv * H;
                        const float sb = ld_nc_f32((kv ? a.v_scale : a.k_scale) + (int64_t)blk * H + h);
                        s_rows[k] = sb;
                        r_rows[k] = recip_ok(sb) ? __frcp_rn(sb) : 0.0f;
                    }
                }
            }

            // ---- quantise and scatter ----
#pragma unroll
            for (int k = 0; k < G; ++k) {
                if (p0 + k >= passes) break;  // warp-uniform
                const int row = (p0 + k) * RPP + sub;
                const bool on = row < rows && lane_on;
                const int kv = row >= H;
                const int h = row - kv * H;
                const float s_row = s_rows[k], r_row = r_rows[k];
                // (lanes off the row read chunk 0: in bounds, their codes unused)
                const int chunk = on ? (kv * H + h) * C + c : 0;
                const float *rt = r_tab + chunk * RCH;                                   // mode 1
                const uint16_t *bt = b_tab + chunk * BCH;                                // mode 1
                const float *st = (kv ? a.v_scale : a.k_scale) + (int64_t)h * D + c * E;  // mode 1

                uint32_t cw[W / 2];  // packed codes, four per word
                uint32_t fix = 0u;   // bit q: codes 4q..4q+3 need the exact path
                const bool force_exact = (MODE == 1) ? !all_fast : (r_row == 0.0f);
                // r_lo <= r (1 - 2^-23) and r_hi >= r (1 + 2^-23) bracket every
                // value fl(x / s) can take, so when x r_lo and x r_hi round to
                // the same integer, so does fl(x / s).  Modes 0 and 2: the row's
                // pair; mode 1: each channel's, from the table.
                const float2 rlo2 = make_float2(__fmul_rn(r_row, kRecipLo), __fmul_rn(r_row, kRecipLo));
                const float2 rhi2 = make_float2(__fmul_rn(r_row, kRecipHi), __fmul_rn(r_row, kRecipHi));
                // Modes 1 and 2 clamp x to +-bf16(fl(127 s)) before the bracket
                // (one min.xorsign.abs per pair): that bound's code is +-127
                // and every larger |x| saturates, so the clamp gives
                // clamp(code(x)) and keeps |x r| below 127.5.
                const uint32_t brow = MODE == 2 ? bf16_bound(s_row) * 0x10001u : 0u;
                // Group q of four values adds its bracket gap (0 to 4, the
                // squared differences of the ends) times 8^q to flagsf: an exact
                // base-8 record of the flagged groups, kept on the FMA pipe.
                float flagsf = 0.0f;
#pragma unroll
                for (int i = 0; i < W; i += 2) {
                    uint32_t mbits[4];
                    float2 dacc = make_float2(0.0f, 0.0f);
                    uint2 b2 = make_uint2(brow, brow);
                    if (MODE == 1) b2 = *reinterpret_cast<const uint2 *>(bt + 2 * i);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        uint32_t wi = w[k][i + e];
                        float2 rlo = rlo2, rhi = rhi2;
                        if (MODE == 1) {
                            const float4 r4 = *reinterpret_cast<const float4 *>(rt + 4 * (i + e));
                            rlo = make_float2(r4.x, r4.y);
                            rhi = make_float2(r4.z, r4.w);
                        }
                        if (MODE != 0)
                            asm("min.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(wi) : "r"(wi), "r"(e ? b2.y : b2.x));
                        const float2 x2 = make_float2(__uint_as_float(wi << 16), __uint_as_float(wi & 0xFFFF0000u));
                        const float2 m2 = __ffma2_rn(x2, rlo, magic2);
                        const float2 h2 = __ffma2_rn(x2, rhi, magic2);
                        // the two ends differ by a small integer or not at all;
                        // their squared differences add up exactly, on the FMA
                        // pipe rather than the busier ALU pipe
                        const float2 dd = __ffma2_rn(m2, neg1, h2);  // h2 - m2, exact
                        dacc = __ffma2_rn(dd, dd, dacc);
                        mbits[2 * e] = __float_as_uint(m2.x);  // low byte = code
                        mbits[2 * e + 1] = __float_as_uint(m2.y);
                    }
                    cw[i / 2] = pack_lo_bytes(mbits[0], mbits[1], mbits[2], mbits[3]);
                    flagsf = __fmaf_rn(__fadd_rn(dacc.x, dacc.y), (float)(1u << (3 * (i / 2))), flagsf);
                }
                if (flagsf != 0.0f) {  // rare: which groups
                    const uint32_t u = (uint32_t)flagsf;
#pragma unroll
                    for (int q = 0; q < W / 2; ++q) fix |= ((u >> (3 * q)) & 7u) ? (1u << q) : 0u;
                }
                // Dynamic mode: the flagged groups (nearly all exact ties,
                // x/s = n + 1/2) are recomputed in registers by code_exact
                // before the store.  The static modes keep the out-of-line
                // pass after the store (fewer registers at four CTAs per SM).
                bool slow = force_exact || (MODE == 0 && fix != 0u && !(s_row >= kExactMinScale));
                if (MODE == 0 && !slow && fix != 0u) {
                    uint32_t f = fix;
                    do {
                        const int q = __ffs(f) - 1;
                        f &= f - 1u;
                        uint32_t w0 = w[k][0], w1 = w[k][1];
#pragma unroll
                        for (int g = 1; g < W / 2; ++g)
                            if (q == g) {
                                w0 = w[k][2 * g];
                                w1 = w[k][2 * g + 1];
                            }
                        const uint32_t cq = pack_lo_bytes(
                            (uint32_t)code_exact(__uint_as_float(w0 << 16), s_row, r_row),
                            (uint32_t)code_exact(__uint_as_float(w0 & 0xFFFF0000u), s_row, r_row),
                            (uint32_t)code_exact(__uint_as_float(w1 << 16), s_row, r_row),
                            (uint32_t)code_exact(__uint_as_float(w1 & 0xFFFF0000u), s_row, r_row));
#pragma unroll
                        for (int g = 0; g < W / 2; ++g)
                            if (q == g) cw[g] = cq;
                    } while (f != 0u);
                    fix = 0u;
                }
                if (slow) fix = (1u << (W / 2)) - 1u;
                if (on) {
                    int8_t *cache = kv ? a.v_cache : a.k_cache;
                    const int64_t dst_row = ((int64_t)blk * H + h) * bs + slot;
                    int8_t *dst = cache + dst_row * D + c * E;
                    if (E == 32) store_codes32<V32>(dst, cw);
                    else store_codes16(dst, cw);
                    if (MODE == 0 && c == 0) (kv ? a.v_scale : a.k_scale)[dst_row] = s_row;
                    if (fix != 0u) {
                        // rare: the flagged groups of four codes again, one by one,
                        // with one division where needed, over the codes just stored
                        const uint16_t *src = (kv ? a.v_states : a.k_states) + t * a.x_tok_stride +
                                              (int64_t)h * a.x_head_stride + c * E;
                        fix_codes<MODE>(src, dst, fix, s_row, r_row, st);
                    }
                }
            }
        }
    }
}

template <int E, int LANES, int MODE, bool V32>
cudaError_t launch_variant(const StoreArgs &a, cudaStream_t stream) {
    auto kern = store_kernel<E, LANES, MODE, V32>;
    const int C = a.g.head_dim / E;
    // mode 1: per (row, lane) chunk, 2E + 4 floats of bracket ends and E + 8 bf16 bounds
    const size_t smem = MODE == 1 ? (size_t)2 * a.g.kv_heads * C * ((2 * E + 4) * 4 + (E + 8) * 2)
                        : MODE == 0 ? sizeof(float) * 256 : 0;
    static OccupancySlots slots;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = occupancy(slots, kern, kWarpsPerCta * 32, smem, &occ);
    if (e != cudaSuccess) return e;
    const int64_t need = (a.num_tokens + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = (int64_t)sm_count() * occ;
    const int grid = (int)(need < cap ? need : cap);
    kern<<<grid, kWarpsPerCta * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int MODE, bool V32>
cudaError_t launch_mode(const StoreArgs &a, cudaStream_t stream) {
    const int D = a.g.head_dim;
    if (D % 32 == 0) {
        const int C = D / 32;  // 1..8
        if (C <= 1) return launch_variant<32, 1, MODE, V32>(a, stream);
        if (C <= 2) return launch_variant<32, 2, MODE, V32>(a, stream);
        if (C <= 4) return launch_variant<32, 4, MODE, V32>(a, stream);
        return launch_variant<32, 8, MODE, V32>(a, stream);
    }
    const int C = D / 16;  // odd multiples of 16: 1..15
    if (C <= 1) return launch_variant<16, 1, MODE, V32>(a, stream);
    if (C <= 2) return launch_variant<16, 2, MODE, V32>(a, stream);
    if (C <= 4) return launch_variant<16, 4, MODE, V32>(a, stream);
    if (C <= 8) return launch_variant<16, 8, MODE, V32>(a, stream);
    return launch_variant<16, 16, MODE, V32>(a, stream);
}

bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; }

}  // namespace

cudaError_t launch_store(const StoreArgs &a, cudaStream_t stream) {
    if (a.num_tokens <= 0) return cudaSuccess;
    const bool v32 = aligned32(a.k_states) && aligned32(a.v_states) && aligned32(a.k_cache) &&
                     aligned32(a.v_cache) && a.x_tok_stride % 16 == 0 &&
                     a.x_head_stride % 16 == 0;
    if (a.g.quant_mode == 0)
        return v32 ? launch_mode<0, true>(a, stream) : launch_mode<0, false>(a, stream);
    if (a.g.quant_mode == 1)
        return v32 ? launch_mode<1, true>(a, stream) : launch_mode<1, false>(a, stream);
    return v32 ? launch_mode<2, true>(a, stream) : launch_mode<2, false>(a, stream);
}

}  // namespace kvc8
