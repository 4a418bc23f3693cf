// kvc8_store.cu -- quantise new bf16 K/V tokens to int8 and scatter them into
// the paged cache (MojoStorePagedKVCacheC8 in mojo_opset pull request #379,
// "feat: [MLU] add mlu experimental ops; fix post norm bug").
//
// Work decomposition: one warp per token.  A token carries 2*H rows (K heads,
// then V heads) of D bf16 values.  A row is split into D/8 chunks of 16 bytes,
// one chunk per lane, so a pass of the warp covers 32/LANES rows; all passes of
// a token (up to 8) are loaded before any is converted, so every lane keeps up
// to 128 bytes of loads in flight.  The grid is persistent (a multiple of the
// SM count) and warps stride over tokens.
//
// Rounding is bit-exact with the definition q = clamp(rne(x / s), -127, 127)
// (one IEEE fp32 division).  Per element the kernel first evaluates
// y = x * fl(1/s); the relative error of y against the exact quotient t = x/s
// is at most 2^-23 + 2^-48, i.e. below 2^-15 for |t| <= 256.  Where y is more
// than 2^-13 away from every half-integer, t and fl(t) lie strictly inside the
// same interval between half-integers as y, so rne(y) = rne(fl(t)) and the
// fast path is exact.  Inside that window (and for scales whose reciprocal
// could leave the normal range) the element is recomputed with the IEEE
// division __fdiv_rn and __float2int_rn.  Values with |y| > 200 saturate
// (then |t| > 199.99 and the code is +-127 either way).
#include "kvc8_internal.cuh"

namespace kvc8 {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kGroup = 8;  // row passes loaded before converting

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

// Fast path: returns the code of y = x * r and sets `near` when y is within
// 2^-13 of a half-integer (the exact path must decide).
__device__ __forceinline__ int quant_fast(float x, float r, bool &near) {
    const float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer (RNE)
    float y = __fmul_rn(x, r);
    y = fminf(fmaxf(y, -200.0f), 200.0f);
    float m = __fadd_rn(y, kMagic);
    float k = __fsub_rn(m, kMagic);
    float d = __fsub_rn(y, k);
    near = fabsf(d) >= 0.4998779296875f;  // 0.5 - 2^-13
    int q = __float_as_int(m) - 0x4B400000;
    return min(127, max(-127, q));
}

__device__ __forceinline__ uint32_t pack4(int q0, int q1, int q2, int q3) {
    uint32_t t01 = __byte_perm((uint32_t)q0, (uint32_t)q1, 0x0040);
    uint32_t t23 = __byte_perm((uint32_t)q2, (uint32_t)q3, 0x0040);
    return __byte_perm(t01, t23, 0x5410);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Largest b in [0, B] with cu[b] <= t (cu[0] = 0 <= t).
__device__ __forceinline__ int seq_of_token(const int32_t *cu, int B, int64_t t) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((int64_t)ld_nc_s32(cu + mid) <= t) lo = mid; else hi = mid;
    }
    return lo;
}

template <int LANES, int MODE>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
store_kernel(const StoreArgs a) {
    constexpr int RPP = 32 / LANES;  // rows per warp pass
    const int H = a.g.kv_heads, D = a.g.head_dim, bs = a.g.block_size;
    const int B = a.g.num_seqs, MB = a.g.max_blocks_per_seq, NB = a.g.num_blocks;
    const int C = D >> 3;  // 16-byte chunks per row
    const int lane = threadIdx.x & 31;
    const int sub = lane / LANES;
    const int c = lane % LANES;
    const bool lane_on = c < C;

    // Static mode: per-(kv, head, channel) scale and reciprocal tables in shared
    // memory, [2][H][D] each; a zero reciprocal marks "use the exact path".
    extern __shared__ float smem[];
    float *s_tab = smem;
    float *r_tab = smem + 2 * H * D;
    if (MODE == 1) {
        for (int i = threadIdx.x; i < 2 * H * D; i += blockDim.x) {
            float s = i < H * D ? ld_nc_f32(a.k_scale + i) : ld_nc_f32(a.v_scale + (i - H * D));
            s_tab[i] = s;
            r_tab[i] = recip_ok(s) ? __frcp_rn(s) : 0.0f;
        }
        __syncthreads();
    }

    const int rows = 2 * H;
    const int passes = (rows + RPP - 1) / RPP;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
    for (int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); t < a.num_tokens;
         t += nwarps) {
        // ---- slot of token t (warp-uniform) ----
        int b;
        int64_t i_in_seq;
        bool bad_len = false;
        if (a.cu_q_lens != nullptr) {
            b = seq_of_token(a.cu_q_lens, B, t);
            int64_t first = ld_nc_s32(a.cu_q_lens + b);
            int64_t next = ld_nc_s32(a.cu_q_lens + b + 1);
            i_in_seq = t - first;
            bad_len = !(first <= t && t < next);
        } else {
            b = (int)t;
            i_in_seq = 0;
        }
        int64_t ctx = ld_nc_s32(a.context_kv_lens + b);
        int64_t pos = ctx + i_in_seq;
        int64_t lb = pos / bs;
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
            if (lane == 0) report(a.dev_error, err);
            continue;
        }
        const int64_t slot = pos - lb * bs;

        for (int p0 = 0; p0 < passes; p0 += kGroup) {
            uint4 v[kGroup];
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                const int row = (p0 + k) * RPP + sub;
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                if (p0 + k < passes && row < rows && lane_on) {
                    const int kv = row >= H;
                    const int h = row - kv * H;
                    const uint16_t *src = (kv ? a.v_states : a.k_states) + t * a.x_tok_stride +
                                          (int64_t)h * a.x_head_stride + c * 8;
                    v[k] = ld_stream_16(src);
                }
            }
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                if (p0 + k >= passes) break;  // warp-uniform
                const int row = (p0 + k) * RPP + sub;
                const bool row_on = row < rows;
                const int kv = row >= H;
                const int h = row - kv * H;
                const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                float x[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x[2 * j] = bf16_lo(w[j]);
                    x[2 * j + 1] = bf16_hi(w[j]);
                }
                int q[8];
                float s_row = 0.0f;
                unsigned near_mask = 0;
                if (MODE == 0) {
                    // |x| ordering equals the ordering of the magnitude bits.
                    uint32_t m2 = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                           __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
                    uint32_t mag = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
                    for (int o = 1; o < LANES; o <<= 1)
                        mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, o));
                    const float amax = __uint_as_float(mag << 16);
                    s_row = __fdiv_rn(amax, 127.0f);
                    const bool fast = recip_ok(s_row);
                    const float r = fast ? __frcp_rn(s_row) : 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        bool nr;
                        q[j] = quant_fast(x[j], r, nr);
                        near_mask |= (unsigned)(nr || !fast) << j;
                    }
                    if (near_mask) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (near_mask & (1u << j)) q[j] = quant_exact(x[j], s_row);
                    }
                } else {
                    const int base = (kv * H + h) * D + c * 8;
                    float r[8];
                    if (lane_on && row_on) {
                        const float4 r0 = *reinterpret_cast<const float4 *>(r_tab + base);
                        const float4 r1 = *reinterpret_cast<const float4 *>(r_tab + base + 4);
                        r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
                        r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) r[j] = 1.0f;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        bool nr;
                        q[j] = quant_fast(x[j], r[j], nr);
                        near_mask |= (unsigned)(nr || r[j] == 0.0f) << j;
                    }
                    if (near_mask && lane_on && row_on) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (near_mask & (1u << j)) q[j] = quant_exact(x[j], s_tab[base + j]);
                    }
                }
                if (row_on && lane_on) {
                    int8_t *cache = kv ? a.v_cache : a.k_cache;
                    const int64_t dst_row = ((int64_t)blk * H + h) * bs + slot;
                    st_8(cache + dst_row * D + c * 8, pack4(q[0], q[1], q[2], q[3]),
                         pack4(q[4], q[5], q[6], q[7]));
                    if (MODE == 0 && c == 0) (kv ? a.v_scale : a.k_scale)[dst_row] = s_row;
                }
            }
        }
    }
}

template <int LANES, int MODE>
cudaError_t launch_variant(const StoreArgs &a, cudaStream_t stream) {
    auto kern = store_kernel<LANES, MODE>;
    const size_t smem = MODE == 1 ? sizeof(float) * 4 * a.g.kv_heads * a.g.head_dim : 0;
    static int dev_cached[64];
    static int occ_cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int occ = 0;
    if (MODE == 0 && dev < 64 && dev_cached[dev]) {
        occ = occ_cached[dev];
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWarpsPerCta * 32, smem);
        if (e != cudaSuccess) return e;
        if (MODE == 0 && dev < 64) {
            occ_cached[dev] = occ;
            dev_cached[dev] = 1;
        }
    }
    if (occ < 1) occ = 1;
    const int64_t need = (a.num_tokens + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = (int64_t)sm_count() * occ;
    const int grid = (int)(need < cap ? need : cap);
    kern<<<grid, kWarpsPerCta * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const StoreArgs &a, cudaStream_t stream) {
    const int C = a.g.head_dim / 8;
    if (C <= 2) return launch_variant<2, MODE>(a, stream);
    if (C <= 4) return launch_variant<4, MODE>(a, stream);
    if (C <= 8) return launch_variant<8, MODE>(a, stream);
    if (C <= 16) return launch_variant<16, MODE>(a, stream);
    return launch_variant<32, MODE>(a, stream);
}

}  // namespace

cudaError_t launch_store(const StoreArgs &a, cudaStream_t stream) {
    if (a.num_tokens <= 0) return cudaSuccess;
    return a.g.quant_mode == 0 ? launch_mode<0>(a, stream) : launch_mode<1>(a, stream);
}

}  // namespace kvc8
