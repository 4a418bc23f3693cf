// kvc8_noalloc.cu -- kvc8_dequant_gather_noalloc: the dequant-gather for
// callers that cannot hand the library a workspace.
//
// Some callers have no way to allocate device memory at the point where they
// gather: a plugin running inside a host runtime that owns every device
// allocation and exposes no allocator to its plugins, or a serving loop that
// must not allocate after start-up (an allocation can synchronise the device
// and break a memory plan fixed in advance).  For them the gather's plan --
// per-sequence output offsets, the tile prefix and the work counter -- lives
// in a fixed array compiled into this library instead of a caller workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds one copy, for the life of the process.  Host code may not use
// the variable's name as a device address (on the host it names a stand-in
// object), so the address is looked up with cudaGetSymbolAddress once per
// device, with that device current, and passed to the kernels.  All calls on a
// device share the one array: the plan kernel rewrites every field it uses
// (including the work counter, which it zeroes) on each call, but two calls
// whose work overlaps on the GPU race on it.
#include <mutex>

#include "kvc8_internal.cuh"

namespace kvc8 {
namespace {

// plan_bytes(KVC8_NOALLOC_MAX_SEQS), rounded up to 256 bytes
constexpr size_t kNoallocScratchBytes =
    ((256 + ((8u * KVC8_NOALLOC_MAX_SEQS + 255) / 256) * 256 +
      ((4u * (KVC8_NOALLOC_MAX_SEQS + 1) + 255) / 256) * 256) + 255) / 256 * 256;

static __device__ __align__(256) unsigned char g_gather_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of this device's scratch array (looked up on first use).
cudaError_t scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gather_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace kvc8

using namespace kvc8;

extern "C" kvc8_status kvc8_dequant_gather_noalloc(
    const kvc8_geom *g, const int8_t *key_cache, const int8_t *value_cache,
    const float *key_scale, const float *value_scale, const int32_t *block_table,
    const int32_t *context_lengths, const int64_t *context_seq_offset, void *key_out,
    void *value_out, int64_t out_rows, int64_t out_tok_stride, int64_t out_head_stride,
    int32_t *dev_error, cudaStream_t stream) {
    // The checks of kvc8_dequant_gather, then the size limit of the array.
    kvc8_status st = check_geom(g);
    if (st != KVC8_OK) return st;
    if (g->num_seqs > KVC8_NOALLOC_MAX_SEQS || plan_bytes(g->num_seqs) > kNoallocScratchBytes)
        return KVC8_ERR_UNSUPPORTED;
    // The set-up comes before the early return, so that a call with
    // num_seqs = 0 at start-up prepares the device without doing any work.
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return KVC8_ERR_CUDA;
    if (g->num_seqs == 0) return KVC8_OK;
    st = check_gather_args(g, key_cache, value_cache, key_scale, value_scale, block_table,
                           context_lengths, key_out, value_out, out_rows, out_tok_stride,
                           out_head_stride);
    if (st != KVC8_OK) return st;
    if (launch_plan(*g, context_lengths, context_seq_offset, nullptr, scratch, dev_error,
                    stream) != cudaSuccess)
        return KVC8_ERR_CUDA;
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
    a.plan = scratch;
    a.dev_error = dev_error;
    return launch_gather(a, /*use_pdl=*/true, stream) == cudaSuccess ? KVC8_OK : KVC8_ERR_CUDA;
}
