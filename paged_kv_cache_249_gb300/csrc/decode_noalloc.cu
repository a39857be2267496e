// decode_noalloc.cu -- pkv_paged_attention_decode_static: the decode entry
// point for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a scratch buffer: an engine that hands
// all of its device memory to the KV block pool and a caching allocator at
// start-up and forbids later allocations, a plain-C host program that has no
// device allocator of its own, or a latency-critical loop where cudaMalloc /
// cudaFree would synchronise the device.  This entry point keeps the split-K
// partials in a fixed array compiled into the library instead of a
// caller-provided workspace, and otherwise runs the same kernels as
// pkv_paged_attention_decode.
#include <mutex>

#include "pkv_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kScratchBytes = PKV_STATIC_SCRATCH_BYTES;

// Split-K partials of the allocation-free entry point.  Every GPU that loads
// the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of g_decode_scratch on device `dev` (which must be current).
// The symbol's name is only a host-side stand-in; the address must come from
// cudaGetSymbolAddress, once per device.  The address is kept for the life of
// the process: a cudaDeviceReset reloads the module and makes it stale, which
// the header states as a limit of this entry point.
pkv_status scratch_address(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p)
            return PKV_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_decode_static(
    const pkv_pool *pool, void *out, pkv_dtype out_dtype, const void *query, int num_seqs,
    int num_heads, int num_kv_heads, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, float scale, int partition_tokens,
    int flags, void *stream) {
    if (!pool || pool->magic != pkv::kPoolMagic) return PKV_ERR_INVALID_ARG;
    // A call whose partials do not fit in the fixed array is refused by the
    // decode's own size check (PKV_ERR_WORKSPACE, before any launch), which
    // sizes them for the partition it actually takes.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const pkv_status st = scratch_address(dev, &scratch);
    if (st != PKV_OK) return st;
    return pkv_paged_attention_decode(pool, out, out_dtype, query, num_seqs, num_heads,
                                      num_kv_heads, block_tables, max_blocks_per_seq, context_lens,
                                      max_context_len, scale, partition_tokens, scratch,
                                      kScratchBytes, flags, stream);
}
