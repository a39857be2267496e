// api.cu -- the C ABI declared in include/pagedkv.h: host-side validation,
// TMA descriptor set-up, variant selection and launches.  Nothing here
// allocates device memory or synchronises (except pkv_get_device_error).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Rows of one staged run of a block: the whole block up to kMaxStageRows; a
// larger block is staged in runs of that many rows, so every block size uses
// the ring geometry tuned for 16-row tiles.
int stage_rows(int block_size, int /*head_dim*/) {
    return block_size < kMaxStageRows ? block_size : kMaxStageRows;
}

// Descriptor of one pool seen as a 2-D tensor [rows = NB*Hkv*BS][head_dim],
// staged in boxes of one 128-byte slab x one run of rows with the 128-byte
// swizzle the kernels read back.
bool encode_pool_map(CUtensorMap *map, void *base, int rows, int head_dim, int block_size,
                     pkv_dtype dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int elem = dtype == PKV_F32 ? 4 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)head_dim * elem};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)stage_rows(block_size, head_dim)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype == PKV_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                         : dtype == PKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct alignas(64) MapPair {
    CUtensorMap k, v;
};
static_assert(sizeof(MapPair) == 256, "two descriptors");
static_assert(sizeof(((pkv_pool *)nullptr)->tma) == 256, "pool descriptor storage");

bool valid_geometry(int num_blocks, int block_size, int num_kv_heads, int head_dim) {
    if (num_blocks <= 0 || num_kv_heads <= 0) return false;
    if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128 &&
        block_size != 256)
        return false;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return false;
    return (long long)num_blocks * num_kv_heads * block_size < (1ll << 31);
}

}  // namespace

namespace {
thread_local cudaError_t t_last_cuda_error = cudaSuccess;
}

pkv_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return PKV_OK;
    t_last_cuda_error = e;
    return PKV_ERR_CUDA;
}

int sm_count(int device) {
    static std::atomic<int> cache[kMaxDevices];
    if (device < 0 || device >= kMaxDevices) return 148;
    int v = cache[device].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0)
        v = 148;
    cache[device].store(v, std::memory_order_relaxed);
    return v;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_version(void) { return 101; }

const char *pkv_last_cuda_error(void) {
    const cudaError_t e = t_last_cuda_error;
    return e == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(e);
}

const char *pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_DEVICE_FAULT: return "device reported a data fault";
        case PKV_ERR_OUT_OF_BLOCKS: return "no free block in the pool";
    }
    return "unknown status";
}

size_t pkv_pool_bytes(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                      pkv_dtype dtype) {
    if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    if (dtype != PKV_F32 && dtype != PKV_BF16 && dtype != PKV_F16) return 0;
    return (size_t)num_blocks * num_kv_heads * block_size * head_dim * (dtype == PKV_F32 ? 4 : 2);
}

pkv_status pkv_block_pool_init(pkv_pool *pool, int num_blocks, int block_size, int num_kv_heads,
                               int head_dim, pkv_dtype dtype, void *k_pool, void *v_pool,
                               int32_t *dev_error, int zero_fill, void *stream) {
    if (!pool || !k_pool || !v_pool) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F32 && dtype != PKV_BF16 && dtype != PKV_F16) return PKV_ERR_INVALID_ARG;
    if (num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (!valid_geometry(num_blocks, block_size, num_kv_heads, head_dim)) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(dev_error, 4))
        return PKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != PKV_OK) return PKV_ERR_CUDA;
    MapPair maps;
    std::memset(&maps, 0, sizeof(maps));
    const int rows = num_blocks * num_kv_heads * block_size;
    if (!encode_pool_map(&maps.k, k_pool, rows, head_dim, block_size, dtype) ||
        !encode_pool_map(&maps.v, v_pool, rows, head_dim, block_size, dtype))
        return PKV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (zero_fill) {
        const size_t bytes = pkv_pool_bytes(num_blocks, block_size, num_kv_heads, head_dim, dtype);
        if (cuda_status(cudaMemsetAsync(k_pool, 0, bytes, st)) != PKV_OK ||
            cuda_status(cudaMemsetAsync(v_pool, 0, bytes, st)) != PKV_OK)
            return PKV_ERR_CUDA;
        if (dev_error && cuda_status(cudaMemsetAsync(dev_error, 0, sizeof(int32_t), st)) != PKV_OK)
            return PKV_ERR_CUDA;
    }
    pool->num_blocks = num_blocks;
    pool->block_size = block_size;
    pool->num_kv_heads = num_kv_heads;
    pool->head_dim = head_dim;
    pool->dtype = dtype;
    pool->device = dev;
    pool->layout = 0;
    pool->num_seqs = 0;
    pool->k_pool = k_pool;
    pool->v_pool = v_pool;
    pool->dev_error = dev_error;
    std::memcpy(pool->tma, &maps, sizeof(maps));
    pool->magic = kPoolMagic;
    return PKV_OK;
}

pkv_status pkv_block_table_upload(int32_t *dev_block_tables, const int32_t *host_block_tables,
                                  int num_seqs, int max_blocks_per_seq, int num_blocks,
                                  void *stream) {
    if (num_seqs < 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!dev_block_tables || !host_block_tables) return PKV_ERR_INVALID_ARG;
    if (!aligned(dev_block_tables, 4) || !aligned(host_block_tables, 4)) return PKV_ERR_INVALID_ARG;
    const size_t n = (size_t)num_seqs * max_blocks_per_seq;
    if (num_blocks > 0)
        for (size_t i = 0; i < n; ++i)
            if (host_block_tables[i] >= num_blocks) return PKV_ERR_INVALID_ARG;
    return cuda_status(cudaMemcpyAsync(dev_block_tables, host_block_tables, n * sizeof(int32_t),
                                       cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_reshape_and_cache(const pkv_pool *pool, const void *key, const void *value,
                                 const int64_t *slot_mapping, int num_tokens, void *stream) {
    if (!pool || pool->magic != kPoolMagic || pool->layout != 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!key || !value || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != PKV_OK) return PKV_ERR_CUDA;
    if (dev != pool->device) return PKV_ERR_INVALID_ARG;
    return launch_reshape_and_cache(*pool, key, value, slot_mapping, num_tokens,
                                    static_cast<cudaStream_t>(stream));
}

// 0 = automatic.  Partitions cost one CTA start-up each (block-table and
// first-tile latency), so take the longest partition (2048, 1024 or 512
// tokens) that still gives about nine waves of CTAs (ctas_per_sm resident
// per SM); no split when the whole context fits in one partition.  `units`
// is num_seqs * num_kv_heads; sms <= 0 sizes for the smallest automatic
// choice.
static int resolve_partition(int partition_tokens, int max_context_len, long long units, int sms,
                             int ctas_per_sm = 3) {
    if (partition_tokens != 0) return partition_tokens;
    if (max_context_len <= kAutoPartitionTokens) return -1;
    if (sms <= 0) return kAutoPartitionTokens;
    const long long target = 9ll * ctas_per_sm * sms;
    for (int pt = 2048; pt > kAutoPartitionTokens; pt /= 2)
        if (units * ((max_context_len + pt - 1) / pt) >= target) return pt;
    return kAutoPartitionTokens;
}

size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                  int partition_tokens) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len <= 0) return 0;
    const int pt = resolve_partition(partition_tokens, max_context_len, 0, 0);
    if (pt <= 0) return 0;
    const size_t parts = ((size_t)max_context_len + pt - 1) / pt;
    if (parts <= 1) return 0;
    const size_t rows = (size_t)num_seqs * num_heads * parts;
    return round_up(rows * head_dim * sizeof(float), 256) + round_up(rows * sizeof(float), 256);
}

static pkv_status decode_impl(const pkv_pool *pool, bool contig, void *out, pkv_dtype out_dtype,
                              const void *query, int num_seqs, int num_heads, int num_kv_heads,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int max_context_len, float scale,
                              int partition_tokens, void *workspace, size_t workspace_bytes,
                              int flags, void *stream) {
    if (!pool || pool->magic != kPoolMagic || pool->layout != (contig ? 1 : 0))
        return PKV_ERR_INVALID_ARG;
    if (contig && num_seqs > pool->num_seqs) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
        max_context_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_kv_heads != pool->num_kv_heads || num_heads % num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16 && out_dtype != PKV_F16)
        return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (flags != PKV_DECODE_PATH_AUTO && flags != PKV_DECODE_PATH_FMA &&
        flags != PKV_DECODE_PATH_MMA)
        return PKV_ERR_INVALID_ARG;
    if (partition_tokens < -1 || partition_tokens > kMaxPartitionTokens ||
        (partition_tokens > 0 && partition_tokens % pool->block_size != 0))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !query || (!block_tables && !contig) || !context_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(query, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (group > kMaxGroup) return PKV_ERR_UNSUPPORTED;
    if (num_kv_heads > 65535 || num_seqs > 65535) return PKV_ERR_UNSUPPORTED;  // grid y
    const bool half16 = pool->dtype != PKV_F32;  // bf16 or fp16: 16-bit tensor-core tiles
    // fp32 storage takes TF32 tiles (three products each) for the larger groups
    bool mma = half16 ? group >= 4 : group >= tf32_min_group(pool->head_dim);
    if (flags == PKV_DECODE_PATH_FMA) mma = false;
    if (flags == PKV_DECODE_PATH_MMA) {
        if (!half16 && pool->head_dim > 128) return PKV_ERR_UNSUPPORTED;
        mma = true;
    }
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != PKV_OK) return PKV_ERR_CUDA;
    if (dev != pool->device) return PKV_ERR_INVALID_ARG;

    // The kernel works in staged runs of U rows: a block of BS > 16 rows is
    // 2^unit_shift runs, and partitions (whole blocks) are whole runs.
    const int BS = pool->block_size, U = stage_rows(BS, pool->head_dim);
    int unit_shift = 0;
    while ((U << unit_shift) < BS) ++unit_shift;
    if (((long long)max_blocks_per_seq << unit_shift) >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;
    const long long table_cap = (long long)max_blocks_per_seq * BS;
    const int ctx_cap = (int)(table_cap < max_context_len ? table_cap : max_context_len);
    const int cap_blocks = (ctx_cap + U - 1) / U;  // runs

    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = query;
    a.out = out;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.dev_error = pool->dev_error;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    // the CUDA-core path takes at most kFmaRowsMax rows of a group per CTA
    a.row_split = mma ? 1 : (group + kFmaRowsMax - 1) / kFmaRowsMax;
    a.rows_per_cta = (group + a.row_split - 1) / a.row_split;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = pool->num_blocks;
    a.ctx_cap = ctx_cap;
    a.out_dtype = out_dtype;
    a.contig = contig ? 1 : 0;
    a.unit_shift = unit_shift;
    a.scale_log2 = scale * 1.4426950408889634f;

    // the tensor-core kernel of a 256-wide head holds 254 registers a thread:
    // two CTAs per SM instead of three
    const int ctas_per_sm = (pool->head_dim == 256 && mma) ? 2 : 3;
    const int pt = resolve_partition(partition_tokens, ctx_cap,
                                     (long long)num_seqs * num_kv_heads * a.row_split, sm_count(dev),
                                     ctas_per_sm);
    int parts = 1;
    if (pt > 0) {
        a.part_blocks = pt / U;
        parts = (cap_blocks + a.part_blocks - 1) / a.part_blocks;
        if (parts < 1) parts = 1;
    }
    if (parts <= 1) {
        a.part_blocks = cap_blocks > 0 ? cap_blocks : 1;
        parts = 1;
    } else {
        if (parts > 65535) return PKV_ERR_UNSUPPORTED;
        const size_t rows = (size_t)num_seqs * num_heads * parts;
        const size_t o_bytes = round_up(rows * pool->head_dim * sizeof(float), 256);
        const size_t need = o_bytes + round_up(rows * sizeof(float), 256);
        if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return PKV_ERR_INVALID_ARG;
        a.ws_o = static_cast<float *>(workspace);
        a.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_bytes);
    }
    a.num_parts = parts;

    MapPair maps;
    std::memcpy(&maps, pool->tma, sizeof(maps));
    DecodeLaunch L;
    L.tmk = &maps.k;
    L.tmv = &maps.v;
    L.args = a;
    L.num_seqs = num_seqs;
    L.head_dim = pool->head_dim;
    L.block_size = U;
    L.runs = unit_shift > 0;
    int gp = 1;
    while (gp < a.rows_per_cta) gp <<= 1;
    L.group_pad = gp;
    L.mma = mma;
    L.stream = static_cast<cudaStream_t>(stream);
    L.device = dev;

    pkv_status st;
    const int hd = pool->head_dim;
    if (pool->dtype == PKV_BF16)
        st = hd == 64 ? launch_decode_bf16_d64(L)
                      : (hd == 128 ? launch_decode_bf16_d128(L) : launch_decode_bf16_d256(L));
    else if (pool->dtype == PKV_F16)
        st = hd == 64 ? launch_decode_f16_d64(L)
                      : (hd == 128 ? launch_decode_f16_d128(L) : launch_decode_f16_d256(L));
    else
        st = hd == 64 ? launch_decode_f32_d64(L)
                      : (hd == 128 ? launch_decode_f32_d128(L) : PKV_ERR_UNSUPPORTED);
    if (st != PKV_OK || parts <= 1) return st;
    return launch_lse_combine(a, num_seqs, pool->head_dim, U, L.stream);
}

pkv_status pkv_paged_attention_decode(const pkv_pool *pool, void *out, pkv_dtype out_dtype,
                                      const void *query, int num_seqs, int num_heads,
                                      int num_kv_heads, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *context_lens,
                                      int max_context_len, float scale, int partition_tokens,
                                      void *workspace, size_t workspace_bytes, int flags,
                                      void *stream) {
    return decode_impl(pool, false, out, out_dtype, query, num_seqs, num_heads, num_kv_heads,
                       block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                       partition_tokens, workspace, workspace_bytes, flags, stream);
}

pkv_status pkv_contiguous_cache_init(pkv_pool *cache, int num_seqs, int capacity,
                                     int num_kv_heads, int head_dim, pkv_dtype dtype,
                                     void *k_cache, void *v_cache, int32_t *dev_error,
                                     int zero_fill, void *stream) {
    const int BS = 16;
    if (!cache || num_seqs <= 0 || capacity <= 0 || capacity % BS != 0) return PKV_ERR_INVALID_ARG;
    const long long rows = (long long)num_seqs * num_kv_heads * capacity;
    if (rows >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;
    // the same descriptor as a pool whose "blocks" are the runs of 16 rows
    const pkv_status st = pkv_block_pool_init(cache, (int)(rows / ((long long)num_kv_heads * BS)),
                                              BS, num_kv_heads, head_dim, dtype, k_cache, v_cache,
                                              dev_error, zero_fill, stream);
    if (st != PKV_OK) return st;
    cache->layout = 1;
    cache->num_seqs = num_seqs;
    cache->num_blocks = capacity / BS;  // blocks per (sequence, kv head) run
    return PKV_OK;
}

pkv_status pkv_contiguous_attention_decode(const pkv_pool *cache, void *out, pkv_dtype out_dtype,
                                           const void *query, int num_seqs, int num_heads,
                                           int num_kv_heads, const int32_t *context_lens,
                                           int max_context_len, float scale,
                                           int partition_tokens, void *workspace,
                                           size_t workspace_bytes, int flags, void *stream) {
    if (!cache) return PKV_ERR_INVALID_ARG;
    return decode_impl(cache, true, out, out_dtype, query, num_seqs, num_heads, num_kv_heads,
                       nullptr, cache->num_blocks, context_lens, max_context_len, scale,
                       partition_tokens, workspace, workspace_bytes, flags, stream);
}

pkv_status pkv_copy_blocks(const pkv_pool *pool, const int32_t *src, const int32_t *dst,
                           int num_pairs, void *stream) {
    if (!pool || pool->magic != kPoolMagic || pool->layout != 0 || num_pairs < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!src || !dst || !aligned(src, 4) || !aligned(dst, 4)) return PKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != PKV_OK) return PKV_ERR_CUDA;
    if (dev != pool->device) return PKV_ERR_INVALID_ARG;
    return launch_copy_blocks(*pool, src, dst, num_pairs, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_check_bounded_wait(const pkv_pool *pool, long long limit_ns, void *stream) {
    if (!pool || pool->magic != kPoolMagic || !pool->dev_error) return PKV_ERR_INVALID_ARG;
    if (limit_ns < 1000 || limit_ns > 2000000000ll) return PKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != PKV_OK) return PKV_ERR_CUDA;
    if (dev != pool->device) return PKV_ERR_INVALID_ARG;
    return launch_bounded_wait_check(pool->dev_error, limit_ns, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_get_device_error(const pkv_pool *pool, void *stream, uint32_t *fault_bits) {
    if (fault_bits) *fault_bits = 0;
    if (!pool || pool->magic != kPoolMagic) return PKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!pool->dev_error) return cuda_status(cudaStreamSynchronize(st));
    int32_t v = 0;
    if (cuda_status(cudaMemcpyAsync(&v, pool->dev_error, sizeof(v), cudaMemcpyDeviceToHost, st)) !=
            PKV_OK ||
        cuda_status(cudaStreamSynchronize(st)) != PKV_OK)
        return PKV_ERR_CUDA;
    if (v != 0) {
        if (cuda_status(cudaMemsetAsync(pool->dev_error, 0, sizeof(int32_t), st)) != PKV_OK ||
            cuda_status(cudaStreamSynchronize(st)) != PKV_OK)
            return PKV_ERR_CUDA;
    }
    if (fault_bits) *fault_bits = (uint32_t)v;
    return v != 0 ? PKV_ERR_DEVICE_FAULT : PKV_OK;
}

}  // extern "C"
