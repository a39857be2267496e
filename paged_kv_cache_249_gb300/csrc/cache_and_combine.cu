// cache_and_combine.cu -- the cache-write scatter and the log-sum-exp combine
// of a partitioned decode.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// ------------------------------------------------------ reshape_and_cache
//
// The KV cache grows by one token per decode iteration (Qualiteg, "About
// PagedAttention for LLM serving", "Characteristics of Autoregressive
// Models..."); the new token's K and V rows go to the slot its block table
// assigns (same page, the section on logical and physical blocks).  One thread
// moves one 16-byte chunk of one (token, kv head) row of K and of V, so a
// warp writes whole 128-byte lines of the destination row.
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                             const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                             const int64_t *__restrict__ slot_mapping, int num_tokens,
                             int num_kv_heads, int block_size, int chunks_per_row,
                             long long num_slots, int32_t *dev_error) {
    griddep_launch();  // a decode launched behind this kernel may start its set-up
    const long long per_token = (long long)num_kv_heads * chunks_per_row;
    const long long total = per_token * num_tokens;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(idx / per_token);
        const int rem = (int)(idx - (long long)t * per_token);
        const int h = rem / chunks_per_row, c = rem % chunks_per_row;
        const long long slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (rem == 0) raise_fault(dev_error, PKV_FAULT_SLOT);
            continue;
        }
        const long long blk = slot / block_size, off = slot % block_size;
        const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
        const size_t src = (size_t)idx;  // key is [T][Hkv][D] contiguous
        k_pool[dst] = __ldg(key + src);
        v_pool[dst] = __ldg(value + src);
    }
}

pkv_status launch_reshape_and_cache(const pkv_pool &pool, const void *key, const void *value,
                                    const int64_t *slot_mapping, int num_tokens,
                                    cudaStream_t stream) {
    if (num_tokens == 0) return PKV_OK;
    const int elem = pool.dtype == PKV_F32 ? 4 : 2;
    const int chunks = pool.head_dim * elem / 16;
    const long long total = (long long)num_tokens * pool.num_kv_heads * chunks;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)sm_count(pool.device) * 8;
    if (blocks > cap) blocks = cap;
    reshape_and_cache_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<uint4 *>(pool.k_pool), static_cast<uint4 *>(pool.v_pool),
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), slot_mapping,
        num_tokens, pool.num_kv_heads, pool.block_size, chunks,
        (long long)pool.num_blocks * pool.block_size, pool.dev_error);
    return cuda_status(cudaGetLastError());
}

// ------------------------------------------------------------ copy_blocks
//
// Copy-on-write of shared blocks: whole physical blocks (all kv heads) of K
// and V, one 16-byte chunk per thread.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                       const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                       int num_pairs, long long chunks_per_block, int num_blocks,
                       int32_t *dev_error) {
    const long long total = chunks_per_block * num_pairs;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(idx / chunks_per_block);
        const long long c = idx - (long long)p * chunks_per_block;
        const int s = __ldg(src + p), d = __ldg(dst + p);
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
            if (c == 0) raise_fault(dev_error, PKV_FAULT_BLOCK_ID);
            continue;
        }
        k_pool[(size_t)d * chunks_per_block + c] = k_pool[(size_t)s * chunks_per_block + c];
        v_pool[(size_t)d * chunks_per_block + c] = v_pool[(size_t)s * chunks_per_block + c];
    }
}

pkv_status launch_copy_blocks(const pkv_pool &pool, const int32_t *src, const int32_t *dst,
                              int num_pairs, cudaStream_t stream) {
    const int elem = pool.dtype == PKV_F32 ? 4 : 2;
    const long long chunks =
        (long long)pool.num_kv_heads * pool.block_size * pool.head_dim * elem / 16;
    long long blocks = (chunks * num_pairs + 255) / 256;
    const long long cap = (long long)sm_count(pool.device) * 8;
    if (blocks > cap) blocks = cap;
    copy_blocks_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<uint4 *>(pool.k_pool), static_cast<uint4 *>(pool.v_pool), src, dst, num_pairs,
        chunks, pool.num_blocks, pool.dev_error);
    return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------- bounded-wait check
//
// Every pipeline wait in the decode kernels is bounded: past its limit the
// kernel records PKV_FAULT_TIMEOUT in the caller's error word and stops, so
// a copy that never lands cannot hang the GPU.  This kernel runs that same
// bounded wait on an mbarrier nothing will ever arrive at, with the caller's
// (short) limit, so a test or a deployment can watch the path work: the
// wait gives up, the fault bit is set, and the context stays usable.
__global__ void bounded_wait_check_kernel(int32_t *dev_error, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // phase 0 never completes: no thread arrives and no copy is in flight
    const bool done = __all_sync(0xffffffffu, mbar_wait_for(&bar, 0, limit_ns));
    if (!done && threadIdx.x == 0) raise_fault(dev_error, PKV_FAULT_TIMEOUT);
}

pkv_status launch_bounded_wait_check(int32_t *dev_error, long long limit_ns, cudaStream_t stream) {
    bounded_wait_check_kernel<<<1, 32, 0, stream>>>(dev_error, (unsigned long long)limit_ns);
    return cuda_status(cudaGetLastError());
}

// ------------------------------------------------------------ lse_combine
//
// A context split into partitions p = 0..P-1 has, per query head, normalised
// partial outputs o_p and their log2-sum-exp lse_p.  The full softmax result
// is sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M) with M = max_p lse_p,
// which is exact: the partitions' exponentials share one max-free total.
// Two kernels, chosen on the host by the number of partitions of the
// longest allowed context.
constexpr int kCombThreads = 256;
constexpr int kCombChunk = 1024;
constexpr int kCombDirect = 16;  // up to this many partitions, the direct loop is faster

// Parts of (sequence, head) blockIdx.x: their count (0 or 1: nothing to do)
// and the max of their log2-sum-exps over the CTA.
struct CombRow {
    int sh, nparts;
    const float *lse, *po;
};

__device__ __forceinline__ CombRow comb_row(const DecodeArgs &a, int head_dim, int block_size,
                                            int sh) {
    CombRow r;
    r.sh = sh;  // s * H + h
    const int s = r.sh / a.num_heads;
    int ctx = __ldg(a.context_lens + s);
    ctx = ctx < 0 ? 0 : (ctx > a.ctx_cap ? a.ctx_cap : ctx);
    const int nblk = (ctx + block_size - 1) / block_size;
    r.nparts = (nblk + a.part_blocks - 1) / a.part_blocks;
    r.lse = a.ws_lse + (size_t)r.sh * a.num_parts;
    r.po = a.ws_o + (size_t)r.sh * a.num_parts * head_dim;
    return r;
}

__device__ __forceinline__ float comb_max(const CombRow &r, float *red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float M = -CUDART_INF_F;
    for (int p = tid; p < r.nparts; p += kCombThreads) M = fmaxf(M, r.lse[p]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kCombThreads / 32; ++w) M = fmaxf(M, red[w]);
    return M;
}

__device__ __forceinline__ void comb_store(const DecodeArgs &a, size_t oi, float res) {
    store_out(a.out, oi, res, a.out_dtype);
}

// Few partitions: one warp per (sequence, head), each lane owning D/32
// adjacent columns.  Every load the row needs (its context length, the
// log2-sum-exps and partial outputs of all kCombDirect possible parts) is
// issued before any is used, so the row costs one round trip to memory;
// parts past the sequence's own count are loaded but never used.
template <int PER>
__global__ void __launch_bounds__(256)
    lse_combine_kernel(const DecodeArgs a, int block_size, int rows) {
    constexpr int D = PER * 32;
    griddep_wait();  // the decode grid's partials are complete
    const int sh = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (sh >= rows) return;
    const int P = a.num_parts;  // <= kCombDirect
    int ctx = __ldg(a.context_lens + sh / a.num_heads);
    const float lse_l = lane < P ? a.ws_lse[(size_t)sh * P + lane] : -CUDART_INF_F;
    const float *po = a.ws_o + (size_t)sh * P * D + lane * PER;
    float v[kCombDirect][PER];
#pragma unroll
    for (int p = 0; p < kCombDirect; ++p) {
        if (p < P) {
            if constexpr (PER == 8) {
                const float4 x = *reinterpret_cast<const float4 *>(po + (size_t)p * D);
                const float4 y = *reinterpret_cast<const float4 *>(po + (size_t)p * D + 4);
                v[p][0] = x.x, v[p][1] = x.y, v[p][2] = x.z, v[p][3] = x.w;
                v[p][4] = y.x, v[p][5] = y.y, v[p][6] = y.z, v[p][7] = y.w;
            } else if constexpr (PER == 4) {
                const float4 x = *reinterpret_cast<const float4 *>(po + (size_t)p * D);
                v[p][0] = x.x, v[p][1] = x.y, v[p][2] = x.z, v[p][3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2 *>(po + (size_t)p * D);
                v[p][0] = x.x, v[p][1] = x.y;
            }
        }
    }
    ctx = ctx < 0 ? 0 : (ctx > a.ctx_cap ? a.ctx_cap : ctx);
    const int nblk = (ctx + block_size - 1) / block_size;
    const int nparts = (nblk + a.part_blocks - 1) / a.part_blocks;
    if (nparts <= 1) return;  // the decode kernel wrote this row directly
    float M = lane < nparts ? lse_l : -CUDART_INF_F;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w_l = lane < nparts && M != -CUDART_INF_F ? fast_exp2(lse_l - M) : 0.f;
    float den = w_l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    float num[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) num[j] = 0.f;
#pragma unroll
    for (int p = 0; p < kCombDirect; ++p) {
        const float w = __shfl_sync(0xffffffffu, w_l, p);
        if (p < nparts) {
#pragma unroll
            for (int j = 0; j < PER; ++j) num[j] = fmaf(w, v[p][j], num[j]);
        }
    }
    const size_t oi = (size_t)sh * D + lane * PER;
#pragma unroll
    for (int j = 0; j < PER; ++j) comb_store(a, oi + j, den > 0.f ? num[j] / den : 0.f);
    // (the consumed partials are left in L2 here: dropping them, as the
    // many-partition combine does, measured 0.45 % slower on 128 sequences
    // of 512-8192 tokens in 1024-token parts)
}

// Many partitions (a long context has hundreds): one CTA per (sequence,
// head).  The CTA computes the weights 2^(lse_p - M) once into shared memory,
// kCombChunk parts at a time; then warp w sums every kCombWarps-th part, each
// lane owning D/32 adjacent columns (one 16-byte load per part for D = 128),
// with kCombUnroll parts in flight, and the warps' sums meet in shared memory.
constexpr int kCombWarps = kCombThreads / 32;
constexpr int kCombUnroll = 8;

template <int PER>
__device__ __forceinline__ void comb_load(const float *p, float (&v)[PER]) {
    if constexpr (PER == 8) {
        const float4 x = *reinterpret_cast<const float4 *>(p);
        const float4 y = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w, v[4] = y.x, v[5] = y.y, v[6] = y.z, v[7] = y.w;
    } else if constexpr (PER == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(p);
        v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
    } else {
        const float2 x = *reinterpret_cast<const float2 *>(p);
        v[0] = x.x, v[1] = x.y;
    }
}

template <int PER>
__global__ void __launch_bounds__(kCombThreads) lse_combine_many_kernel(const DecodeArgs a, int block_size) {
    constexpr int D = PER * 32;
    __shared__ float w_s[kCombChunk];
    __shared__ float red_m[kCombWarps], red_d[kCombWarps];
    __shared__ __align__(16) float acc_s[kCombWarps][D];
    griddep_wait();  // the decode grid's partials are complete
    const CombRow r = comb_row(a, D, block_size, blockIdx.x);
    if (r.nparts <= 1) return;  // the decode kernel wrote this row directly
    const float M = comb_max(r, red_m);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float num[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) num[j] = 0.f;
    float den = 0.f;
    for (int p0 = 0; p0 < r.nparts; p0 += kCombChunk) {
        const int n = r.nparts - p0 < kCombChunk ? r.nparts - p0 : kCombChunk;
        __syncthreads();  // the previous chunk's weights are consumed
        for (int i = tid; i < n; i += kCombThreads) {
            const float w = M == -CUDART_INF_F ? 0.f : fast_exp2(r.lse[p0 + i] - M);
            w_s[i] = w;
            den += w;
        }
        __syncthreads();
        const float *col = r.po + (size_t)p0 * D + lane * PER;
        int i = warp;
        for (; i + (kCombUnroll - 1) * kCombWarps < n; i += kCombUnroll * kCombWarps) {
            float v[kCombUnroll][PER];
#pragma unroll
            for (int u = 0; u < kCombUnroll; ++u) comb_load<PER>(col + (size_t)(i + u * kCombWarps) * D, v[u]);
#pragma unroll
            for (int u = 0; u < kCombUnroll; ++u) {
                const float w = w_s[i + u * kCombWarps];
#pragma unroll
                for (int j = 0; j < PER; ++j) num[j] = fmaf(w, v[u][j], num[j]);
            }
        }
        for (; i < n; i += kCombWarps) {
            float v[PER];
            comb_load<PER>(col + (size_t)i * D, v);
            const float w = w_s[i];
#pragma unroll
            for (int j = 0; j < PER; ++j) num[j] = fmaf(w, v[j], num[j]);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    if (lane == 0) red_d[warp] = den;
#pragma unroll
    for (int j = 0; j < PER; ++j) acc_s[warp][lane * PER + j] = num[j];
    __syncthreads();
    den = 0.f;
#pragma unroll
    for (int w = 0; w < kCombWarps; ++w) den += red_d[w];
    for (int d = tid; d < D; d += kCombThreads) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < kCombWarps; ++w) x += acc_s[w][d];
        comb_store(a, (size_t)r.sh * D + d, den > 0.f ? x / den : 0.f);
    }
    // every warp has used its loads (the barrier above): the row's partial
    // lines are dead, and would otherwise be written back from L2 during the
    // next decode (48 MB per call on a 128k-token batch in 512-token parts)
    for (int q = tid; q < r.nparts * (D / 32); q += kCombThreads) l2_discard_line(r.po + (size_t)q * 32);
}

pkv_status launch_lse_combine(const DecodeArgs &a, int num_seqs, int head_dim, int block_size,
                              cudaStream_t stream) {
    const long long n = (long long)num_seqs * a.num_heads;
    if (n == 0) return PKV_OK;
    if (a.num_parts <= kCombDirect) {
        const dim3 grid((unsigned)((n + 7) / 8));
        if (head_dim == 64)
            return cuda_status(launch_dependent(lse_combine_kernel<2>, grid, dim3(256), 0, stream, a,
                                                block_size, (int)n));
        if (head_dim == 256)
            return cuda_status(launch_dependent(lse_combine_kernel<8>, grid, dim3(256), 0, stream, a,
                                                block_size, (int)n));
        return cuda_status(launch_dependent(lse_combine_kernel<4>, grid, dim3(256), 0, stream, a,
                                            block_size, (int)n));
    }
    const dim3 grid((unsigned)n);
    if (head_dim == 64)
        return cuda_status(launch_dependent(lse_combine_many_kernel<2>, grid, dim3(kCombThreads), 0,
                                            stream, a, block_size));
    if (head_dim == 256)
        return cuda_status(launch_dependent(lse_combine_many_kernel<8>, grid, dim3(kCombThreads), 0,
                                            stream, a, block_size));
    return cuda_status(launch_dependent(lse_combine_many_kernel<4>, grid, dim3(kCombThreads), 0, stream,
                                        a, block_size));
}

}  // namespace pkv
