// pkv_internal.h -- launch descriptors shared by the host API and the kernel
// translation units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr uint32_t kPoolMagic = 0x504b5631u;  // "PKV1"
constexpr int kAutoPartitionTokens = 512;
constexpr int kMaxPartitionTokens = 8192;
constexpr int kMaxGroup = 16;

// Arguments of one decode launch; every pointer is a device pointer.
struct DecodeArgs {
    const void *q;              // [S][H][D] pool dtype
    void *out;                  // [S][H][D] fp32 or bf16
    float *ws_o;                // [S][H][P][D] normalised partition outputs (split only)
    float *ws_lse;              // [S][H][P] log2-sum-exp of each partition (split only)
    const int32_t *block_tables;
    const int32_t *context_lens;
    int32_t *dev_error;
    int num_heads;
    int num_kv_heads;
    int group;                  // num_heads / num_kv_heads
    int max_blocks_per_seq;
    int num_blocks;
    int ctx_cap;                // min(max_blocks_per_seq * BS, max_context_len)
    int part_blocks;            // KV blocks per partition (one CTA each)
    int num_parts;              // gridDim.z: partitions of the longest allowed context
    int out_bf16;
    int contig;                 // 1: contiguous cache, block b of (s, g) is row run (s*Hkv+g)*num_blocks+b
    float scale_log2;           // scale * log2(e)
};

struct DecodeLaunch {
    const CUtensorMap *tmk;
    const CUtensorMap *tmv;
    DecodeArgs args;
    int num_seqs;
    int head_dim;
    int block_size;
    int group_pad;              // FMA path: query rows per CTA (power of two >= group)
    bool mma;
    cudaStream_t stream;
    int device;
};

pkv_status launch_decode_f32_d64(const DecodeLaunch &L);
pkv_status launch_decode_f32_d128(const DecodeLaunch &L);
pkv_status launch_decode_bf16_d64(const DecodeLaunch &L);
pkv_status launch_decode_bf16_d128(const DecodeLaunch &L);

pkv_status launch_lse_combine(const DecodeArgs &a, int num_seqs, int head_dim, int block_size,
                              cudaStream_t stream);

pkv_status launch_reshape_and_cache(const pkv_pool &pool, const void *key, const void *value,
                                    const int64_t *slot_mapping, int num_tokens,
                                    cudaStream_t stream);

pkv_status launch_copy_blocks(const pkv_pool &pool, const int32_t *src, const int32_t *dst,
                              int num_pairs, cudaStream_t stream);

int sm_count(int device);

// Record `e` as this thread's last CUDA error (if it is one) and map it to a
// status: PKV_OK for cudaSuccess, PKV_ERR_CUDA otherwise.
pkv_status cuda_status(cudaError_t e);

}  // namespace pkv
