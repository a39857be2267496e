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
// CUDA-core decode: query rows of a group one CTA takes at most.  A larger
// group is split over CTAs of the same kv head, launched side by side so the
// repeated reads of each K/V tile mostly hit L2: each thread holds its slice
// of every row's query and accumulator, and 16 rows spilled (fp32, G = 16:
// 0.14 of the copy peak whole, 0.38 in CTAs of 8 rows, 0.40 in CTAs of 4)
constexpr int kFmaRowsMax = 4;
// fp32 storage: groups from this size on take TF32 tensor-core tiles (a
// 16-row tile costs the same for any group).  Measured on the gqa_8b batch
// (decode µs, CUDA cores / TF32): head 128, G = 5, 8, 12, 16: 945 / 976,
// 952 / 986, 1338 / 1036, 1736 / 1046; head 64, G = 5, 16: 644 / 496,
// 1250 / 527.
constexpr int tf32_min_group(int head_dim) { return head_dim == 128 ? 9 : 5; }
constexpr int kMaxStageRows = 16;  // rows of one staged run; larger blocks are staged in runs
constexpr int kSpRowsMax = 32;  // shared-prefix decode: query rows per work item (two MMA tiles)
// Query rows of a shared-prefix work item for a head size: two 16-row tiles
// for a 128-wide head; one tile for a 256-wide head (the same accumulator
// registers) and for a 64-wide one, whose lighter items then fit four CTAs
// per SM (measured faster than two CTAs of two-tile items, although a group
// with more members than one item holds reads its prefix once per item).
// fp32 storage takes one tile at every head size (fp32 accumulators of TF32 tiles).
constexpr int sp_rows_for(int head_dim, int elem_bytes = 2) {
    return head_dim == 128 && elem_bytes == 2 ? kSpRowsMax : 16;
}

// Arguments of one decode launch; every pointer is a device pointer.
struct DecodeArgs {
    const void *q;              // [S][H][D] pool dtype
    void *out;                  // [S][H][D] in out_dtype (fp32, bf16 or fp16)
    float *ws_o;                // [S][H][P][D] normalised partition outputs (split only)
    float *ws_lse;              // [S][H][P] log2-sum-exp of each partition (split only)
    const int32_t *block_tables;
    const int32_t *context_lens;
    int32_t *dev_error;
    int num_heads;
    int num_kv_heads;
    int group;                  // num_heads / num_kv_heads
    int row_split;              // CTAs per kv head, each with its own query rows of the group
    int rows_per_cta;           // ceil(group / row_split)
    int max_blocks_per_seq;
    int num_blocks;
    int ctx_cap;                // min(max_blocks_per_seq * BS, max_context_len)
    int part_blocks;            // staged runs per partition (one CTA each)
    int num_parts;              // gridDim.z: partitions of the longest allowed context
    int out_dtype;              // pkv_dtype of out
    int contig;                 // 1: contiguous cache, block b of (s, g) is row run (s*Hkv+g)*num_blocks+b
    int unit_shift;             // a pool block is 2^unit_shift staged runs of BS rows (blocks over 16 rows)
    float scale_log2;           // scale * log2(e)
};

struct DecodeLaunch {
    const CUtensorMap *tmk;
    const CUtensorMap *tmv;
    DecodeArgs args;
    int num_seqs;
    int head_dim;
    int block_size;             // rows of a staged run (16)
    int group_pad;              // FMA path: query rows per CTA (power of two >= group)
    bool mma;
    bool runs;                  // pool blocks are staged in several runs (unit_shift > 0)
    cudaStream_t stream;
    int device;
};

// One work item of the shared-prefix decode, written by the planning kernel
// (as two 16-byte stores).
struct alignas(16) SpEntry {
    int seq0;      // first sequence of the item's query rows
    int nseq;      // sequences in the item (rows = nseq * group)
    int tbl_seq;   // sequence whose block-table row names the item's blocks
    int b0, b1;    // logical blocks [b0, b1)
    int slot;      // partial slot (of every row's sequence) the item writes
    int tok_end;   // context positions >= tok_end are masked
    int reserved;
};
static_assert(sizeof(SpEntry) == 32, "work item is two 16-byte words");

// Arguments of the persistent shared-prefix decode kernel.
struct SpArgs {
    const void *q;              // [S][H][D] pool dtype
    void *out;                  // [S][H][D] in out_dtype (fp32, bf16 or fp16)
    float *ws_o;                // [S][H][num_slots][D] partial outputs
    float *ws_lse;              // [S][H][num_slots] their log2-sum-exp
    const int32_t *block_tables;
    int32_t *dev_error;
    const SpEntry *entries;     // work list: prefix items at [0, count[0]), suffix items at
                                // [suffix_base, suffix_base + count[1]) (planning kernel)
    const int32_t *nparts;      // [S] partials of each sequence (planning kernel)
    const int32_t *seq_share;   // [S][2] group leader and shared blocks (planning kernel)
    const int32_t *block_tables_chk;  // block tables, for the combine's agreement check
    int32_t *counter;           // work counter, zeroed by the planning kernel
    const int32_t *count;       // workspace header: [0], [1] prefix and suffix entries,
                                // [kSpHdrMagic..] the plan's geometry (planning kernel)
    int suffix_base;
    int num_seqs;
    int block_size;             // tokens per pool block
    int unit_shift;             // a block is 2^unit_shift staged runs (blocks over 16 tokens);
                                // work items count runs
    int num_heads;
    int num_kv_heads;
    int group;
    int max_blocks_per_seq;
    int num_blocks;
    int num_slots;
    int out_dtype;              // pkv_dtype of out
    int members_per_item;       // sequences a prefix item holds (query rows per item / group)
    float scale_log2;
};

// Workspace header of the shared-prefix plan: where the plan records the
// geometry it was made for, and the value that marks a written plan.
constexpr int kSpHdrMagic = 8;
constexpr int32_t kSpPlanMagic = 0x50504c31;  // "PPL1"

// Whether the plan in the workspace was made for this call's geometry.  The
// members per prefix item follow the pool's head size and storage type (the
// query rows one item's tiles hold), so a plan made for another pool is
// refused rather than read with items larger than this kernel's tiles.
__host__ __device__ inline bool sp_plan_matches(const SpArgs &a) {
    const int32_t *h = a.count + kSpHdrMagic;
    return h[0] == kSpPlanMagic && h[1] == a.num_seqs && h[2] == a.num_heads &&
           h[3] == a.num_kv_heads && h[4] == a.block_size && h[5] == a.num_slots &&
           h[6] == a.suffix_base && h[7] == a.members_per_item;
}

struct SpLaunch {
    const CUtensorMap *tmk;
    const CUtensorMap *tmv;
    SpArgs args;
    int head_dim;
    int block_size;
    cudaStream_t stream;
    int device;
    int *grid_warps;            // if set: store the persistent grid's warps here, launch nothing
};

pkv_status launch_shared_prefix_d64(const SpLaunch &L);       // bf16 pools
pkv_status launch_shared_prefix_d128(const SpLaunch &L);      // bf16 pools
pkv_status launch_shared_prefix_f16_d64(const SpLaunch &L);
pkv_status launch_shared_prefix_f16_d128(const SpLaunch &L);
pkv_status launch_shared_prefix_d256(const SpLaunch &L);      // bf16 pools
pkv_status launch_shared_prefix_f16_d256(const SpLaunch &L);
pkv_status launch_shared_prefix_f32_d64(const SpLaunch &L);
pkv_status launch_shared_prefix_f32_d128(const SpLaunch &L);

pkv_status launch_decode_f32_d64(const DecodeLaunch &L);
pkv_status launch_decode_f32_d128(const DecodeLaunch &L);
pkv_status launch_decode_bf16_d64(const DecodeLaunch &L);
pkv_status launch_decode_bf16_d128(const DecodeLaunch &L);
pkv_status launch_decode_f16_d64(const DecodeLaunch &L);
pkv_status launch_decode_f16_d128(const DecodeLaunch &L);
pkv_status launch_decode_bf16_d256(const DecodeLaunch &L);
pkv_status launch_decode_f16_d256(const DecodeLaunch &L);

pkv_status launch_lse_combine(const DecodeArgs &a, int num_seqs, int head_dim, int block_size,
                              cudaStream_t stream);

pkv_status launch_reshape_and_cache(const pkv_pool &pool, const void *key, const void *value,
                                    const int64_t *slot_mapping, int num_tokens,
                                    cudaStream_t stream);

pkv_status launch_bounded_wait_check(int32_t *dev_error, long long limit_ns, cudaStream_t stream);
pkv_status launch_copy_blocks(const pkv_pool &pool, const int32_t *src, const int32_t *dst,
                              int num_pairs, cudaStream_t stream);

int sm_count(int device);

// Record `e` as this thread's last CUDA error (if it is one) and map it to a
// status: PKV_OK for cudaSuccess, PKV_ERR_CUDA otherwise.
pkv_status cuda_status(cudaError_t e);

}  // namespace pkv
