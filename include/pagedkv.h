/*
 * pagedkv.h -- C ABI of a paged KV-cache decode-attention library for
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow the PagedAttention pages:
 *   - the KV cache is cut into fixed-size blocks that need not be contiguous
 *     in device memory (Qualiteg, "About PagedAttention for LLM serving",
 *     "[Regarding Problem 1]", point 1-2; the same page puts a block at
 *     roughly 16 to 256 tokens);
 *   - logical blocks of a sequence map onto physical blocks through a block
 *     table (same page, the section on logical blocks, physical blocks and
 *     the block table that links them);
 *   - the cache grows by one token per iteration (same page, "Characteristics
 *     of Autoregressive Models ..."), which pkv_reshape_and_cache writes;
 *   - attention is computed over the non-contiguous blocks without padding
 *     (same page, "[Regarding Problem 2] 2-1"; vAttention, section 3.1
 *     "Requires re-writing the attention kernel", which also names the
 *     grouped-query case), which pkv_paged_attention_decode computes.
 *
 * Conventions shared by every call
 *   - Every device buffer is owned by the caller.  The library allocates no
 *     device memory and keeps no mutable global state.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work; nothing synchronises except
 *     pkv_get_device_error.  So every call can be captured in a CUDA graph
 *     (once its kernels have run eagerly once: their one-time attribute
 *     set-up is not a stream operation) and replayed with new contents in
 *     the captured buffers.
 *   - Invalid arguments are rejected on the host with PKV_ERR_INVALID_ARG or
 *     PKV_ERR_UNSUPPORTED before anything is launched.  A failed launch
 *     returns PKV_ERR_CUDA.  No C++ exception crosses this boundary.
 *   - Data-dependent faults that only the device can see (a block-table
 *     entry outside the pool, a slot past the pool, a context length beyond
 *     the table) never trap: the kernel skips the bad work and ORs a
 *     PKV_FAULT_* bit into the pool's error word, if one was given.
 *   - All device pointers must be 16-byte aligned; the split-K workspace
 *     must be 256-byte aligned.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, block_size, group, dtype */
    PKV_ERR_CUDA = 3,          /* a CUDA runtime/driver call or launch failed */
    PKV_ERR_WORKSPACE = 4,     /* split-K workspace missing or too small */
    PKV_ERR_DEVICE_FAULT = 5,  /* the device error word was non-zero */
    PKV_ERR_OUT_OF_BLOCKS = 6  /* the block manager has no free block left */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_F16 = 2 } pkv_dtype;

/* Bits a kernel ORs into *pool->dev_error. */
#define PKV_FAULT_BLOCK_ID 1u  /* block-table entry outside [0, num_blocks): block skipped */
#define PKV_FAULT_SLOT 2u      /* slot_mapping entry >= num_blocks*block_size: token skipped */
#define PKV_FAULT_CONTEXT 4u   /* context_len < 0, > max_blocks_per_seq*block_size or
                                  > max_context_len: clamped */
#define PKV_FAULT_TIMEOUT 8u   /* a shared-memory pipeline wait ran past its bound */
#define PKV_FAULT_PREFIX 16u   /* a shared-prefix group description was inconsistent (see
                                  pkv_paged_attention_decode_shared_prefix) */

/* Flags of pkv_paged_attention_decode. */
#define PKV_DECODE_PATH_AUTO 0  /* tensor cores when the GQA group makes dense tiles */
#define PKV_DECODE_PATH_FMA 1   /* CUDA-core dot products for every group size (groups above
                                   4 rows are split over CTAs of the same kv head) */
#define PKV_DECODE_PATH_MMA 2   /* tensor-core tiles for every group size: bf16/fp16 tiles for
                                   16-bit pools, TF32 tiles with three products each for fp32
                                   pools (head_dim 64 or 128) */

/*
 * Block pool: K and V are separate device buffers, each laid out
 * [num_blocks][num_kv_heads][block_size][head_dim] row-major, so one
 * (block, kv head) tile is block_size*head_dim contiguous elements and every
 * row starts on a 16-byte boundary.  Filled by pkv_block_pool_init; treat as
 * read-only afterwards.  `tma` holds the two TMA tensor descriptors (K, V)
 * the decode kernel stages tiles with; it is only valid on `device`.
 */
typedef struct pkv_pool {
    uint32_t magic;               /* set by pkv_block_pool_init; other values = not initialised */
    int num_blocks;
    int block_size;
    int num_kv_heads;
    int head_dim;
    pkv_dtype dtype;
    int device;
    int layout;                   /* 0 = paged block pool, 1 = contiguous per-sequence cache */
    int num_seqs;                 /* contiguous layout only: sequences the cache holds */
    void *k_pool;
    void *v_pool;
    int32_t *dev_error;           /* device int32 or NULL */
    uint64_t tma[32];             /* 2 x 128-byte descriptors, 64-byte aligned copy inside */
} pkv_pool;

/* Bytes of ONE pool (K or V): num_blocks*num_kv_heads*block_size*head_dim*elem. 0 if invalid. */
size_t pkv_pool_bytes(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                      pkv_dtype dtype);

/*
 * Describe a caller-allocated block pool and prepare it for the kernels.
 * k_pool/v_pool: device buffers of pkv_pool_bytes(...) bytes each, on the
 * current device.  dev_error: device int32 error word or NULL.  zero_fill:
 * non-zero clears both pools and the error word on `stream`.
 * Supported: block_size in {16, 32, 64, 128, 256} (the page's range of
 * roughly 16 to 256 tokens; the kernels stage every block in runs of 16
 * rows); head_dim in {64, 128, 256} (256: BF16 or F16 pools); dtype F32,
 * BF16 or F16 (the shared-prefix decode takes BF16 or F16 pools);
 * num_blocks*num_kv_heads*block_size < 2^31.
 */
pkv_status pkv_block_pool_init(pkv_pool *pool, int num_blocks, int block_size, int num_kv_heads,
                               int head_dim, pkv_dtype dtype, void *k_pool, void *v_pool,
                               int32_t *dev_error, int zero_fill, void *stream);

/*
 * Asynchronous host-to-device copy of a [num_seqs][max_blocks_per_seq] int32
 * block table.  Entry (s, i) is the physical block of logical block i of
 * sequence s; entries a sequence does not need may hold any value (-1 by
 * convention).  If num_blocks > 0, every entry must be < num_blocks (negative
 * = unused) or nothing is copied and PKV_ERR_INVALID_ARG is returned.  The
 * host buffer must stay valid until the copy has run (pinned memory makes the
 * copy truly asynchronous).
 */
pkv_status pkv_block_table_upload(int32_t *dev_block_tables, const int32_t *host_block_tables,
                                  int num_seqs, int max_blocks_per_seq, int num_blocks,
                                  void *stream);

/*
 * Cache write of the new tokens: for each t < num_tokens with
 * slot = slot_mapping[t] >= 0, copy key[t][h][:] and value[t][h][:] to row
 * slot % block_size of physical block slot / block_size, kv head h, for every
 * h.  key/value: device [num_tokens][num_kv_heads][head_dim], pool dtype,
 * contiguous.  slot_mapping: device int64 [num_tokens].  A negative slot is
 * padding and skipped; a slot >= num_blocks*block_size sets PKV_FAULT_SLOT
 * and is skipped.  Bytes are copied exactly.  The non-negative slots of one
 * call must be distinct: if two tokens name one slot, which of them lands
 * there is not specified.  (A sequence whose new token falls inside a block
 * it shares must be given its own copy of that block first; see
 * pkv_copy_blocks and the block manager.)
 */
pkv_status pkv_reshape_and_cache(const pkv_pool *pool, const void *key, const void *value,
                                 const int64_t *slot_mapping, int num_tokens, void *stream);

/*
 * Workspace bytes pkv_paged_attention_decode needs for split-K partials:
 * num_seqs*num_heads*ceil(max_context_len/partition)*(head_dim+1)*4, rounded
 * up to 256.  partition_tokens 0 (automatic) sizes for the smallest
 * partition the automatic choice uses (512 tokens); -1 (never split) needs 0.
 */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                  int partition_tokens);

/*
 * Decode-step attention of one new query token per sequence over its paged
 * KV cache:
 *   out[s][h][:] = sum_j softmax_j(scale * <query[s][h], K_s[j]>) V_s[j],
 * j over logical positions 0 .. context_lens[s]-1, K_s[j]/V_s[j] the row of
 * kv head h / (num_heads/num_kv_heads) in physical block
 * block_tables[s][j / block_size], row j % block_size.  context_lens counts
 * the new token, which pkv_reshape_and_cache must already have written.
 * A sequence with context length 0 gets a zero row.
 *
 * query: device [num_seqs][num_heads][head_dim] in the pool dtype.
 * out: device [num_seqs][num_heads][head_dim] in out_dtype (F32, BF16 or
 *   F16).  Scores and sums are fp32 whatever the storage type.  AUTO takes
 *   tensor-core tiles for groups of 4 or more with BF16 or F16 pools and,
 *   with F32 pools, for groups of 9 or more at head_dim 128 and of 5 or more
 *   at head_dim 64 (TF32, each product as three TF32 products, each k-step
 *   summed in fp32: within the fp32 tolerance), CUDA-core dot products
 *   otherwise.
 * block_tables: device int32 [num_seqs][max_blocks_per_seq].
 * context_lens: device int32 [num_seqs].
 * max_context_len: host upper bound on every context length (grid sizing;
 *   larger lengths are clamped and flagged PKV_FAULT_CONTEXT).
 * partition_tokens: 0 = automatic (no split, or 512-2048-token partitions
 *   chosen from the batch shape), -1 = never split, > 0 = split every
 *   sequence into partitions of this many tokens (a multiple of block_size,
 *   at most 8192) and combine them with a log-sum-exp pass.
 * workspace: device buffer of at least pkv_decode_workspace_bytes(...) bytes
 *   when a split can happen (may be NULL with partition_tokens = -1).
 * flags: one of PKV_DECODE_PATH_*.
 * Supported groups: num_heads / num_kv_heads in 1..16; num_seqs <= 65535.
 */
pkv_status pkv_paged_attention_decode(const pkv_pool *pool, void *out, pkv_dtype out_dtype,
                                      const void *query, int num_seqs, int num_heads,
                                      int num_kv_heads, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *context_lens,
                                      int max_context_len, float scale, int partition_tokens,
                                      void *workspace, size_t workspace_bytes, int flags,
                                      void *stream);

/* Size of the fixed split-K scratch array behind pkv_paged_attention_decode_static. */
#define PKV_STATIC_SCRATCH_BYTES (64u << 20)

/*
 * Allocation-free variant of pkv_paged_attention_decode (the pages have no
 * counterpart; it exists for callers of this library that cannot allocate
 * device memory: an engine that gives all device memory to the KV pool and a
 * caching allocator at start-up, a plain-C host program without a device
 * allocator, or a latency-critical loop where cudaMalloc/cudaFree would
 * synchronise the device).  Same arguments and result as
 * pkv_paged_attention_decode, minus the workspace: split-K partials go to a
 * fixed device array of PKV_STATIC_SCRATCH_BYTES (64 MiB) compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  Nothing is allocated: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *  - The first call on a device looks the array's device address up
 *    (cudaGetSymbolAddress, with that device current) and keeps it for the
 *    life of the process; make that first call before any stream capture.
 *    A cudaDeviceReset rebuilds the device's modules, so the kept address is
 *    stale afterwards: do not use this entry point across a cudaDeviceReset.
 *  - A call whose partials need more than PKV_STATIC_SCRATCH_BYTES returns
 *    PKV_ERR_WORKSPACE without launching anything.  The need is the one the
 *    decode computes for the partition it actually takes (with
 *    partition_tokens = 0, the automatic choice of 512 to 2048 tokens), which
 *    is at most pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim,
 *    max_context_len, partition_tokens).
 *  - Every call on a device shares the one array and leaves its contents
 *    behind; nothing in it needs to start at zero (each partial is written
 *    before it is read).  Calls that overlap on the GPU (other streams, other
 *    host threads) race on the array: serialise them.
 */
pkv_status pkv_paged_attention_decode_static(const pkv_pool *pool, void *out,
                                             pkv_dtype out_dtype, const void *query,
                                             int num_seqs, int num_heads, int num_kv_heads,
                                             const int32_t *block_tables, int max_blocks_per_seq,
                                             const int32_t *context_lens, int max_context_len,
                                             float scale, int partition_tokens, int flags,
                                             void *stream);

/*
 * Contiguous-layout variant, for measuring what paging costs (the pages note
 * that a paged kernel is slower than one reading contiguous K and V: the
 * Hacker News thread, and vAttention section 3.1).  Not part of the paged
 * path: it reads a conventional cache where sequence s, kv head g holds its
 * tokens in rows [s][g][0 .. capacity) of a [num_seqs][num_kv_heads]
 * [capacity][head_dim] K (and V) buffer.  capacity: a multiple of 16.  The
 * kernel is the paged kernel with the block table replaced by identity
 * numbering, so for the same tokens it returns bitwise the paged result.
 */
pkv_status pkv_contiguous_cache_init(pkv_pool *cache, int num_seqs, int capacity,
                                     int num_kv_heads, int head_dim, pkv_dtype dtype,
                                     void *k_cache, void *v_cache, int32_t *dev_error,
                                     int zero_fill, void *stream);
/* Decode attention over a contiguous cache; arguments as
 * pkv_paged_attention_decode without the block table. */
pkv_status pkv_contiguous_attention_decode(const pkv_pool *cache, void *out, pkv_dtype out_dtype,
                                           const void *query, int num_seqs, int num_heads,
                                           int num_kv_heads, const int32_t *context_lens,
                                           int max_context_len, float scale,
                                           int partition_tokens, void *workspace,
                                           size_t workspace_bytes, int flags, void *stream);

/*
 * Shared-prefix decode: the same result as pkv_paged_attention_decode for a
 * batch in which groups of sequences share the physical blocks of a common
 * prompt prefix (sequences forked from one prompt: parallel sampling, beam
 * search; the Hacker News thread on PagedAttention describes such sharing of
 * blocks between a sequence's siblings, and Qualiteg's "About PagedAttention
 * for LLM serving" the per-sequence block tables that make it possible).
 * Each shared block is staged once per kv head for up to 32 query rows of
 * the group (16 for 64- and 256-wide heads; a larger group stages it once per
 * such set of rows, the repeats mostly from L2) and multiplied against those
 * members' query rows on tensor cores; each member's own blocks after the
 * prefix are read as usual; a log-sum-exp pass merges the parts.
 *
 * Groups: group i is sequences group_starts[i] .. group_starts[i+1]-1, and
 * every member's first prefix_lens[i] / block_size block-table entries name
 * the same physical blocks.  group_starts: device int32 [num_groups + 1],
 * non-decreasing from 0 to num_seqs (a sequence that shares nothing is a
 * group of one).  prefix_lens: device int32 [num_groups], tokens, a multiple
 * of the block size, at most max_prefix_len and at most every member's
 * context length.  max_prefix_len: host bound used to size the workspace.
 * The other arguments are those of pkv_paged_attention_decode; context_lens
 * count every token, prefix included.
 *
 * A group description that breaks these rules (group_starts not covering the
 * batch in order, a prefix length that is negative, not a whole number of
 * blocks, above max_prefix_len or above a member's context, or members whose
 * tables differ inside the prefix) sets PKV_FAULT_PREFIX.  Apart from table
 * disagreement, which is only detected (after the fact: the first member's
 * blocks are used), the offending group is then computed without sharing,
 * so the output is still exact.
 *
 * partition_tokens: 0 = automatic (prefix parts of 512, 1024 or 2048 tokens,
 * chosen on the device: the longest that still gives the persistent decode
 * grid three prefix items for every four warps, every two warps for F32
 * pools; parts of 256 tokens for each sequence's own blocks), -1 = one part
 * each, > 0 = parts of that many tokens (a multiple of block_size, at most
 * 8192).  workspace: device buffer (256-byte
 * aligned) of at least pkv_shared_prefix_workspace_bytes(...) bytes; it also
 * holds the work list, so every call needs one.  Supported: BF16 or F16
 * pools (head_dim 64, 128 or 256; the work items of 64- and 256-wide heads
 * carry 16 query rows instead of 32), and F32 pools of head_dim 64 or 128
 * (items of 16 rows as TF32 tiles, three products each, k-steps summed in
 * fp32), num_heads / num_kv_heads in 1..16, out_dtype F32, BF16 or F16.
 */
size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                         int max_context_len, int max_prefix_len,
                                         int partition_tokens);
pkv_status pkv_paged_attention_decode_shared_prefix(
    const pkv_pool *pool, void *out, pkv_dtype out_dtype, const void *query, int num_seqs,
    int num_heads, int num_kv_heads, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, float scale, const int32_t *group_starts,
    const int32_t *prefix_lens, int num_groups, int max_prefix_len, int partition_tokens,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * The shared-prefix decode in two calls, for a model whose layers share one
 * decode step's batch: the plan depends only on the group description and
 * the context lengths, which every layer of a step has in common, so one
 * plan serves all of them.
 *
 * pkv_shared_prefix_plan: checks the group description and writes the work
 * list into `workspace` (arguments as in pkv_paged_attention_decode_shared_
 * prefix; block tables and queries are not needed yet).
 *
 * pkv_paged_attention_decode_shared_prefix_run: the decode and combine from
 * that plan, for one layer's pool, queries and output.  num_seqs, num_heads,
 * num_kv_heads, the block size, max_context_len, max_prefix_len and
 * partition_tokens must be those of the plan, and the pool must hold as many
 * query rows per work item as the plan's (the same head size and storage
 * type, or ones with the same rows per item): a run whose geometry differs
 * from the plan in the workspace (or that finds no plan there) sets
 * PKV_FAULT_PREFIX and writes nothing.  Runs on one plan must be ordered on
 * the GPU (one stream): each run's last kernel re-arms the plan for the
 * next.  The block tables must be those the plan's groups describe.
 */
pkv_status pkv_shared_prefix_plan(const pkv_pool *pool, int num_seqs, int num_heads,
                                  int num_kv_heads, int max_blocks_per_seq,
                                  const int32_t *context_lens, int max_context_len,
                                  const int32_t *group_starts, const int32_t *prefix_lens,
                                  int num_groups, int max_prefix_len, int partition_tokens,
                                  void *workspace, size_t workspace_bytes, void *stream);
pkv_status pkv_paged_attention_decode_shared_prefix_run(
    const pkv_pool *pool, void *out, pkv_dtype out_dtype, const void *query, int num_seqs,
    int num_heads, int num_kv_heads, const int32_t *block_tables, int max_blocks_per_seq,
    int max_context_len, float scale, int max_prefix_len, int partition_tokens, void *workspace,
    size_t workspace_bytes, void *stream);

/*
 * Copy whole physical blocks (every kv head, K and V): block dst[i] becomes a
 * copy of block src[i], i < num_pairs.  src/dst: device int32 arrays.  Used
 * for the block manager's copy-on-write, before the new token is written.
 * A pair naming a block outside the pool sets PKV_FAULT_BLOCK_ID and is
 * skipped.  Pairs of one call must not chain (no dst is another pair's src).
 */
pkv_status pkv_copy_blocks(const pkv_pool *pool, const int32_t *src, const int32_t *dst,
                           int num_pairs, void *stream);

/*
 * Host-side block manager (host memory only, no CUDA call, not thread-safe).
 * It hands out physical blocks of a pool of num_blocks blocks as sequences
 * grow and takes them back when they finish (Qualiteg, "[Regarding Problem
 * 1]", point 1-3: blocks are taken and returned on demand instead of reserved
 * up front), keeps each sequence's logical-to-physical block list (the same
 * page's section on logical and physical blocks), and lets forked
 * sequences share blocks (prompt-prefix sharing) with reference counts:
 * appending to a shared, partly filled last block first moves the writer to
 * a fresh block and queues a (src, dst) copy for pkv_copy_blocks.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* New manager over blocks 0..num_blocks-1, all free; lowest ids first. */
pkv_status pkv_bm_create(int num_blocks, int block_size, pkv_block_manager **out);
void pkv_bm_destroy(pkv_block_manager *bm);
/* Free blocks, or -1 for a NULL manager. */
int pkv_bm_free_blocks(const pkv_block_manager *bm);
/* Reference count of a physical block (0 = free), -1 if out of range. */
int pkv_bm_refcount(const pkv_block_manager *bm, int32_t block);
/* Register a new sequence of num_tokens tokens (its prompt) and allocate its
 * blocks; slots (may be NULL) receives each token's flat pool slot, for the
 * cache write.  PKV_ERR_OUT_OF_BLOCKS leaves the manager unchanged. */
pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id, int64_t num_tokens,
                               int64_t *slots);
/* child shares every block of parent (reference counts + 1). */
pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child);
/* Grow a sequence by one token; *slot receives the new token's pool slot.
 * May allocate a block, or copy-on-write a shared last block. */
pkv_status pkv_bm_append_token(pkv_block_manager *bm, int64_t seq_id, int64_t *slot);
/* Drop a sequence; blocks no other sequence holds become free. */
pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);
/* Tokens of a sequence, -1 if unknown. */
int64_t pkv_bm_context_len(const pkv_block_manager *bm, int64_t seq_id);
/* Pending copy-on-write copies, and draining them (returns how many were
 * written to src/dst, at most capacity). */
int pkv_bm_pending_copies(const pkv_block_manager *bm);
int pkv_bm_take_copies(pkv_block_manager *bm, int32_t *src, int32_t *dst, int capacity);
/* Host block tables [num_seqs][max_blocks_per_seq] (-1 padded) and context
 * lengths of the listed sequences, ready for pkv_block_table_upload. */
pkv_status pkv_bm_block_tables(const pkv_block_manager *bm, const int64_t *seq_ids, int num_seqs,
                               int max_blocks_per_seq, int32_t *block_tables,
                               int32_t *context_lens);

/* Group description for the shared-prefix decode: for each group of the
 * listed sequences (group g = seq_ids[group_starts[g] .. group_starts[g+1]),
 * host arrays), prefix_lens[g] receives the tokens of the longest run of
 * leading blocks that every member holds in its table and has filled
 * (0 for a group of one).  Sequences forked from one prompt and listed side
 * by side make a group. */
pkv_status pkv_bm_shared_prefix(const pkv_block_manager *bm, const int64_t *seq_ids, int num_seqs,
                                const int32_t *group_starts, int num_groups,
                                int32_t *prefix_lens);

/*
 * Synchronise `stream`, read the pool's device error word into *fault_bits
 * (may be NULL) and clear it.  Returns PKV_ERR_DEVICE_FAULT if it was
 * non-zero, PKV_OK if zero or if the pool has no error word.
 */
pkv_status pkv_get_device_error(const pkv_pool *pool, void *stream, uint32_t *fault_bits);

/*
 * Check of the kernels' watchdog: every shared-memory pipeline wait in the
 * decode kernels gives up after a bound (2 s), records PKV_FAULT_TIMEOUT in
 * the pool's error word and stops, so a copy that never lands cannot hang
 * the GPU.  This call runs that same bounded wait on a barrier nothing
 * arrives at, with limit_ns (1 us .. 2 s) as the bound: after it,
 * pkv_get_device_error reports PKV_FAULT_TIMEOUT and the context is still
 * usable.  The pool must have an error word.  Enqueued on `stream`; takes
 * about limit_ns of GPU time.
 */
pkv_status pkv_check_bounded_wait(const pkv_pool *pool, long long limit_ns, void *stream);

/* Static description of a status code. */
const char *pkv_status_string(pkv_status status);

/*
 * Description of the CUDA error behind the calling thread's most recent
 * PKV_ERR_CUDA (static string; "no CUDA error recorded" if none).
 */
const char *pkv_last_cuda_error(void);

/* Library ABI version (major*100 + minor). */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
