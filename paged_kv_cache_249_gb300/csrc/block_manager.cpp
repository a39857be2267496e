// block_manager.cpp -- host-side manager of the physical block pool.
//
// The pages' memory manager: blocks are handed out as a sequence grows and
// returned when it finishes (on demand rather than reserved up front:
// Qualiteg, "About PagedAttention for LLM serving", "[Regarding Problem 1]",
// point 1-3), each sequence's logical blocks map to physical ones through its
// block table (same page, the section on logical and physical blocks), and
// requests that share a prompt prefix share its
// KV blocks (the prefix-sharing use discussed on the Hacker News page).
// Shared blocks are reference-counted; writing into a shared, partly filled
// last block first moves the writer to a private copy (copy-on-write), which
// the caller performs on the device with pkv_copy_blocks.
//
// Host memory only; no CUDA call.  Not thread-safe: one manager per thread
// or external locking.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pagedkv.h"

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_list;  // stack of free physical blocks
    std::vector<int32_t> refcount;   // per physical block
    struct Seq {
        std::vector<int32_t> blocks;
        int64_t len = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;
    std::vector<std::pair<int32_t, int32_t>> copies;  // pending (src, dst) block copies

    int32_t take() {
        const int32_t b = free_list.back();
        free_list.pop_back();
        refcount[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--refcount[b] == 0) free_list.push_back(b);
    }
};

namespace {

bool fits_table(int64_t tokens, int block_size) {
    return (tokens + block_size - 1) / block_size < (int64_t)1 << 30;
}

}  // namespace

extern "C" {

pkv_status pkv_bm_create(int num_blocks, int block_size, pkv_block_manager **out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return PKV_ERR_OUT_OF_BLOCKS;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refcount.assign(num_blocks, 0);
    bm->free_list.resize(num_blocks);
    // lowest block ids are handed out first
    for (int i = 0; i < num_blocks; ++i) bm->free_list[i] = num_blocks - 1 - i;
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int pkv_bm_free_blocks(const pkv_block_manager *bm) {
    return bm ? (int)bm->free_list.size() : -1;
}

int pkv_bm_refcount(const pkv_block_manager *bm, int32_t block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->refcount[block];
}

pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id, int64_t num_tokens,
                               int64_t *slots) {
    if (!bm || num_tokens < 0 || !fits_table(num_tokens, bm->block_size))
        return PKV_ERR_INVALID_ARG;
    if (bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    const int64_t need = (num_tokens + bm->block_size - 1) / bm->block_size;
    if (need > (int64_t)bm->free_list.size()) return PKV_ERR_OUT_OF_BLOCKS;
    pkv_block_manager::Seq seq;
    seq.blocks.reserve(need);
    for (int64_t i = 0; i < need; ++i) seq.blocks.push_back(bm->take());
    seq.len = num_tokens;
    if (slots)
        for (int64_t t = 0; t < num_tokens; ++t)
            slots[t] = (int64_t)seq.blocks[t / bm->block_size] * bm->block_size + t % bm->block_size;
    bm->seqs.emplace(seq_id, std::move(seq));
    return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child)) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq seq = it->second;  // same physical blocks
    for (int32_t b : seq.blocks) ++bm->refcount[b];
    bm->seqs.emplace(child, std::move(seq));
    return PKV_OK;
}

pkv_status pkv_bm_append_token(pkv_block_manager *bm, int64_t seq_id, int64_t *slot) {
    if (!bm || !slot) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq &seq = it->second;
    if (!fits_table(seq.len + 1, bm->block_size)) return PKV_ERR_INVALID_ARG;
    const int64_t pos = seq.len;
    const int64_t lb = pos / bm->block_size;
    if (lb == (int64_t)seq.blocks.size()) {
        if (bm->free_list.empty()) return PKV_ERR_OUT_OF_BLOCKS;
        seq.blocks.push_back(bm->take());
    } else if (bm->refcount[seq.blocks[lb]] > 1) {
        // copy-on-write: the partly filled last block is shared
        if (bm->free_list.empty()) return PKV_ERR_OUT_OF_BLOCKS;
        const int32_t src = seq.blocks[lb];
        const int32_t dst = bm->take();
        bm->release(src);
        seq.blocks[lb] = dst;
        bm->copies.emplace_back(src, dst);
    }
    seq.len = pos + 1;
    *slot = (int64_t)seq.blocks[lb] * bm->block_size + pos % bm->block_size;
    return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    for (int32_t b : it->second.blocks) bm->release(b);
    bm->seqs.erase(it);
    return PKV_OK;
}

int64_t pkv_bm_context_len(const pkv_block_manager *bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : it->second.len;
}

int pkv_bm_take_copies(pkv_block_manager *bm, int32_t *src, int32_t *dst, int capacity) {
    if (!bm || capacity < 0 || (capacity > 0 && (!src || !dst))) return -1;
    const int n = std::min<int>(capacity, (int)bm->copies.size());
    for (int i = 0; i < n; ++i) {
        src[i] = bm->copies[i].first;
        dst[i] = bm->copies[i].second;
    }
    bm->copies.erase(bm->copies.begin(), bm->copies.begin() + n);
    return n;
}

int pkv_bm_pending_copies(const pkv_block_manager *bm) {
    return bm ? (int)bm->copies.size() : -1;
}

pkv_status pkv_bm_block_tables(const pkv_block_manager *bm, const int64_t *seq_ids, int num_seqs,
                               int max_blocks_per_seq, int32_t *block_tables,
                               int32_t *context_lens) {
    if (!bm || num_seqs < 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!seq_ids || !block_tables || !context_lens)) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < num_seqs; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
        const auto &seq = it->second;
        if ((int64_t)seq.blocks.size() > max_blocks_per_seq || seq.len > INT32_MAX)
            return PKV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < num_seqs; ++i) {
        const auto &seq = bm->seqs.find(seq_ids[i])->second;
        int32_t *row = block_tables + (size_t)i * max_blocks_per_seq;
        std::fill(row, row + max_blocks_per_seq, -1);
        std::copy(seq.blocks.begin(), seq.blocks.end(), row);
        context_lens[i] = (int32_t)seq.len;
    }
    return PKV_OK;
}

pkv_status pkv_bm_shared_prefix(const pkv_block_manager *bm, const int64_t *seq_ids, int num_seqs,
                                const int32_t *group_starts, int num_groups,
                                int32_t *prefix_lens) {
    if (!bm || num_seqs < 0 || num_groups < 0) return PKV_ERR_INVALID_ARG;
    if (num_groups == 0) return num_seqs == 0 ? PKV_OK : PKV_ERR_INVALID_ARG;
    if (!group_starts || !prefix_lens || (num_seqs > 0 && !seq_ids)) return PKV_ERR_INVALID_ARG;
    if (group_starts[0] != 0 || group_starts[num_groups] != num_seqs) return PKV_ERR_INVALID_ARG;
    std::vector<const pkv_block_manager::Seq *> rows((size_t)num_seqs);
    for (int i = 0; i < num_seqs; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
        rows[(size_t)i] = &it->second;
    }
    for (int g = 0; g < num_groups; ++g)
        if (group_starts[g] > group_starts[g + 1]) return PKV_ERR_INVALID_ARG;
    for (int g = 0; g < num_groups; ++g) {
        const int a = group_starts[g], b = group_starts[g + 1];
        int64_t common = 0;
        if (b - a >= 2) {
            // leading blocks that every member holds, full in every member
            int64_t full = INT64_MAX;
            for (int i = a; i < b; ++i) full = std::min(full, rows[(size_t)i]->len / bm->block_size);
            while (common < full) {
                const int32_t blk = rows[(size_t)a]->blocks[(size_t)common];
                bool same = true;
                for (int i = a + 1; i < b && same; ++i) same = rows[(size_t)i]->blocks[(size_t)common] == blk;
                if (!same) break;
                ++common;
            }
        }
        const int64_t tokens = common * bm->block_size;
        prefix_lens[g] = tokens > INT32_MAX ? INT32_MAX / bm->block_size * bm->block_size : (int32_t)tokens;
    }
    return PKV_OK;
}

}  // extern "C"
