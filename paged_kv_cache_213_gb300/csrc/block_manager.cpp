// block_manager.cpp -- host-side block manager of the paged KV cache: free
// list, reference counts, per-sequence block tables, fork and copy-on-write
// of a shared partially filled tail block.  See include/pagedkv_blocks.h for
// the page passages it follows and the reading adopted where the page's
// listing and its worked solution disagree.
#include <climits>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv_blocks.h"

struct pkv_block_manager {
    struct Seq {
        std::vector<int32_t> table;
        int64_t length = 0;
    };
    int block_size = 0;
    std::vector<int32_t> refcount;  // per physical block
    std::vector<int32_t> filled;    // rows written, per physical block
    std::vector<int32_t> free_list; // LIFO: back() is handed out next
    std::unordered_map<int64_t, Seq> seqs;

    bool allocate(int32_t *out) {
        if (free_list.empty()) return false;
        const int32_t b = free_list.back();
        free_list.pop_back();
        refcount[b] = 1;
        filled[b] = 0;
        *out = b;
        return true;
    }
    void release(int32_t b) {
        if (--refcount[b] <= 0) {
            refcount[b] = 0;
            filled[b] = 0;
            free_list.push_back(b);
        }
    }
};

extern "C" {

pkv_block_manager *pkv_bm_create(int64_t num_blocks, int block_size) {
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
    auto *bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return nullptr;
    try {
        bm->block_size = block_size;
        bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
        bm->filled.assign(static_cast<size_t>(num_blocks), 0);
        bm->free_list.reserve(static_cast<size_t>(num_blocks));
        for (int64_t i = 0; i < num_blocks; ++i) bm->free_list.push_back(static_cast<int32_t>(i));
    } catch (...) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm || bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    bm->seqs.emplace(seq_id, pkv_block_manager::Seq{});
    return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child)) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq copy = it->second;
    for (int32_t b : copy.table) ++bm->refcount[b];
    bm->seqs.emplace(child, std::move(copy));
    return PKV_OK;
}

int pkv_bm_append_slot(pkv_block_manager *bm, int64_t seq_id, int64_t *slot, int32_t *copy_src,
                       int32_t *copy_dst, int32_t *copy_tokens) {
    if (!bm || !slot || !copy_src || !copy_dst || !copy_tokens) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq &s = it->second;
    *copy_src = -1;
    *copy_dst = -1;
    *copy_tokens = 0;
    if (s.table.empty() || bm->filled[s.table.back()] >= bm->block_size) {
        // no tail block, or a full one (shared or not): start a fresh block
        int32_t b;
        if (!bm->allocate(&b)) return PKV_ERR_OUT_OF_BLOCKS;
        s.table.push_back(b);
    } else if (bm->refcount[s.table.back()] > 1) {
        // shared, partially filled tail: clone it, the clone replaces the tail
        const int32_t tail = s.table.back();
        int32_t b;
        if (!bm->allocate(&b)) return PKV_ERR_OUT_OF_BLOCKS;
        --bm->refcount[tail];
        bm->filled[b] = bm->filled[tail];
        *copy_src = tail;
        *copy_dst = b;
        *copy_tokens = bm->filled[tail];
        s.table.back() = b;
    }
    const int32_t tail = s.table.back();
    *slot = static_cast<int64_t>(tail) * bm->block_size + bm->filled[tail];
    ++bm->filled[tail];
    ++s.length;
    return PKV_OK;
}

int pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    for (int32_t b : it->second.table) bm->release(b);
    bm->seqs.erase(it);
    return PKV_OK;
}

int64_t pkv_bm_num_free_blocks(const pkv_block_manager *bm) {
    return bm ? static_cast<int64_t>(bm->free_list.size()) : -1;
}

int pkv_bm_sequence_length(const pkv_block_manager *bm, int64_t seq_id, int64_t *length) {
    if (!bm || !length) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    *length = it->second.length;
    return PKV_OK;
}

int pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *out,
                       int64_t capacity, int64_t *num_blocks) {
    if (!bm || !num_blocks || capacity < 0 || (capacity > 0 && !out)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    const auto &t = it->second.table;
    *num_blocks = static_cast<int64_t>(t.size());
    for (int64_t i = 0; i < capacity && i < static_cast<int64_t>(t.size()); ++i) out[i] = t[i];
    return PKV_OK;
}

int pkv_bm_block_info(const pkv_block_manager *bm, int32_t block, int32_t *refcount,
                      int32_t *tokens) {
    if (!bm || block < 0 || block >= static_cast<int32_t>(bm->refcount.size()))
        return PKV_ERR_INVALID_ARG;
    if (refcount) *refcount = bm->refcount[block];
    if (tokens) *tokens = bm->filled[block];
    return PKV_OK;
}

int pkv_bm_prefix_groups(const pkv_block_manager *bm, const int64_t *seq_ids, int n,
                         int32_t *group_offsets, int32_t *group_prefix_lens, int *num_groups,
                         int *max_group_size, int *max_prefix_len) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !group_offsets || !group_prefix_lens)))
        return PKV_ERR_INVALID_ARG;
    std::vector<const std::vector<int32_t> *> tables(static_cast<size_t>(n));
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
        tables[static_cast<size_t>(i)] = &it->second.table;
    }
    int groups = 0, most = 0, longest = 0;
    if (n > 0) group_offsets[0] = 0;
    for (int i = 0; i < n;) {
        const std::vector<int32_t> &first = *tables[static_cast<size_t>(i)];
        int e = i + 1;
        size_t common = first.size();  // leading entries all members hold in common
        while (e < n && !first.empty() && !tables[static_cast<size_t>(e)]->empty() &&
               (*tables[static_cast<size_t>(e)])[0] == first[0]) {
            const std::vector<int32_t> &t = *tables[static_cast<size_t>(e)];
            size_t c = 0;
            while (c < common && c < t.size() && t[c] == first[c]) ++c;
            common = c;
            ++e;
        }
        const long long prefix = e - i > 1 ? static_cast<long long>(common) * bm->block_size : 0;
        const int p = prefix > INT32_MAX ? INT32_MAX : static_cast<int>(prefix);
        group_prefix_lens[groups] = p;
        group_offsets[++groups] = e;
        if (e - i > most) most = e - i;
        if (p > longest) longest = p;
        i = e;
    }
    if (num_groups) *num_groups = groups;
    if (max_group_size) *max_group_size = most;
    if (max_prefix_len) *max_prefix_len = longest;
    return PKV_OK;
}

}  // extern "C"
