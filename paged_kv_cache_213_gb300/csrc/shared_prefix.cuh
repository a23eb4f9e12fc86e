// shared_prefix.cuh -- the one rule both decode passes use to decide how many
// 16-token tiles of a prefix-shared group are processed by the shared pass.
#pragma once

#include <climits>

#include "mma_tile.cuh"
#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {

// Context length of sequence b, clamped to [0, min(max_blocks_per_seq *
// block_size, max_context_len)] (out-of-range values are flagged elsewhere).
__device__ __forceinline__ int shared_len_of(const DecodeArgs &a, int b) {
    const int L = a.context_lens[b];
    const long long cap_ll = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    const int cap = static_cast<int>(cap_ll < a.max_context_len ? cap_ll : a.max_context_len);
    return L < 0 ? 0 : (L > cap ? cap : L);
}

// Whole tiles of group gi that every member holds inside the shared prefix:
// floor(min(prefix tokens, shortest member) / 16).  min_len is the shortest
// clamped length among the group's members.
__device__ __forceinline__ int shared_tiles(const DecodeArgs &a, int gi, int min_len) {
    int p = a.group_prefix[gi];
    if (p < 0) p = 0;
    return (p < min_len ? p : min_len) / kMmaTile;
}

}  // namespace pkv
