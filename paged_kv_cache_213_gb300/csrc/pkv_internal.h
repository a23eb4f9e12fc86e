// pkv_internal.h -- launch interfaces between the C ABI layer (api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "pagedkv.h"

namespace pkv {

// Launch with the programmatic stream-serialization attribute, so that the
// kernel's CTAs may be scheduled while the previous kernel in the stream
// drains; the kernel must call grid_dependency_wait() before touching memory
// that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct AppendArgs {
    const void *k_new;
    const void *v_new;
    const int64_t *slot_mapping;
    void *k_cache;
    void *v_cache;
    int num_tokens;
    int n_kv_heads;
    int head_dim;
    int block_size;
    int64_t num_blocks;
    int32_t *err;
};

struct DecodeArgs {
    void *out;                    // fp16 [B][H][D]
    const void *q;                // fp16 [B][H][D]
    const void *k_cache;          // fp16 [NB][Hk][bs][D]
    const void *v_cache;
    const int32_t *block_tables;  // [B][MB]
    const int32_t *context_lens;  // [B]
    float *ws_acc;                // [B][H][max_parts][D]  unnormalised partial sums
    float *ws_m;                  // [B][H][max_parts]     partial max (log2 units)
    float *ws_l;                  // [B][H][max_parts]     partial sum of 2^(s - m)
    float *lse_out;               // [B][H] or null
    int32_t *err;                 // or null
    int num_seqs;
    int max_blocks_per_seq;
    int64_t num_blocks;
    float scale_log2;             // scale * log2(e)
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    int block_size;
    int max_context_len;          // clamp bound, > 0
    int partition_tokens;         // multiple of 16 and of block_size
    int max_parts;                // ceil(max_context_len / partition_tokens)
    // prefix-shared groups (num_groups = 0: none)
    const int32_t *group_offsets; // [num_groups + 1] consecutive ranges of sequences
    const int32_t *group_prefix;  // [num_groups] shared prefix tokens
    int num_groups;
    int sh_chunks;                // CTA chunks per group in the shared pass
    int sh_parts;                 // partitions of the shared prefix
    int sh_part_tiles;            // 16-token tiles per partition
    int sh_warps;                 // warps per shared-pass CTA
    int sh_tables_ready = 0;      // shared pass: the kernel before writes no
                                  // lengths, tables or groups (PKV_TABLES_READY)
    float *sh_acc;                // [B][H][sh_parts][D] shared-pass partial sums
    float *sh_m;                  // [B][H][sh_parts]
    float *sh_l;                  // [B][H][sh_parts]
    // Where the balanced kernel waits for the kernel before it in the stream
    // (programmatic dependent launch):
    //  0: first thing;
    //  1: the kernel before is the shared-prefix pass, which writes only
    //     sh_acc / sh_m / sh_l: prologue and private tiles run before the
    //     wait, which comes before the first read of those partials;
    //  2: the kernel before writes no lengths or tables (this library's
    //     append, or a caller's kernel under PKV_TABLES_READY): the prologue
    //     (lengths, block ids, split; under fuse_append also the check of
    //     empty sequences' slots) runs before the wait, which comes before
    //     the first read of q, the caches, the appended rows or the
    //     workspace.
    int defer_dep_wait;
    // FP8 caches (balanced kernel only): k_cache / v_cache hold E4M3 codes,
    // scale_log2 already includes k_scale, and outputs are multiplied by v_scale
    int kv_fp8 = 0;
    float v_scale = 1.f;          // 1 for fp16 caches
    // multi-token attention: q, out, lse rows are query tokens; sequence b owns
    // rows [query_start[b], query_start[b+1]) (its last tokens, causal)
    const int32_t *query_start = nullptr;
    int total_q = 0;
    int max_q_len = 0;            // host bound of n_b; a longer sequence is flagged
    // The append inside the attention kernel (paged_decode_step under
    // PKV_APPEND_NEWEST; fp16 caches, per-warp balanced split only): token b
    // of append_k / append_v ([B][Hk][D] fp16) is sequence b's newest token,
    // at slot append_slots[b] (negative: no token).  The warp that loads a
    // segment's last tile writes the token's rows to the cache and into that
    // tile in shared memory, so no separate append kernel runs before.
    const void *append_k = nullptr;
    const void *append_v = nullptr;
    const int64_t *append_slots = nullptr;
    int fuse_append = 0;
    // Test hook (the environment variable PKV_TEST_WAIT_POLLS, read at every
    // call): >= 0 makes each warp's first wait for K/V data give up after
    // that many non-blocking polls, so that the timeout path (flag, drain the
    // copies in flight, stop) runs without a fault; -1 (unset) leaves every
    // wait at its one-second bound.
    int first_wait_polls = -1;
};
// The test hook's value for this call (-1 when PKV_TEST_WAIT_POLLS is unset).
int test_wait_polls();

// The balanced kernel's workspace starts with one int32 arrival counter per
// worker slot, kBalancedCounterBytes in all, whatever the plan (the
// producer/consumer kernel keeps its counters there too).  They must be zero
// when a launch starts.  Each of the n pieces of a cut segment adds 1 to the
// segment's counter; the one that sees n - 1 merges, then subtracts n (a
// reduction without a result, which the warp does not wait for), so a
// correct launch leaves the counter zero.  An arrival that sees a value >= n
// (unsigned) proves that the counter did not start at zero: it flags
// PKV_ERRBIT_WORKSPACE and sets the counter to kCounterPoison, which every
// later arrival, in this launch and the next ones, also sees as >= n, even
// after a merge's subtraction.  A stale start c is thus always caught when it
// is negative or >= n (the first arrival sees c).  A c in [1, n) lets the
// arrival that sees n - 1 merge early; it is caught when another piece
// arrives before that merge's subtraction, and missed otherwise.
constexpr int kBalancedMaxWorkers = 16384;
constexpr size_t kBalancedCounterBytes = static_cast<size_t>(kBalancedMaxWorkers) * 4;
static_assert(kBalancedCounterBytes == PKV_WORKSPACE_COUNTER_BYTES,
              "the header states the counter region's size");
constexpr int kCounterPoison = 1 << 30;
static_assert(2 * kBalancedMaxWorkers < kCounterPoison,
              "a poisoned count stays >= n after a merge subtracts n");

// True when an arrival that saw `old` on a counter of `last + 1` pieces
// proves that the counter did not start at zero.
__host__ __device__ inline bool counter_not_zeroed(int old, int last) {
    return static_cast<unsigned>(old) > static_cast<unsigned>(last);
}

// Workspace carve-up shared by the planner and the launcher.
struct WorkspaceLayout {
    size_t acc_offset, m_offset, l_offset, total;
};
WorkspaceLayout workspace_layout(int num_seqs, int n_q_heads, int head_dim, int max_parts);

cudaError_t launch_append(const AppendArgs &a, cudaStream_t stream);
// dst <- src, 16 bytes per thread (both 16-byte aligned, bytes a multiple of
// 16); src may be mapped host memory.
cudaError_t launch_copy_in(void *dst, const void *src, size_t bytes, cudaStream_t stream);
// FP8 (E4M3) caches: k_cache / v_cache hold one byte per value, head_dim % 16 == 0.
cudaError_t launch_append_f8(const AppendArgs &a, float k_scale, float v_scale,
                             cudaStream_t stream);
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *src,
                               const int32_t *dst, const int32_t *tokens, int num_copies,
                               int n_kv_heads, int head_dim, int block_size, long long num_blocks,
                               int32_t *err, cudaStream_t stream);
// Returns cudaErrorInvalidValue for a (head_dim, group) pair with no kernel.
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
bool decode_supported(int head_dim, int group);
// PKV_DECODE_KERNEL: 0 unset (automatic), 1 "simt", 2 "mma" (the grid kernels),
// 3 "warp" (the balanced split on per-warp ranges), 4 "pipe" (the balanced
// split on the producer/consumer kernel).
int kernel_override();
// Tensor-core kernel (decode_mma.cu): partition pass only, no merge.
bool decode_mma_supported(const DecodeArgs &a);
cudaError_t launch_decode_mma(const DecodeArgs &a, cudaStream_t stream);
// 2-D TMA map [rows][D] fp16 of a cache, 16x64 boxes, 128-byte swizzle.
bool make_cache_map(CUtensorMap *m, const void *base, long long rows, int D);
// The same over an E4M3 cache (one byte per element): one box is a whole
// 16-row tile, D bytes wide, with the D-byte swizzle (128B or 64B).
bool make_cache_map_e4m3(CUtensorMap *m, const void *base, long long rows, int D);

// Balanced (work-split per warp) tensor-core kernel (decode_balanced.cu).
struct BalancedPlan {
    int ctas;        // grid size
    int warps;       // warps per CTA
    int workers;     // units of the split: warps (kind 0) or CTAs (kind 1)
    size_t ws_bytes; // workspace bytes
    int kind = 0;    // 0: per-warp ranges (decode_balanced.cu); 1: producer/consumer
                     // CTAs (decode_pipeline.cu)
    int heads = 0;   // kind 1: KV heads per unit
};
bool balanced_supported(int num_seqs, int head_dim, int group, int block_size,
                        long long cache_rows);
// Grid and workspace for the balanced kernel (host query of the SM count
// and occupancy); false if the device query fails.
bool balanced_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int max_len,
                   BalancedPlan *plan, bool kv_fp8 = false);
cudaError_t launch_decode_balanced(const DecodeArgs &a, const BalancedPlan &plan,
                                   cudaStream_t stream);
// The producer/consumer kernel (decode_pipeline.cu): fp16 caches, no prefix
// groups, n_kv_heads 1, 2, 4 or a multiple of 8; a one-wave grid of CTAs,
// each over an equal range of (head group, sequence, 16-token tile) units.
bool pipeline_supported(int num_seqs, int n_kv_heads, int head_dim, int group, int block_size,
                        long long cache_rows);
bool pipeline_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int max_len,
                   BalancedPlan *plan);
cudaError_t launch_decode_pipeline(const DecodeArgs &a, const BalancedPlan &plan,
                                   cudaStream_t stream);
// Shared-prefix pass (decode_shared.cu): each warp holds 16 query rows.
int shared_members_per_warp(int group);
int shared_max_warps();
int shared_ctas_per_sm(int head_dim, int group, int warps, bool kv_fp8 = false);
cudaError_t launch_decode_shared(const DecodeArgs &a, cudaStream_t stream);
// Multi-token causal attention (decode_multi.cu): grid (max_parts, Hk x row
// blocks, B) plus the merge kernel when max_parts > 1; workspace as
// workspace_layout(total_q, n_q_heads, head_dim, max_parts).
int multi_row_blocks(int max_q_len, int group);
cudaError_t launch_decode_multi(const DecodeArgs &a, int row_blocks, cudaStream_t stream);
// Multi-token attention on the balanced split (decode_balanced_multi.cu):
// max_q_len * group <= 16 query rows per segment, fp16 caches; workspace as
// for the balanced decode, with 16-row records (zeroed counters first).
bool balanced_multi_supported(int num_seqs, int max_q_len, int head_dim, int group,
                              int block_size);
bool balanced_multi_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int max_len,
                         BalancedPlan *plan);
cudaError_t launch_decode_balanced_multi(const DecodeArgs &a, const BalancedPlan &plan,
                                         cudaStream_t stream);

}  // namespace pkv
