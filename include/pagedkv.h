/*
 * pagedkv.h -- C ABI of the paged KV cache decode path for GB300 (sm_103a).
 *
 * Two operations, both asynchronous on the caller's CUDA stream:
 *
 *  paged_kv_append         writes each sequence's newest token K/V into its
 *                          slot of the block pool;
 *  paged_decode_attention  attends every sequence's newest query over all of
 *                          its cached tokens, gathered through its block table.
 *
 * Sources (page title, section):
 *  - "Distributed LLM Inference Serving Platform", section 2 (Mental Model &
 *    Architectural Abstraction): a sequence's KV cache is split into
 *    fixed-size logical blocks (16 tokens) mapped to non-contiguous physical
 *    blocks of one HBM pool by a per-sequence block table; prompt blocks may
 *    be shared by several sequences (copy-on-write, reference counts).
 *  - same page, section 3 (Core Terminology, PagedAttention row): the
 *    attention kernel reads K and V through the page tables.
 *  - same page, section 5.1 (End-to-End Request Lifecycle): each decode step
 *    every active sequence submits its latest token, its K/V are written into
 *    the assigned physical block (a new block when the tail block is full),
 *    and attention runs over all blocks in the sequence's table.
 *  - same page, section 1 and the Lab 3 roofline solution (nHeads = 64,
 *    nKvHeads = 8): grouped-query attention, query head h reads KV head
 *    h / (n_q_heads / n_kv_heads).
 *  - "Roadmap: vLLM-style serving features for TornadoVM batched decode",
 *    Serving / scheduling list: block-pool KV with a per-slot block table.
 *
 * Data layout (the pages fix none; this is the library's reading):
 *  - k_cache, v_cache: fp16 (IEEE binary16) [num_blocks][n_kv_heads]
 *    [block_size][head_dim], contiguous.  Token t of sequence b, KV head j
 *    lives at row t % block_size of physical block block_tables[b][t /
 *    block_size].
 *  - block_tables: int32 [num_seqs][max_blocks_per_seq], row-major.  Only the
 *    first ceil(context_lens[b] / block_size) entries of row b are read.
 *  - context_lens: int32 [num_seqs]; sequence b attends tokens
 *    [0, context_lens[b]) -- the token appended this step included.
 *  - slot_mapping: int64 [num_tokens]; slot = physical_block * block_size +
 *    row; a negative slot marks a padding token that is skipped.
 *  - q, out: fp16 [num_seqs][n_q_heads][head_dim]; k_new, v_new: fp16
 *    [num_tokens][n_kv_heads][head_dim]; lse_out: fp32 [num_seqs][n_q_heads].
 *
 * Ownership: every pointer is a device pointer the caller allocates and owns
 * (except where a host pointer is stated).  The library allocates no memory
 * and keeps no state besides a cached per-device attribute lookup (and the
 * static scratch array of paged_decode_attention_noalloc).  Tensor
 * pointers (q, out, caches, k_new, v_new) must be 16-byte aligned.
 *
 * Errors: a call that detects a bad argument on the host returns a negative
 * pkv_status and launches nothing.  Problems only the device can see (a
 * block id outside [0, num_blocks), a slot beyond the pool, a context length
 * outside [0, max_blocks_per_seq * block_size] or above max_context_len, a
 * copy that did not complete within about a second, a workspace whose
 * arrival counters did not start at zero) set bits in the optional
 * device word *err_word (PKV_ERRBIT_*): the offending block or token is
 * skipped, nothing traps, and the result for that sequence is unspecified.
 * Read the word with paged_kv_get_error.  Launch failures return
 * PKV_ERR_CUDA.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1, /* null or misaligned pointer, bad size, n_q % n_kv != 0 */
    PKV_ERR_UNSUPPORTED = -2, /* head_dim, block_size or group size not built */
    PKV_ERR_WORKSPACE = -3,   /* workspace missing or smaller than paged_decode_plan says */
    PKV_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
    PKV_ERR_INDEX = -5        /* the device flagged a bad index (see the error word) */
} pkv_status;

/* Bits of the device error word. */
#define PKV_ERRBIT_BLOCK_ID 0x1 /* block table entry outside [0, num_blocks) */
#define PKV_ERRBIT_SLOT 0x2     /* slot_mapping entry >= num_blocks * block_size */
#define PKV_ERRBIT_CONTEXT 0x4  /* context length < 0, > max_blocks_per_seq*block_size,
                                   or > max_context_len */
#define PKV_ERRBIT_TIMEOUT 0x8  /* a bounded wait for a block copy gave up */
#define PKV_ERRBIT_WORKSPACE 0x10 /* an arrival counter of the workspace did not
                                     start at zero (see PKV_WORKSPACE_COUNTER_BYTES) */
#define PKV_ERRBIT_APPEND 0x20  /* under PKV_APPEND_NEWEST, a token that is not its
                                   sequence's newest (see paged_decode_step_ex) */

/*
 * Every call that keeps split-K arrival counters (the balanced split, the
 * producer/consumer split and the multi-token balanced split) keeps them in
 * the first PKV_WORKSPACE_COUNTER_BYTES bytes of its workspace, or in the
 * whole workspace when that is smaller.  Those bytes must be zero when the
 * call's kernel starts; each call leaves them zero again unless it flagged
 * PKV_ERRBIT_TIMEOUT or PKV_ERRBIT_WORKSPACE; paged_decode_workspace_clear
 * zeroes them.  A kernel that meets a counter holding a value no zeroed
 * workspace can produce sets PKV_ERRBIT_WORKSPACE.  That is certain when the
 * stale value is negative or at least the number of pieces counted on it
 * (a float's or a pointer's bit pattern, -1); a small positive stale value
 * is caught only when a piece arrives before the early merge it causes.
 * After the flag the results of the sequences whose split was counted are
 * unspecified (some may be left unwritten); nothing faults or waits on a
 * count, and the caller clears the counters before the next call.  The rest
 * of a workspace is written before it is read within a call.
 */
#define PKV_WORKSPACE_COUNTER_BYTES 65536

/*
 * Slot-mapped append ("Distributed LLM Inference Serving Platform", section
 * 5.1, Chunked Prefill and Continuous Decode Loop items): for token i and KV
 * head j, copies k_new[i][j][:] and v_new[i][j][:] bit for bit into row
 * slot_mapping[i] % block_size of physical block slot_mapping[i] / block_size.
 *
 *  k_new, v_new   device, fp16 [num_tokens][n_kv_heads][head_dim]
 *  slot_mapping   device, int64 [num_tokens]; < 0 = skip
 *  k_cache, v_cache device, fp16 [num_blocks][n_kv_heads][block_size][head_dim]
 *  head_dim       a multiple of 8
 *  err_word       device int32, may be NULL; PKV_ERRBIT_SLOT is or-ed in for a
 *                 slot >= num_blocks * block_size (that token is skipped)
 *  cuda_stream    cudaStream_t (NULL = legacy default stream)
 * Two tokens with the same slot in one call: which one lands is unspecified.
 * num_tokens == 0 is a no-op.
 */
int paged_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                    void *k_cache, void *v_cache, int num_tokens, int n_kv_heads,
                    int head_dim, int block_size, int64_t num_blocks, int32_t *err_word,
                    void *cuda_stream);

/*
 * Split planning for paged_decode_attention (host only; no device work).
 * partition_tokens = 0 asks for the automatic choice, which depends on the
 * current device (SM count and occupancy; a CUDA query that fails with
 * PKV_ERR_CUDA when no device is present).  For block sizes that are a
 * multiple of 16 and up to 2048 sequences the automatic choice is the
 * balanced split: the (sequence, KV head, 16-token tile) work units are cut
 * into equal contiguous ranges, one per warp of a grid that fills the GPU
 * once, and segments cut by a range boundary are merged by log-sum-exp.
 * Otherwise it is a fixed partition size.  A nonzero partition_tokens selects
 * fixed partitions of that many tokens and is checked and echoed: a positive
 * multiple of 16 and of block_size with partition_tokens / block_size <= 2048.
 *  max_context_len <= 0 means max_blocks_per_seq * block_size.
 *  *partition_tokens_out  (host, may be NULL) tokens per fixed partition, or
 *                         0 for the balanced split
 *  *workspace_bytes_out   (host, may be NULL) workspace the call needs; 0 when
 *                         every sequence fits one fixed partition
 */
int paged_decode_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                      int block_size, int max_blocks_per_seq, int max_context_len,
                      int partition_tokens, int *partition_tokens_out,
                      size_t *workspace_bytes_out);

/*
 * Paged decode attention ("Distributed LLM Inference Serving Platform",
 * sections 2, 3 and 5.1; grouped-query mapping from section 1):
 *
 *   out[b][h][:] = sum_t softmax_t(scale * q[b][h] . K_t) V_t,  t in [0, L_b)
 *
 * with K_t, V_t the rows of KV head h / (n_q_heads / n_kv_heads) gathered
 * through block_tables[b].  Logits and the softmax run in fp32 (online
 * max/sum rescaling); the output is rounded to fp16 (round to nearest even).
 * Long contexts are split (balanced split or fixed partitions, see
 * paged_decode_plan) and the partial results merged by log-sum-exp
 * (flash-decoding split).
 * L_b = 0 gives out = 0 and lse = -inf.
 *
 *  out            fp16 [num_seqs][n_q_heads][head_dim], device memory or pinned
 *                 (page-locked, mapped) host memory: the kernels write it with
 *                 plain stores, so with a host buffer the results reach the
 *                 host as they are written, with no copy after the call
 *  q              device fp16 [num_seqs][n_q_heads][head_dim]
 *  k_cache, v_cache, block_tables, context_lens   as in the layout notes
 *  scale          multiplies q . K before the softmax (1/sqrt(head_dim) usually)
 *  head_dim       64 or 128;  block_size 1, 2, 4, 8, 16, 32, 64, 128 or 256;
 *                 n_q_heads / n_kv_heads in {1, 2, 4, 8}
 *  max_context_len an upper bound on every context length (no device sync
 *                 is needed to know it); <= 0 means max_blocks_per_seq*block_size
 *  partition_tokens 0 = automatic (see paged_decode_plan)
 *  workspace      device scratch of at least the planned bytes (256-byte
 *                 aligned), may be NULL when the plan needs 0 bytes; the
 *                 caller owns it; calls that overlap in time need separate
 *                 workspaces.  Its first PKV_WORKSPACE_COUNTER_BYTES bytes
 *                 must be zero before its first use (a whole zero-filled
 *                 workspace will do): the balanced split keeps per-segment
 *                 arrival counters there, and every call leaves them zero
 *                 again (after a call that flagged PKV_ERRBIT_TIMEOUT or
 *                 PKV_ERRBIT_WORKSPACE, zero them once more)
 *  lse_out        device fp32 [num_seqs][n_q_heads] natural-log sum of
 *                 exp(logits), may be NULL
 *  err_word       device int32, may be NULL (see the header comment)
 *  cuda_stream    cudaStream_t
 */
int paged_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens,
                           int num_seqs, int max_blocks_per_seq, int64_t num_blocks,
                           float scale, int n_q_heads, int n_kv_heads, int head_dim,
                           int block_size, int max_context_len, int partition_tokens,
                           void *workspace, size_t workspace_bytes, float *lse_out,
                           int32_t *err_word, void *cuda_stream);

/*
 * paged_decode_attention with launch flags.  The pages have no counterpart:
 * this is how the call overlaps the kernel before it on the stream.
 *  PKV_TABLES_READY  the caller guarantees that the kernel launched just
 *                    before this call on cuda_stream (if any) writes neither
 *                    context_lens nor block_tables -- in a decode loop the
 *                    tables are copied in before the layers run, and the
 *                    kernel before the attention writes q and the caches.
 *                    The call then reads the lengths and block ids and
 *                    plans its work split while that kernel drains
 *                    (programmatic dependent launch), and waits for it only
 *                    before it reads q, the caches or the workspace.  If the
 *                    guarantee does not hold, the results are unspecified.
 * flags = 0 is paged_decode_attention.  The flag takes effect on the
 * balanced split (partition_tokens = 0); fixed partitions ignore it.  Other
 * unknown flag bits are rejected with PKV_ERR_INVALID_ARG.
 */
#define PKV_TABLES_READY 0x1u
int paged_decode_attention_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *context_lens,
                              int num_seqs, int max_blocks_per_seq, int64_t num_blocks,
                              float scale, int n_q_heads, int n_kv_heads, int head_dim,
                              int block_size, int max_context_len, int partition_tokens,
                              void *workspace, size_t workspace_bytes, float *lse_out,
                              int32_t *err_word, void *cuda_stream, uint32_t flags);

/*
 * One decode step in one call: paged_kv_append of num_tokens new tokens, then
 * paged_decode_attention, on cuda_stream.  Same arguments, results and errors
 * as the two calls in sequence (the attention's arguments are checked first,
 * so a rejected call writes nothing).  Because the kernel before the
 * attention is then known to write only the caches, the attention's prologue
 * (context lengths, block-table reads, work split) runs while the append
 * drains, and only its first K/V load waits for the append (programmatic
 * dependent launch).  The pages have no separate call for this; section 5.1
 * of "Distributed LLM Inference Serving Platform" describes the two steps of
 * one decode iteration.
 */
int paged_decode_step(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                      int num_tokens, void *out, const void *q, void *k_cache, void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                      int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads,
                      int n_kv_heads, int head_dim, int block_size, int max_context_len,
                      int partition_tokens, void *workspace, size_t workspace_bytes,
                      float *lse_out, int32_t *err_word, void *cuda_stream);

/*
 * paged_decode_step with flags.  The pages have no counterpart: this is how
 * one decode step runs as one kernel.
 *  PKV_APPEND_NEWEST  the caller guarantees that num_tokens == num_seqs and
 *                     that token b is sequence b's newest token:
 *                     slot_mapping[b] is the slot of position
 *                     context_lens[b] - 1 of sequence b (block
 *                     block_tables[b][(L - 1) / block_size], row
 *                     (L - 1) % block_size), or negative for no token.  The
 *                     attention kernel then does the append itself: the warp
 *                     that loads a sequence's last 16-token tile writes the
 *                     token's K/V rows to the cache and into that tile, so no
 *                     append kernel runs and no wait for one.  Results and
 *                     cache contents are those of paged_decode_step.  A token
 *                     whose slot is not its sequence's newest position, or
 *                     that belongs to an empty sequence, sets
 *                     PKV_ERRBIT_APPEND; the former is still written to its
 *                     slot, but the results of any sequence that reads that
 *                     slot are then unspecified.
 *  PKV_TABLES_READY   with PKV_APPEND_NEWEST, as for
 *                     paged_decode_attention_ex, where the kernel before
 *                     also writes no slot_mapping: the step's prologue runs
 *                     while that kernel drains.
 * The flags take effect where the step runs the balanced split on per-warp
 * ranges (block_size a multiple of 16, partition_tokens 0, batches of few
 * (sequence, KV head) segments); elsewhere the call is paged_decode_step.
 * Other flag bits are rejected with PKV_ERR_INVALID_ARG.
 */
#define PKV_APPEND_NEWEST 0x2u
int paged_decode_step_ex(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                         int num_tokens, void *out, const void *q, void *k_cache, void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                         int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads,
                         int n_kv_heads, int head_dim, int block_size, int max_context_len,
                         int partition_tokens, void *workspace, size_t workspace_bytes,
                         float *lse_out, int32_t *err_word, void *cuda_stream, uint32_t flags);

/*
 * How many kernels paged_decode_step_ex launches for these sizes and flags
 * (fp16 caches; the E4M3 step launches the append and the attention)
 * (host only; the automatic split queries the current device, as
 * paged_decode_plan does): the append unless the attention does it
 * (PKV_APPEND_NEWEST on per-warp ranges), then one attention kernel, or two
 * for fixed partitions with a merge.  *launches_out (host) receives it.
 * Returns the status that paged_decode_plan would, or PKV_ERR_INVALID_ARG
 * for unknown flag bits.
 */
int paged_decode_step_launches(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                               int block_size, int max_blocks_per_seq, int max_context_len,
                               int partition_tokens, int num_tokens, uint32_t flags,
                               int *launches_out);

/*
 * Prefix-aware (cascade) decode attention ("Distributed LLM Inference Serving
 * Platform", section 2 and Lab 1: prompt blocks shared by parallel
 * completions; section 5.1 Ingestion: a cached common prefix referenced by
 * several requests).  Same result as paged_decode_attention, but the leading
 * blocks that a group of sequences shares are read from HBM once per chunk
 * of up to 64 / (n_q_heads / n_kv_heads) members instead of once per member:
 * a first pass attends every member's queries over the shared tiles, the
 * balanced pass attends each member's private suffix and merges the two by
 * log-sum-exp.
 *
 *  group_offsets      device int32 [num_groups + 1], non-decreasing, with
 *                     group_offsets[0] = 0 and group_offsets[num_groups] =
 *                     num_seqs: group i is sequences [offsets[i],
 *                     offsets[i+1])
 *  group_prefix_lens  device int32 [num_groups]: tokens whose blocks every
 *                     member of the group holds at the same logical index as
 *                     the group's first sequence (same physical block ids).
 *                     The shared pass uses floor(min(prefix, shortest member)
 *                     / 16) whole tiles; the rest is private.  Groups of one
 *                     sequence, or with prefix 0, have no shared pass.
 *  max_group_size, max_prefix_len   host upper bounds (grid sizing)
 * Other arguments as paged_decode_attention (partition_tokens is implied:
 * the balanced split).  Needs block_size a multiple of 16 and at most 2048
 * sequences (PKV_ERR_UNSUPPORTED otherwise).  If a member's table does not
 * hold the group's first sequence's block ids for the shared prefix, that
 * member's result uses the first sequence's blocks there.
 * When the groups' shared blocks take at most a quarter of the L2 cache
 * (num_groups * max_prefix_len * n_kv_heads * head_dim * 4 bytes), or no
 * group has two members, the call runs paged_decode_attention instead: its
 * reads of blocks shared by several sequences then hit L2, so the shared
 * pass would only add work.  The environment variable PKV_PREFIX_PASS=shared
 * (or =regular), read at every call, fixes the choice.
 * paged_decode_prefix_shared_plan gives the workspace bytes (for whichever
 * path the call takes); its counter bytes (PKV_WORKSPACE_COUNTER_BYTES) must
 * be zero before first use, as for the balanced split.  pkv_bm_prefix_groups
 * (pagedkv_blocks.h) derives the groups from the library's block manager.
 */
int paged_decode_prefix_shared_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                                    int block_size, int max_blocks_per_seq, int max_context_len,
                                    int num_groups, int max_group_size, int max_prefix_len,
                                    size_t *workspace_bytes_out);
int paged_decode_attention_prefix_shared(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads, int n_kv_heads,
    int head_dim, int block_size, int max_context_len, const int32_t *group_offsets,
    const int32_t *group_prefix_lens, int num_groups, int max_group_size, int max_prefix_len,
    void *workspace, size_t workspace_bytes, float *lse_out, int32_t *err_word,
    void *cuda_stream);

/*
 * FP8 KV cache.  "Roadmap: vLLM-style serving features for TornadoVM batched
 * decode", KV-cache list, names a quantized (Q8/FP8) KV cache as future work
 * and fixes no format; this library's reading:
 *  - k_cache, v_cache hold one byte per value: OCP FP8 E4M3 codes ("e4m3fn":
 *    1 sign, 4 exponent bits with bias 7, 3 fraction bits, no infinities,
 *    S.1111.111 is NaN, largest finite 448), same [num_blocks][n_kv_heads]
 *    [block_size][head_dim] layout as the fp16 caches (a 16 x 128 tile is
 *    2 KiB);
 *  - one scale per cache tensor (k_scale, v_scale; finite, > 0), chosen by
 *    the caller, e.g. max |value| / 448;
 *  - paged_kv_append_fp8 stores code = E4M3(fp32(x) / k_scale) for each fp16
 *    value x of k_new (v_scale for v_new): one correctly rounded fp32
 *    division, then round to nearest, ties to even, with finite overflow and
 *    infinities saturated to +-448 (a NaN stores a NaN code);
 *  - paged_decode_attention_fp8 attends over the values code * k_scale and
 *    code * v_scale, with the same results as paged_decode_attention
 *    otherwise (fp32 accumulation, fp16 out, lse).
 * Requirements: head_dim % 16 == 0 for the append; the attention runs on the
 * balanced split only (head_dim 64 or 128, n_q/n_kv in {1, 2, 4, 8},
 * block_size a multiple of 16, at most 2048 sequences; PKV_ERR_UNSUPPORTED
 * otherwise).  paged_decode_plan_fp8 gives its workspace bytes; its counter
 * bytes (PKV_WORKSPACE_COUNTER_BYTES) must be zero before its first use, as
 * for the fp16 call.
 * Pointers, errors and ownership as for the fp16 calls.
 */
int paged_kv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                        void *k_cache, void *v_cache, int num_tokens, int n_kv_heads,
                        int head_dim, int block_size, int64_t num_blocks, float k_scale,
                        float v_scale, int32_t *err_word, void *cuda_stream);
int paged_decode_plan_fp8(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                          int block_size, int max_blocks_per_seq, int max_context_len,
                          size_t *workspace_bytes_out);
int paged_decode_attention_fp8(void *out, const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                               int64_t num_blocks, float scale, float k_scale, float v_scale,
                               int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                               int max_context_len, void *workspace, size_t workspace_bytes,
                               float *lse_out, int32_t *err_word, void *cuda_stream);

/*
 * paged_decode_attention_prefix_shared with launch flags (PKV_TABLES_READY as
 * for paged_decode_attention_ex, covering group_offsets and
 * group_prefix_lens too).  Under the flag the shared pass reads the groups
 * and lengths before its dependency wait and waits before it reads q or the
 * caches; when the call runs the regular attention, that is
 * paged_decode_attention_ex with the flag.  flags = 0 is
 * paged_decode_attention_prefix_shared; unknown bits give PKV_ERR_INVALID_ARG.
 */
int paged_decode_attention_prefix_shared_ex(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads, int n_kv_heads,
    int head_dim, int block_size, int max_context_len, const int32_t *group_offsets,
    const int32_t *group_prefix_lens, int num_groups, int max_group_size, int max_prefix_len,
    void *workspace, size_t workspace_bytes, float *lse_out, int32_t *err_word,
    void *cuda_stream, uint32_t flags);

/*
 * paged_decode_attention_fp8 with launch flags (PKV_TABLES_READY, as for
 * paged_decode_attention_ex).  flags = 0 is paged_decode_attention_fp8.
 */
int paged_decode_attention_fp8_ex(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs,
                                  int max_blocks_per_seq, int64_t num_blocks, float scale,
                                  float k_scale, float v_scale, int n_q_heads, int n_kv_heads,
                                  int head_dim, int block_size, int max_context_len,
                                  void *workspace, size_t workspace_bytes, float *lse_out,
                                  int32_t *err_word, void *cuda_stream, uint32_t flags);

/*
 * Prefix-aware decode attention over E4M3 caches: paged_decode_attention_
 * prefix_shared with the caches, scales and results of
 * paged_decode_attention_fp8 (same reading of the FP8 format and scales; the
 * KV-cache list of "Roadmap: vLLM-style serving features for TornadoVM
 * batched decode" together with section 2 of "Distributed LLM Inference
 * Serving Platform").  The shared pass reads each shared E4M3 tile once per
 * chunk of members and widens it in the tile math.  The L2 rule counts one
 * byte per value (num_groups * max_prefix_len * n_kv_heads * head_dim * 2
 * bytes); below it, or with no group of two, the call runs
 * paged_decode_attention_fp8.  paged_decode_prefix_shared_plan_fp8 gives the
 * workspace bytes; its counter bytes (PKV_WORKSPACE_COUNTER_BYTES) must be
 * zero before its first use.
 * Groups, arguments, requirements and errors as for the two calls above.
 */
int paged_decode_prefix_shared_plan_fp8(int num_seqs, int n_q_heads, int n_kv_heads,
                                        int head_dim, int block_size, int max_blocks_per_seq,
                                        int max_context_len, int num_groups, int max_group_size,
                                        int max_prefix_len, size_t *workspace_bytes_out);
int paged_decode_attention_prefix_shared_fp8(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, float k_scale, float v_scale,
    int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_context_len,
    const int32_t *group_offsets, const int32_t *group_prefix_lens, int num_groups,
    int max_group_size, int max_prefix_len, void *workspace, size_t workspace_bytes,
    float *lse_out, int32_t *err_word, void *cuda_stream);
/* The same with launch flags (PKV_TABLES_READY, covering the groups too). */
int paged_decode_attention_prefix_shared_fp8_ex(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, float k_scale, float v_scale,
    int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_context_len,
    const int32_t *group_offsets, const int32_t *group_prefix_lens, int num_groups,
    int max_group_size, int max_prefix_len, void *workspace, size_t workspace_bytes,
    float *lse_out, int32_t *err_word, void *cuda_stream, uint32_t flags);

/*
 * Multi-token (causal) paged attention: several new tokens of each sequence
 * attend in one call -- verifying speculative draft tokens, or a chunk of a
 * chunked prefill ("Roadmap: vLLM-style serving features for TornadoVM
 * batched decode", Deferred list: batch-prefill verify, multi-token chunked
 * prefill; "Distributed LLM Inference Serving Platform", section 9.2).
 *  q, out       fp16 [total_q][n_q_heads][head_dim]; lse_out fp32
 *               [total_q][n_q_heads] (nullable)
 *  query_start  device int32 [num_seqs + 1], query_start[0] = 0,
 *               query_start[num_seqs] = total_q: sequence b owns the query
 *               rows [query_start[b], query_start[b+1]), n_b of them
 *  context_lens device int32 [num_seqs]: cached tokens L_b, the n_b new
 *               tokens included (append them first); n_b <= L_b
 * Query token i of sequence b sits at position L_b - n_b + i and attends the
 * tokens [0, L_b - n_b + i] of its block table (causal); n_b = 1 is the
 * decode of paged_decode_attention.  max_q_len: host upper bound of n_b.
 * partition_tokens: 0 = the library's choice, else KV tokens per split-K
 * partition (a multiple of 16 and of block_size).  With 0, when
 * max_q_len * (n_q_heads / n_kv_heads) <= 16 and num_seqs <= 1024, the call
 * runs the balanced split of paged_decode_attention with every segment's
 * query rows -- the (token, head) pairs of its n_b tokens -- in one tile: the
 * workspace then holds arrival counters (PKV_WORKSPACE_COUNTER_BYTES), which
 * must be zero before its first use and which every call leaves zeroed (after
 * a call that flagged PKV_ERRBIT_TIMEOUT or PKV_ERRBIT_WORKSPACE, zero them
 * once more).  Otherwise it runs fixed partitions,
 * whose workspace (0 bytes when one partition covers max_context_len) needs
 * no zero-fill.  paged_decode_multi_plan gives the partition size (0 for the
 * balanced split) and the workspace bytes.
 * Requirements: block_size a multiple of 16, head_dim 64 or 128, n_q/n_kv in
 * {1, 2, 4, 8} (PKV_ERR_UNSUPPORTED otherwise).  A sequence with n_b > L_b,
 * n_b > max_q_len, L_b outside [0, min(max_blocks_per_seq * block_size,
 * max_context_len)] or rows outside [0, total_q) sets PKV_ERRBIT_CONTEXT and
 * its rows (out and lse) are left unwritten.  Other arguments, errors and
 * ownership as for paged_decode_attention.
 */
int paged_decode_multi_plan(int num_seqs, int total_q, int max_q_len, int n_q_heads,
                            int n_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                            int max_context_len, int partition_tokens, int *partition_tokens_out,
                            size_t *workspace_bytes_out);
int paged_decode_attention_multi(void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, const int32_t *query_start,
                                 int num_seqs, int total_q, int max_q_len,
                                 int max_blocks_per_seq, int64_t num_blocks, float scale,
                                 int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                 int max_context_len, int partition_tokens, void *workspace,
                                 size_t workspace_bytes, float *lse_out, int32_t *err_word,
                                 void *cuda_stream);
/*
 * paged_decode_attention_multi with launch flags: PKV_TABLES_READY as for
 * paged_decode_attention_ex, covering query_start too.  It takes effect on
 * the balanced split; fixed partitions ignore it.  flags = 0 is
 * paged_decode_attention_multi; unknown bits give PKV_ERR_INVALID_ARG.
 */
int paged_decode_attention_multi_ex(void *out, const void *q, const void *k_cache,
                                    const void *v_cache, const int32_t *block_tables,
                                    const int32_t *context_lens, const int32_t *query_start,
                                    int num_seqs, int total_q, int max_q_len,
                                    int max_blocks_per_seq, int64_t num_blocks, float scale,
                                    int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                    int max_context_len, int partition_tokens, void *workspace,
                                    size_t workspace_bytes, float *lse_out, int32_t *err_word,
                                    void *cuda_stream, uint32_t flags);

/*
 * Allocation-free variant of paged_decode_attention.  The pages have no
 * counterpart to this call.  It serves callers that cannot allocate device
 * memory and so cannot supply the split-K workspace: an operator running
 * inside a host framework's plugin interface that is handed its input and
 * output tensors but no allocator, or a foreign-language binding without
 * access to a CUDA allocator.
 *
 * Same arguments and results as paged_decode_attention, without workspace
 * and workspace_bytes.  The split-K partial results go to a static device
 * array of PKV_NOALLOC_SCRATCH_BYTES bytes inside the library, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *  - Returns PKV_ERR_WORKSPACE, launching nothing, when the problem's split
 *    needs more than the array holds: more than PKV_NOALLOC_SCRATCH_BYTES
 *    for the balanced split (partition_tokens 0, whose need paged_decode_plan
 *    reports), or more than PKV_NOALLOC_SCRATCH_BYTES -
 *    PKV_WORKSPACE_COUNTER_BYTES for fixed partitions (a larger
 *    partition_tokens lowers their need).
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and caches it; make that
 *    first call before any stream capture on that device.
 *  - The array's first PKV_WORKSPACE_COUNTER_BYTES bytes hold the balanced
 *    split's arrival counters, which must be zero when its kernel starts.
 *    Each balanced call clears them on cuda_stream first (cudaMemsetAsync,
 *    which allocates nothing), so neither a fixed-partition call nor a call
 *    that flagged PKV_ERRBIT_TIMEOUT leaves stale counts for the next one;
 *    fixed-partition plans keep their partial sums after those bytes.  Every other byte is
 *    written before it is read within a call.
 *  - All calls share the one array, and it keeps the last call's contents.
 *    Calls whose kernels overlap in time on the GPU (on different streams,
 *    or from different host threads) race on the array and give wrong
 *    results; serialise them.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
int paged_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs,
                                   int max_blocks_per_seq, int64_t num_blocks, float scale,
                                   int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                   int max_context_len, int partition_tokens, float *lse_out,
                                   int32_t *err_word, void *cuda_stream);

/*
 * Copies bytes from src to dst on cuda_stream with a kernel in which every
 * thread moves one 16-byte piece.  src may be pinned (page-locked, mapped)
 * host memory: a decode step's inputs staged on the host then cross the host
 * link in about one round trip, and the copy is a kernel that the step's own
 * launch follows on the stream.  Both pointers 16-byte aligned, bytes a
 * multiple of 16 (PKV_ERR_INVALID_ARG otherwise); bytes = 0 is a no-op.
 */
int paged_copy_in(void *dst, const void *src, size_t bytes, void *cuda_stream);

/*
 * Zeroes the arrival counters of a workspace on cuda_stream: the first
 * min(workspace_bytes, PKV_WORKSPACE_COUNTER_BYTES) bytes (one
 * cudaMemsetAsync; no allocation, no host wait, so it may be captured in a
 * CUDA graph).  Call it once on a new workspace and after a call that
 * flagged PKV_ERRBIT_TIMEOUT or PKV_ERRBIT_WORKSPACE.  workspace may be NULL
 * only when workspace_bytes is 0 (a no-op).  Returns PKV_ERR_INVALID_ARG for
 * a NULL workspace with bytes, PKV_ERR_CUDA when the memset fails.
 */
int paged_decode_workspace_clear(void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * One decode step over E4M3 caches: paged_kv_append_fp8 of num_tokens new
 * tokens, then paged_decode_attention_fp8, on cuda_stream, with the same
 * arguments, results and errors as those two calls (the attention's
 * arguments are checked first, so a rejected call writes nothing).  The
 * attention's prologue runs while the append drains.  paged_decode_step_fp8_ex
 * accepts the flags of paged_decode_step_ex; the step keeps its two kernels
 * under PKV_APPEND_NEWEST (folded into the E4M3 attention, which is bound by
 * instruction issue, the append slowed it).  Other flag bits are rejected
 * with PKV_ERR_INVALID_ARG.
 */
int paged_decode_step_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                          int num_tokens, void *out, const void *q, void *k_cache, void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int64_t num_blocks, float scale,
                          float k_scale, float v_scale, int n_q_heads, int n_kv_heads,
                          int head_dim, int block_size, int max_context_len, void *workspace,
                          size_t workspace_bytes, float *lse_out, int32_t *err_word,
                          void *cuda_stream);
int paged_decode_step_fp8_ex(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int num_tokens, void *out, const void *q, void *k_cache,
                             void *v_cache, const int32_t *block_tables,
                             const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                             int64_t num_blocks, float scale, float k_scale, float v_scale,
                             int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                             int max_context_len, void *workspace, size_t workspace_bytes,
                             float *lse_out, int32_t *err_word, void *cuda_stream,
                             uint32_t flags);

/*
 * Reads the device error word: waits for cuda_stream, copies *err_word to the
 * host, stores it in *bits_out (host, may be NULL) and returns PKV_OK when it
 * is 0, PKV_ERR_INDEX otherwise.  Does not clear the word.
 */
int paged_kv_get_error(const int32_t *err_word, void *cuda_stream, int32_t *bits_out);

/* Static English text for a pkv_status value. */
const char *paged_kv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
