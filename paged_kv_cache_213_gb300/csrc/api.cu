// api.cu -- the extern "C" entry points declared in include/pagedkv.h:
// argument checks on the host, split planning, kernel launches on the
// caller's stream.  Allocates nothing.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "pagedkv.h"
#include "pagedkv_blocks.h"
#include "pkv_internal.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool block_size_ok(int bs) {
    return bs == 1 || bs == 2 || bs == 4 || bs == 8 || bs == 16 || bs == 32 || bs == 64 ||
           bs == 128 || bs == 256;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count(int *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) {
            *out = cached;
            return PKV_OK;
        }
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return PKV_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return PKV_OK;
}

// Tokens per partition when the caller leaves the choice to the library:
// the largest power of two in [128, 2048] (and >= the block size) that still
// gives an upper-bound grid of at least 12 CTAs per SM, and no larger than
// the longest context needs.
int auto_partition(int num_seqs, int n_kv_heads, int max_len, int block_size, int sms) {
    const int step = block_size > 16 ? block_size : 16;
    int P = 2048;
    while (P > 128 && P / 2 >= step) {
        const long long parts = (max_len + P - 1) / P;
        if (static_cast<long long>(num_seqs) * n_kv_heads * parts >= 12LL * sms) break;
        P /= 2;
    }
    const int cover = (max_len + step - 1) / step * step;  // one partition suffices
    if (cover > 0 && cover < P) P = cover;
    return P < step ? step : P;
}

struct Plan {
    int max_len;
    int partition;   // 0: the balanced kernel (no fixed partitions)
    int max_parts;
    size_t ws_bytes;
    bool balanced;
    pkv::BalancedPlan bal;
};

// allow_pipeline: the balanced split may run on the producer/consumer kernel
// (fp16 caches, no prefix groups); otherwise on per-warp ranges.
int make_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
              int max_blocks_per_seq, int max_context_len, int partition_tokens, Plan *plan,
              bool allow_pipeline = true) {
    if (num_seqs < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 ||
        max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (!block_size_ok(block_size)) return PKV_ERR_UNSUPPORTED;
    if (!pkv::decode_supported(head_dim, n_q_heads / n_kv_heads)) return PKV_ERR_UNSUPPORTED;
    const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
    if (cap > (1LL << 30)) return PKV_ERR_INVALID_ARG;
    long long max_len = max_context_len <= 0 ? cap : max_context_len;
    if (max_len > cap) max_len = cap;
    int P = partition_tokens;
    const int group = n_q_heads / n_kv_heads;
    const int mode = pkv::kernel_override();
    if (P == 0 && (mode == 0 || mode >= 3) &&
        pkv::balanced_supported(num_seqs, head_dim, group, block_size, 0)) {
        // work split evenly over CTAs or warps; the grid and workspace follow the device.
        // Batches of more (sequence, KV head) segments than twice the SMs
        // (many short ones, e.g. continuous batching) run on the
        // producer/consumer kernel, whose CTAs read every head of a block at
        // once; fewer, longer segments run on per-warp ranges (measured on
        // GB300: Mistral-shaped mix 50.5 -> 40.5 us; LLaMA-3-8B-shaped layer
        // 35.0 against 36.8 us, 32k contexts 165.9 against 175.0 us).
        const int ml = static_cast<int>(max_len);
        int sms = 0;
        if (sm_count(&sms) != PKV_OK) return PKV_ERR_CUDA;
        const bool many = static_cast<long long>(num_seqs) * n_kv_heads > 2LL * sms;
        bool done = false;
        if (allow_pipeline && ((mode == 0 && many) || mode == 4) &&
            pkv::pipeline_supported(num_seqs, n_kv_heads, head_dim, group, block_size, 0))
            done = pkv::pipeline_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, ml, &plan->bal);
        if (!done && !pkv::balanced_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, ml, &plan->bal))
            return PKV_ERR_CUDA;
        plan->balanced = true;
        plan->max_len = static_cast<int>(max_len);
        plan->partition = 0;
        plan->max_parts = 1;
        plan->ws_bytes = plan->bal.ws_bytes;
        return PKV_OK;
    }
    plan->balanced = false;
    if (P == 0) {
        int sms = 0;
        const int rc = sm_count(&sms);
        if (rc != PKV_OK) return rc;
        P = auto_partition(num_seqs, n_kv_heads, static_cast<int>(max_len), block_size, sms);
    } else {
        if (P < 16 || P % 16 != 0 || P % block_size != 0 || P / block_size > 2048)
            return PKV_ERR_INVALID_ARG;
    }
    const long long parts = (max_len + P - 1) / P;
    if (parts > 65535) return PKV_ERR_UNSUPPORTED;
    plan->max_len = static_cast<int>(max_len);
    plan->partition = P;
    plan->max_parts = parts < 1 ? 1 : static_cast<int>(parts);
    plan->ws_bytes = plan->max_parts > 1
                         ? pkv::workspace_layout(num_seqs, n_q_heads, head_dim, plan->max_parts).total
                         : 0;
    return PKV_OK;
}

}  // namespace

extern "C" {

int paged_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                    void *k_cache, void *v_cache, int num_tokens, int n_kv_heads, int head_dim,
                    int block_size, int64_t num_blocks, int32_t *err_word, void *cuda_stream) {
    if (num_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 ||
        num_blocks <= 0 || block_size <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8) || (err_word && !aligned(err_word, 4)))
        return PKV_ERR_INVALID_ARG;
    pkv::AppendArgs a{k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens,
                      n_kv_heads, head_dim, block_size, num_blocks, err_word};
    const cudaError_t e = pkv::launch_append(a, static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int paged_decode_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                      int max_blocks_per_seq, int max_context_len, int partition_tokens,
                      int *partition_tokens_out, size_t *workspace_bytes_out) {
    Plan plan{};
    const int rc = make_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, max_context_len, partition_tokens, &plan);
    if (rc != PKV_OK) return rc;
    if (partition_tokens_out) *partition_tokens_out = plan.partition;
    if (workspace_bytes_out) *workspace_bytes_out = plan.ws_bytes;
    return PKV_OK;
}

}  // extern "C"

namespace {

// The step appends inside the attention kernel (one launch): the caller's
// PKV_APPEND_NEWEST, one token per sequence, and per-warp balanced ranges.
bool step_fuses(const Plan &plan, int num_seqs, int num_tokens, uint32_t flags) {
    return (flags & PKV_APPEND_NEWEST) && num_tokens == num_seqs && num_seqs > 0 &&
           plan.balanced && plan.bal.kind == 0;
}

// The decode step's new tokens, when the attention kernel does their append
// (paged_decode_step_ex under PKV_APPEND_NEWEST).
struct FusedAppend {
    const void *k_new;
    const void *v_new;
    const int64_t *slot_mapping;
};

// paged_decode_attention; defer = 2 when this library's append was launched
// just before on the same stream (the prologue may then run under it).  With
// fa, the plan must be the balanced split on per-warp ranges.
int decode_attention_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads,
                          int n_kv_heads, int head_dim, int block_size, int max_context_len,
                          int partition_tokens, void *workspace, size_t workspace_bytes,
                          float *lse_out, int32_t *err_word, void *cuda_stream, int defer,
                          const FusedAppend *fa = nullptr);

}  // namespace

extern "C" {

int paged_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens,
                           int num_seqs, int max_blocks_per_seq, int64_t num_blocks, float scale,
                           int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                           int max_context_len, int partition_tokens, void *workspace,
                           size_t workspace_bytes, float *lse_out, int32_t *err_word,
                           void *cuda_stream) {
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                 max_blocks_per_seq, num_blocks, scale, n_q_heads, n_kv_heads,
                                 head_dim, block_size, max_context_len, partition_tokens,
                                 workspace, workspace_bytes, lse_out, err_word, cuda_stream, 0);
}

int paged_decode_attention_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *context_lens,
                              int num_seqs, int max_blocks_per_seq, int64_t num_blocks,
                              float scale, int n_q_heads, int n_kv_heads, int head_dim,
                              int block_size, int max_context_len, int partition_tokens,
                              void *workspace, size_t workspace_bytes, float *lse_out,
                              int32_t *err_word, void *cuda_stream, uint32_t flags) {
    if (flags & ~PKV_TABLES_READY) return PKV_ERR_INVALID_ARG;
    // with the tables ready, the kernel before writes at most q, the caches
    // and the workspace: the same contract as after this library's append
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                 max_blocks_per_seq, num_blocks, scale, n_q_heads, n_kv_heads,
                                 head_dim, block_size, max_context_len, partition_tokens,
                                 workspace, workspace_bytes, lse_out, err_word, cuda_stream,
                                 (flags & PKV_TABLES_READY) ? 2 : 0);
}

int paged_decode_step(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                      int num_tokens, void *out, const void *q, void *k_cache, void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                      int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads,
                      int n_kv_heads, int head_dim, int block_size, int max_context_len,
                      int partition_tokens, void *workspace, size_t workspace_bytes,
                      float *lse_out, int32_t *err_word, void *cuda_stream) {
    return paged_decode_step_ex(k_new, v_new, slot_mapping, num_tokens, out, q, k_cache, v_cache,
                                block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                num_blocks, scale, n_q_heads, n_kv_heads, head_dim, block_size,
                                max_context_len, partition_tokens, workspace, workspace_bytes,
                                lse_out, err_word, cuda_stream, 0);
}

int paged_decode_step_launches(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                               int block_size, int max_blocks_per_seq, int max_context_len,
                               int partition_tokens, int num_tokens, uint32_t flags,
                               int *launches_out) {
    if ((flags & ~(PKV_TABLES_READY | PKV_APPEND_NEWEST)) || num_tokens < 0)
        return PKV_ERR_INVALID_ARG;
    Plan plan{};
    const int rc = make_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, max_context_len, partition_tokens, &plan);
    if (rc != PKV_OK) return rc;
    const int attention = num_seqs == 0 ? 0 : (!plan.balanced && plan.ws_bytes > 0 ? 2 : 1);
    const int append = num_tokens > 0 && !step_fuses(plan, num_seqs, num_tokens, flags) ? 1 : 0;
    if (launches_out) *launches_out = attention + append;
    return PKV_OK;
}

int paged_decode_step_ex(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                         int num_tokens, void *out, const void *q, void *k_cache, void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                         int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads,
                         int n_kv_heads, int head_dim, int block_size, int max_context_len,
                         int partition_tokens, void *workspace, size_t workspace_bytes,
                         float *lse_out, int32_t *err_word, void *cuda_stream, uint32_t flags) {
    if (flags & ~(PKV_TABLES_READY | PKV_APPEND_NEWEST)) return PKV_ERR_INVALID_ARG;
    // check the attention's arguments first so that a rejected call changes nothing
    Plan plan{};
    int rc = make_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                       max_context_len, partition_tokens, &plan);
    if (rc != PKV_OK) return rc;
    if (num_seqs > 0 && plan.ws_bytes > 0 &&
        (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256)))
        return PKV_ERR_WORKSPACE;
    if (step_fuses(plan, num_seqs, num_tokens, flags)) {
        // one kernel: the attention appends each sequence's newest token itself
        if (!k_new || !v_new || !slot_mapping || !aligned(k_new, 16) || !aligned(v_new, 16) ||
            !aligned(slot_mapping, 8))
            return PKV_ERR_INVALID_ARG;
        const FusedAppend fa{k_new, v_new, slot_mapping};
        return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens,
                                     num_seqs, max_blocks_per_seq, num_blocks, scale, n_q_heads,
                                     n_kv_heads, head_dim, block_size, max_context_len,
                                     partition_tokens, workspace, workspace_bytes, lse_out,
                                     err_word, cuda_stream,
                                     (flags & PKV_TABLES_READY) ? 2 : 0, &fa);
    }
    rc = paged_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens, n_kv_heads,
                         head_dim, block_size, num_blocks, err_word, cuda_stream);
    if (rc != PKV_OK) return rc;
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                 max_blocks_per_seq, num_blocks, scale, n_q_heads, n_kv_heads,
                                 head_dim, block_size, max_context_len, partition_tokens,
                                 workspace, workspace_bytes, lse_out, err_word, cuda_stream,
                                 num_tokens > 0 ? 2 : 0);
}

}  // extern "C"

namespace {

int decode_attention_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads,
                          int n_kv_heads, int head_dim, int block_size, int max_context_len,
                          int partition_tokens, void *workspace, size_t workspace_bytes,
                          float *lse_out, int32_t *err_word, void *cuda_stream, int defer,
                          const FusedAppend *fa) {
    if (num_blocks <= 0 || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    Plan plan{};
    int rc = make_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                       max_context_len, partition_tokens, &plan);
    if (rc != PKV_OK) return rc;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
        (lse_out && !aligned(lse_out, 4)) || (err_word && !aligned(err_word, 4)))
        return PKV_ERR_INVALID_ARG;
    if (n_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    pkv::DecodeArgs a{};
    if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes ||
                              !aligned(workspace, 256)))
        return PKV_ERR_WORKSPACE;
    if (plan.balanced) {
        a.ws_acc = static_cast<float *>(workspace);  // base of the balanced layout
    } else if (plan.ws_bytes > 0) {
        const pkv::WorkspaceLayout w =
            pkv::workspace_layout(num_seqs, n_q_heads, head_dim, plan.max_parts);
        char *base = static_cast<char *>(workspace);
        a.ws_acc = reinterpret_cast<float *>(base + w.acc_offset);
        a.ws_m = reinterpret_cast<float *>(base + w.m_offset);
        a.ws_l = reinterpret_cast<float *>(base + w.l_offset);
    }
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.lse_out = lse_out;
    a.err = err_word;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.max_context_len = plan.max_len;
    a.partition_tokens = plan.partition;
    a.max_parts = plan.max_parts;
    a.defer_dep_wait = plan.balanced ? defer : 0;
    a.first_wait_polls = pkv::test_wait_polls();
    if (fa) {  // the caller checked the plan: balanced, per-warp ranges
        a.append_k = fa->k_new;
        a.append_v = fa->v_new;
        a.append_slots = fa->slot_mapping;
        a.fuse_append = 1;
    }
    if (plan.balanced &&
        static_cast<long long>(num_blocks) * n_kv_heads * block_size >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    const cudaError_t e = !plan.balanced         ? pkv::launch_decode(a, stream)
                          : plan.bal.kind == 1   ? pkv::launch_decode_pipeline(a, plan.bal, stream)
                                                 : pkv::launch_decode_balanced(a, plan.bal, stream);
    if (e == cudaErrorInvalidValue) return PKV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// FP8 (E4M3) KV caches
// ---------------------------------------------------------------------------

int paged_kv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                        void *k_cache, void *v_cache, int num_tokens, int n_kv_heads,
                        int head_dim, int block_size, int64_t num_blocks, float k_scale,
                        float v_scale, int32_t *err_word, void *cuda_stream) {
    if (num_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim % 16 != 0 ||
        num_blocks <= 0 || block_size <= 0)
        return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) ||
        !(v_scale > 0.f))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8) || (err_word && !aligned(err_word, 4)))
        return PKV_ERR_INVALID_ARG;
    pkv::AppendArgs a{k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens,
                      n_kv_heads, head_dim, block_size, num_blocks, err_word};
    const cudaError_t e =
        pkv::launch_append_f8(a, k_scale, v_scale, static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"

namespace {

// The balanced plan for E4M3 caches (its own occupancy, hence grid and workspace).
int make_plan_fp8(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                  int max_blocks_per_seq, int max_context_len, Plan *plan) {
    int rc = make_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                       max_context_len, 0, plan, false);
    if (rc != PKV_OK) return rc;
    if (!plan->balanced) return PKV_ERR_UNSUPPORTED;  // E4M3 runs on the balanced kernel only
    if (!pkv::balanced_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, plan->max_len, &plan->bal,
                            true))
        return PKV_ERR_CUDA;
    plan->ws_bytes = plan->bal.ws_bytes;
    return PKV_OK;
}

}  // namespace

namespace {

// paged_decode_attention_fp8; defer as decode_attention_impl.
int fp8_attention_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                       int max_blocks_per_seq, int64_t num_blocks, float scale, float k_scale,
                       float v_scale, int n_q_heads, int n_kv_heads, int head_dim,
                       int block_size, int max_context_len, void *workspace,
                       size_t workspace_bytes, float *lse_out, int32_t *err_word,
                       void *cuda_stream, int defer) {
    if (num_blocks <= 0 || !std::isfinite(scale) || !std::isfinite(k_scale) ||
        !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PKV_ERR_INVALID_ARG;
    Plan plan{};
    int rc = make_plan_fp8(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, max_context_len, &plan);
    if (rc != PKV_OK) return rc;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
        (lse_out && !aligned(lse_out, 4)) || (err_word && !aligned(err_word, 4)))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    if (static_cast<long long>(num_blocks) * n_kv_heads * block_size >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;  // row indices are 32-bit
    pkv::DecodeArgs a{};
    a.ws_acc = static_cast<float *>(workspace);
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.lse_out = lse_out;
    a.err = err_word;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    // the logits of E4M3 keys: q . (code * k_scale) * scale
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * k_scale * 1.4426950408889634);
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.max_context_len = plan.max_len;
    a.partition_tokens = 0;
    a.max_parts = 1;
    a.kv_fp8 = 1;
    a.v_scale = v_scale;
    a.defer_dep_wait = defer;
    a.first_wait_polls = pkv::test_wait_polls();
    const cudaError_t e =
        pkv::launch_decode_balanced(a, plan.bal, static_cast<cudaStream_t>(cuda_stream));
    if (e == cudaErrorInvalidValue) return PKV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

int paged_decode_plan_fp8(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                          int block_size, int max_blocks_per_seq, int max_context_len,
                          size_t *workspace_bytes_out) {
    Plan plan{};
    const int rc = make_plan_fp8(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                 max_blocks_per_seq, max_context_len, &plan);
    if (rc == PKV_OK && workspace_bytes_out) *workspace_bytes_out = plan.ws_bytes;
    return rc;
}

int paged_decode_attention_fp8_ex(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs,
                                  int max_blocks_per_seq, int64_t num_blocks, float scale,
                                  float k_scale, float v_scale, int n_q_heads, int n_kv_heads,
                                  int head_dim, int block_size, int max_context_len,
                                  void *workspace, size_t workspace_bytes, float *lse_out,
                                  int32_t *err_word, void *cuda_stream, uint32_t flags) {
    if (flags & ~PKV_TABLES_READY) return PKV_ERR_INVALID_ARG;
    return fp8_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              max_blocks_per_seq, num_blocks, scale, k_scale, v_scale, n_q_heads,
                              n_kv_heads, head_dim, block_size, max_context_len, workspace,
                              workspace_bytes, lse_out, err_word, cuda_stream,
                              (flags & PKV_TABLES_READY) ? 2 : 0);
}

int paged_decode_step_fp8_ex(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int num_tokens, void *out, const void *q, void *k_cache,
                             void *v_cache, const int32_t *block_tables,
                             const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                             int64_t num_blocks, float scale, float k_scale, float v_scale,
                             int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                             int max_context_len, void *workspace, size_t workspace_bytes,
                             float *lse_out, int32_t *err_word, void *cuda_stream,
                             uint32_t flags) {
    if (flags & ~(PKV_TABLES_READY | PKV_APPEND_NEWEST)) return PKV_ERR_INVALID_ARG;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    // check the attention's arguments first so that a rejected call changes nothing
    if (num_blocks <= 0 || !std::isfinite(scale) || !std::isfinite(k_scale) ||
        !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PKV_ERR_INVALID_ARG;
    Plan plan{};
    int rc = make_plan_fp8(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, max_context_len, &plan);
    if (rc != PKV_OK) return rc;
    if (num_seqs > 0 && (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256)))
        return PKV_ERR_WORKSPACE;
    // The append kernel, then the attention with its prologue under it.  The
    // E4M3 attention is bound by instruction issue: an append folded into it
    // (as the fp16 step does under PKV_APPEND_NEWEST) slowed every E4M3 call,
    // so the flag is accepted and the step keeps its two kernels.
    rc = paged_kv_append_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens,
                             n_kv_heads, head_dim, block_size, num_blocks, k_scale, v_scale,
                             err_word, cuda_stream);
    if (rc != PKV_OK) return rc;
    return fp8_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              max_blocks_per_seq, num_blocks, scale, k_scale, v_scale, n_q_heads,
                              n_kv_heads, head_dim, block_size, max_context_len, workspace,
                              workspace_bytes, lse_out, err_word, cuda_stream,
                              num_tokens > 0 ? 2 : 0);
}

int paged_decode_step_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                          int num_tokens, void *out, const void *q, void *k_cache, void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int64_t num_blocks, float scale,
                          float k_scale, float v_scale, int n_q_heads, int n_kv_heads,
                          int head_dim, int block_size, int max_context_len, void *workspace,
                          size_t workspace_bytes, float *lse_out, int32_t *err_word,
                          void *cuda_stream) {
    return paged_decode_step_fp8_ex(k_new, v_new, slot_mapping, num_tokens, out, q, k_cache,
                                    v_cache, block_tables, context_lens, num_seqs,
                                    max_blocks_per_seq, num_blocks, scale, k_scale, v_scale,
                                    n_q_heads, n_kv_heads, head_dim, block_size, max_context_len,
                                    workspace, workspace_bytes, lse_out, err_word, cuda_stream, 0);
}

int paged_decode_attention_fp8(void *out, const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                               int64_t num_blocks, float scale, float k_scale, float v_scale,
                               int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                               int max_context_len, void *workspace, size_t workspace_bytes,
                               float *lse_out, int32_t *err_word, void *cuda_stream) {
    return paged_decode_attention_fp8_ex(out, q, k_cache, v_cache, block_tables, context_lens,
                                         num_seqs, max_blocks_per_seq, num_blocks, scale, k_scale,
                                         v_scale, n_q_heads, n_kv_heads, head_dim, block_size,
                                         max_context_len, workspace, workspace_bytes, lse_out,
                                         err_word, cuda_stream, 0);
}

}  // extern "C"

namespace {

struct SharedPlan {
    Plan base;  // the balanced split of the private suffixes
    int chunks, parts, part_tiles, warps;
    size_t sh_acc, sh_m, sh_l, total;
    // the shared blocks fit well inside L2: the call runs the regular
    // attention (plan `regular`), whose reads of shared blocks hit L2 anyway
    bool regular_path;
    Plan regular;
};

// L2 bytes of the current device (0 when the query fails).
long long l2_bytes() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return 0;
    return n;
}

// fp8: E4M3 caches (one byte per value; both passes widen in the tile math).
int make_shared_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                     int max_blocks_per_seq, int max_context_len, int num_groups,
                     int max_group_size, int max_prefix_len, SharedPlan *sp, bool fp8 = false) {
    if (num_groups < 0 || max_group_size < 0 || max_prefix_len < 0) return PKV_ERR_INVALID_ARG;
    if (pkv::kernel_override() == 1 || pkv::kernel_override() == 2) return PKV_ERR_UNSUPPORTED;
    // Shared prefixes that fit in a quarter of L2 are read from DRAM about
    // once by the regular attention too (its readers of a shared block hit
    // L2), and the regular path has no second pass to pay for: on the
    // Mistral-shaped mix (one 512-token prefix, 2 MB) 40.5 us against 62.5 us
    // through the two passes.  The 70B-shaped batch's prefixes (16 x 3968
    // tokens, 260 MB) stay on the prefix-aware path.
    const long long shared_bytes = static_cast<long long>(num_groups) * max_prefix_len *
                                   n_kv_heads * head_dim * 2 * (fp8 ? 1 : 2);
    const long long l2 = l2_bytes();
    sp->regular_path = l2 > 0 && (max_group_size < 2 || shared_bytes <= l2 / 4);
    // PKV_PREFIX_PASS=shared / =regular fixes the choice (read at every call)
    if (const char *e = std::getenv("PKV_PREFIX_PASS")) {
        if (std::strcmp(e, "shared") == 0) sp->regular_path = false;
        if (std::strcmp(e, "regular") == 0) sp->regular_path = true;
    }
    if (sp->regular_path) {
        int rc = fp8 ? make_plan_fp8(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                     max_blocks_per_seq, max_context_len, &sp->regular)
                     : make_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                 max_blocks_per_seq, max_context_len, 0, &sp->regular);
        if (rc != PKV_OK) return rc;
        sp->total = sp->regular.ws_bytes;
        return PKV_OK;
    }
    // the suffix pass runs on the per-warp kernel, which folds in the shared partials
    int rc = fp8 ? make_plan_fp8(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                 max_blocks_per_seq, max_context_len, &sp->base)
                 : make_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, max_context_len, 0, &sp->base, false);
    if (rc != PKV_OK) return rc;
    if (!sp->base.balanced) return PKV_ERR_UNSUPPORTED;
    const int g = n_q_heads / n_kv_heads;
    const int mpw = pkv::shared_members_per_warp(g);
    const int max_tiles =
        (max_prefix_len < sp->base.max_len ? max_prefix_len : sp->base.max_len) / 16;
    // warps per CTA: those the largest group needs, at most shared_max_warps()
    const int need_w = max_group_size > 0 ? (max_group_size + mpw - 1) / mpw : 1;
    sp->warps = need_w < pkv::shared_max_warps() ? need_w : pkv::shared_max_warps();
    const int mpc = sp->warps * mpw;
    sp->chunks = max_group_size > 0 ? (max_group_size + mpc - 1) / mpc : 1;
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != PKV_OK) return rc;
    const int per_sm = pkv::shared_ctas_per_sm(head_dim, g, sp->warps, fp8);
    if (per_sm <= 0) return PKV_ERR_CUDA;
    // one wave of CTAs over the (group chunk, KV head) pairs, at least 4 tiles each
    const long long pairs =
        static_cast<long long>(num_groups > 0 ? num_groups : 1) * sp->chunks * n_kv_heads;
#ifndef PKV_SHARED_WAVES
#define PKV_SHARED_WAVES 1
#endif
    long long parts = (static_cast<long long>(PKV_SHARED_WAVES) * per_sm * sms) / pairs;
    const long long max_parts = max_tiles > 4 ? max_tiles / 4 : 1;
    if (parts > max_parts) parts = max_parts;
    if (parts < 1) parts = 1;
    if (parts > 65535) parts = 65535;
    sp->part_tiles = max_tiles > 0 ? static_cast<int>((max_tiles + parts - 1) / parts) : 1;
    sp->parts = max_tiles > 0 ? (max_tiles + sp->part_tiles - 1) / sp->part_tiles : 1;
    if (static_cast<long long>(num_groups) * sp->chunks > 2147483647LL) return PKV_ERR_UNSUPPORTED;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rows = static_cast<size_t>(num_seqs) * n_q_heads * sp->parts;
    sp->sh_acc = up(sp->base.ws_bytes);
    sp->sh_m = sp->sh_acc + up(rows * head_dim * 4);
    sp->sh_l = sp->sh_m + up(rows * 4);
    sp->total = sp->sh_l + up(rows * 4);
    return PKV_OK;
}

}  // namespace

extern "C" {

int paged_decode_prefix_shared_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                                    int block_size, int max_blocks_per_seq, int max_context_len,
                                    int num_groups, int max_group_size, int max_prefix_len,
                                    size_t *workspace_bytes_out) {
    SharedPlan sp{};
    const int rc = make_shared_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                    max_blocks_per_seq, max_context_len, num_groups,
                                    max_group_size, max_prefix_len, &sp);
    if (rc == PKV_OK && workspace_bytes_out) *workspace_bytes_out = sp.total;
    return rc;
}

int paged_decode_prefix_shared_plan_fp8(int num_seqs, int n_q_heads, int n_kv_heads,
                                        int head_dim, int block_size, int max_blocks_per_seq,
                                        int max_context_len, int num_groups, int max_group_size,
                                        int max_prefix_len, size_t *workspace_bytes_out) {
    SharedPlan sp{};
    const int rc = make_shared_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                    max_blocks_per_seq, max_context_len, num_groups,
                                    max_group_size, max_prefix_len, &sp, true);
    if (rc == PKV_OK && workspace_bytes_out) *workspace_bytes_out = sp.total;
    return rc;
}

}  // extern "C"

namespace {

// paged_decode_attention_prefix_shared(_fp8): fp8 selects E4M3 caches with
// scales k_scale, v_scale (1, 1 for fp16).
int prefix_shared_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                       int max_blocks_per_seq, int64_t num_blocks, float scale, float k_scale,
                       float v_scale, bool fp8, int n_q_heads, int n_kv_heads, int head_dim,
                       int block_size, int max_context_len, const int32_t *group_offsets,
                       const int32_t *group_prefix_lens, int num_groups, int max_group_size,
                       int max_prefix_len, void *workspace, size_t workspace_bytes,
                       float *lse_out, int32_t *err_word, void *cuda_stream,
                       uint32_t flags = 0) {
    if (flags & ~PKV_TABLES_READY) return PKV_ERR_INVALID_ARG;
    const bool ready = (flags & PKV_TABLES_READY) != 0;
    if (num_blocks <= 0 || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (fp8 && (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) ||
                !(v_scale > 0.f)))
        return PKV_ERR_INVALID_ARG;
    if (num_groups > 0 && (!group_offsets || !group_prefix_lens || !aligned(group_offsets, 4) ||
                           !aligned(group_prefix_lens, 4)))
        return PKV_ERR_INVALID_ARG;
    SharedPlan sp{};
    int rc = make_shared_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                              max_blocks_per_seq, max_context_len, num_groups, max_group_size,
                              max_prefix_len, &sp, fp8);
    if (rc != PKV_OK) return rc;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
        (lse_out && !aligned(lse_out, 4)) || (err_word && !aligned(err_word, 4)))
        return PKV_ERR_INVALID_ARG;
    if (sp.regular_path)
        return fp8 ? paged_decode_attention_fp8_ex(out, q, k_cache, v_cache, block_tables,
                                                   context_lens, num_seqs, max_blocks_per_seq,
                                                   num_blocks, scale, k_scale, v_scale, n_q_heads,
                                                   n_kv_heads, head_dim, block_size,
                                                   max_context_len, workspace, workspace_bytes,
                                                   lse_out, err_word, cuda_stream, flags)
                   : decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens,
                                           num_seqs, max_blocks_per_seq, num_blocks, scale,
                                           n_q_heads, n_kv_heads, head_dim, block_size,
                                           max_context_len, 0, workspace, workspace_bytes,
                                           lse_out, err_word, cuda_stream, ready ? 2 : 0);
    if (!workspace || workspace_bytes < sp.total || !aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    if (static_cast<long long>(num_blocks) * n_kv_heads * block_size >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;
    char *base = static_cast<char *>(workspace);
    pkv::DecodeArgs a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.ws_acc = static_cast<float *>(workspace);
    a.lse_out = lse_out;
    a.err = err_word;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    // E4M3 keys: q . (code * k_scale) * scale; outputs times v_scale
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * (fp8 ? k_scale : 1.f) *
                                      1.4426950408889634);
    a.kv_fp8 = fp8 ? 1 : 0;
    a.v_scale = fp8 ? v_scale : 1.f;
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.max_context_len = sp.base.max_len;
    a.partition_tokens = 0;
    a.max_parts = 1;
    a.group_offsets = group_offsets;
    a.group_prefix = group_prefix_lens;
    a.num_groups = num_groups;
    a.sh_chunks = sp.chunks;
    a.sh_parts = sp.parts;
    a.sh_part_tiles = sp.part_tiles;
    a.sh_warps = sp.warps;
    a.sh_acc = reinterpret_cast<float *>(base + sp.sh_acc);
    a.sh_m = reinterpret_cast<float *>(base + sp.sh_m);
    a.sh_l = reinterpret_cast<float *>(base + sp.sh_l);
    // the suffix pass: after the shared pass (see its wait), else on its own
    a.defer_dep_wait = num_groups > 0 ? 1 : (ready ? 2 : 0);
    a.sh_tables_ready = ready ? 1 : 0;
    a.first_wait_polls = pkv::test_wait_polls();
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e = cudaSuccess;
    if (num_groups > 0) e = pkv::launch_decode_shared(a, stream);
    if (e == cudaSuccess) e = pkv::launch_decode_balanced(a, sp.base.bal, stream);
    if (e == cudaErrorInvalidValue) return PKV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

int paged_decode_attention_prefix_shared(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads, int n_kv_heads,
    int head_dim, int block_size, int max_context_len, const int32_t *group_offsets,
    const int32_t *group_prefix_lens, int num_groups, int max_group_size, int max_prefix_len,
    void *workspace, size_t workspace_bytes, float *lse_out, int32_t *err_word,
    void *cuda_stream) {
    return prefix_shared_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              max_blocks_per_seq, num_blocks, scale, 1.f, 1.f, false, n_q_heads,
                              n_kv_heads, head_dim, block_size, max_context_len, group_offsets,
                              group_prefix_lens, num_groups, max_group_size, max_prefix_len,
                              workspace, workspace_bytes, lse_out, err_word, cuda_stream);
}

int paged_decode_attention_prefix_shared_ex(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads, int n_kv_heads,
    int head_dim, int block_size, int max_context_len, const int32_t *group_offsets,
    const int32_t *group_prefix_lens, int num_groups, int max_group_size, int max_prefix_len,
    void *workspace, size_t workspace_bytes, float *lse_out, int32_t *err_word,
    void *cuda_stream, uint32_t flags) {
    return prefix_shared_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              max_blocks_per_seq, num_blocks, scale, 1.f, 1.f, false, n_q_heads,
                              n_kv_heads, head_dim, block_size, max_context_len, group_offsets,
                              group_prefix_lens, num_groups, max_group_size, max_prefix_len,
                              workspace, workspace_bytes, lse_out, err_word, cuda_stream, flags);
}

int paged_decode_attention_prefix_shared_fp8(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, float k_scale, float v_scale,
    int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_context_len,
    const int32_t *group_offsets, const int32_t *group_prefix_lens, int num_groups,
    int max_group_size, int max_prefix_len, void *workspace, size_t workspace_bytes,
    float *lse_out, int32_t *err_word, void *cuda_stream) {
    return prefix_shared_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              max_blocks_per_seq, num_blocks, scale, k_scale, v_scale, true,
                              n_q_heads, n_kv_heads, head_dim, block_size, max_context_len,
                              group_offsets, group_prefix_lens, num_groups, max_group_size,
                              max_prefix_len, workspace, workspace_bytes, lse_out, err_word,
                              cuda_stream);
}

int paged_decode_attention_prefix_shared_fp8_ex(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, float k_scale, float v_scale,
    int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_context_len,
    const int32_t *group_offsets, const int32_t *group_prefix_lens, int num_groups,
    int max_group_size, int max_prefix_len, void *workspace, size_t workspace_bytes,
    float *lse_out, int32_t *err_word, void *cuda_stream, uint32_t flags) {
    return prefix_shared_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              max_blocks_per_seq, num_blocks, scale, k_scale, v_scale, true,
                              n_q_heads, n_kv_heads, head_dim, block_size, max_context_len,
                              group_offsets, group_prefix_lens, num_groups, max_group_size,
                              max_prefix_len, workspace, workspace_bytes, lse_out, err_word,
                              cuda_stream, flags);
}

}  // extern "C"

namespace {

struct MultiPlan {
    int max_len, partition, max_parts, row_blocks;
    size_t ws_bytes;
    bool balanced;        // the balanced split (partition 0)
    pkv::BalancedPlan bal;
};

int make_multi_plan(int num_seqs, int total_q, int max_q_len, int n_q_heads, int n_kv_heads,
                    int head_dim, int block_size, int max_blocks_per_seq, int max_context_len,
                    int partition_tokens, MultiPlan *mp) {
    if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || n_q_heads <= 0 || n_kv_heads <= 0 ||
        head_dim <= 0 || max_blocks_per_seq <= 0 || n_q_heads % n_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (block_size % 16 != 0 || !block_size_ok(block_size)) return PKV_ERR_UNSUPPORTED;
    const int group = n_q_heads / n_kv_heads;
    if ((head_dim != 64 && head_dim != 128) ||
        (group != 1 && group != 2 && group != 4 && group != 8))
        return PKV_ERR_UNSUPPORTED;
    const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
    if (cap > (1LL << 30)) return PKV_ERR_INVALID_ARG;
    long long max_len = max_context_len <= 0 ? cap : max_context_len;
    if (max_len > cap) max_len = cap;
    mp->max_len = static_cast<int>(max_len);
    mp->row_blocks = pkv::multi_row_blocks(max_q_len > 0 ? max_q_len : 1, group);
    mp->balanced = false;
    int P = partition_tokens;
    const int mode = pkv::kernel_override();
    if (P == 0 && (mode == 0 || mode >= 3) &&
        pkv::balanced_multi_supported(num_seqs, max_q_len, head_dim, group, block_size)) {
        // every segment's query rows fit one MMA tile: the work split evenly
        // over warps, as for decode (LLaMA-3-8B-shaped layer, 4 tokens per
        // sequence on GB300, calls back to back: 47.0 us on fixed partitions,
        // 39.2 us here)
        if (!pkv::balanced_multi_plan(num_seqs, n_q_heads, n_kv_heads, head_dim,
                                      static_cast<int>(max_len), &mp->bal))
            return PKV_ERR_CUDA;
        mp->balanced = true;
        mp->partition = 0;
        mp->max_parts = 1;
        mp->ws_bytes = mp->bal.ws_bytes;
        return PKV_OK;
    }
    if (P == 0) {
        // the largest power of two in [64, 1024] whose grid still has about
        // eight CTAs per SM (a CTA serves up to four row blocks), and at most
        // a quarter of the longest context: with skewed lengths one long
        // sequence's partitions otherwise set the time (Mistral-shaped mix,
        // two tokens per sequence: 146 us at 2048, 96 at 1024, 82 at 256;
        // 2048 was never the fastest in a sweep over the five workloads)
        int sms = 0;
        const int rc = sm_count(&sms);
        if (rc != PKV_OK) return rc;
        P = 1024;
        const int groups = (mp->row_blocks + 3) / 4;
        const long long items = static_cast<long long>(num_seqs) * n_kv_heads * groups;
        while (P > 64 && items * ((max_len + P - 1) / P) < 8LL * sms) P /= 2;
        while (P > 64 && 4LL * P > max_len) P /= 2;
    } else if (P < 16 || P % 16 != 0 || P % block_size != 0) {
        return PKV_ERR_INVALID_ARG;
    }
    const long long parts = max_len > 0 ? (max_len + P - 1) / P : 1;
    if (parts > 65535) return PKV_ERR_UNSUPPORTED;
    mp->partition = P;
    mp->max_parts = static_cast<int>(parts);
    mp->ws_bytes = mp->max_parts > 1
                       ? pkv::workspace_layout(total_q, n_q_heads, head_dim, mp->max_parts).total
                       : 0;
    return PKV_OK;
}

}  // namespace

extern "C" {

int paged_decode_multi_plan(int num_seqs, int total_q, int max_q_len, int n_q_heads,
                            int n_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                            int max_context_len, int partition_tokens, int *partition_tokens_out,
                            size_t *workspace_bytes_out) {
    MultiPlan mp{};
    const int rc = make_multi_plan(num_seqs, total_q, max_q_len, n_q_heads, n_kv_heads, head_dim,
                                   block_size, max_blocks_per_seq, max_context_len,
                                   partition_tokens, &mp);
    if (rc != PKV_OK) return rc;
    if (partition_tokens_out) *partition_tokens_out = mp.partition;
    if (workspace_bytes_out) *workspace_bytes_out = mp.ws_bytes;
    return PKV_OK;
}

int paged_decode_attention_multi_ex(void *out, const void *q, const void *k_cache,
                                    const void *v_cache, const int32_t *block_tables,
                                    const int32_t *context_lens, const int32_t *query_start,
                                    int num_seqs, int total_q, int max_q_len,
                                    int max_blocks_per_seq, int64_t num_blocks, float scale,
                                    int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                    int max_context_len, int partition_tokens, void *workspace,
                                    size_t workspace_bytes, float *lse_out, int32_t *err_word,
                                    void *cuda_stream, uint32_t flags) {
    if (flags & ~PKV_TABLES_READY) return PKV_ERR_INVALID_ARG;
    if (num_blocks <= 0 || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    MultiPlan mp{};
    int rc = make_multi_plan(num_seqs, total_q, max_q_len, n_q_heads, n_kv_heads, head_dim,
                             block_size, max_blocks_per_seq, max_context_len, partition_tokens,
                             &mp);
    if (rc != PKV_OK) return rc;
    if (num_seqs == 0 || total_q == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start, 4) ||
        (lse_out && !aligned(lse_out, 4)) || (err_word && !aligned(err_word, 4)))
        return PKV_ERR_INVALID_ARG;
    if (mp.ws_bytes > 0 &&
        (!workspace || workspace_bytes < mp.ws_bytes || !aligned(workspace, 256)))
        return PKV_ERR_WORKSPACE;
    if (static_cast<long long>(num_blocks) * n_kv_heads * block_size >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
    pkv::DecodeArgs a{};
    if (mp.balanced) {
        a.ws_acc = static_cast<float *>(workspace);  // counters, then records
    } else if (mp.ws_bytes > 0) {
        const pkv::WorkspaceLayout w =
            pkv::workspace_layout(total_q, n_q_heads, head_dim, mp.max_parts);
        char *base = static_cast<char *>(workspace);
        a.ws_acc = reinterpret_cast<float *>(base + w.acc_offset);
        a.ws_m = reinterpret_cast<float *>(base + w.m_offset);
        a.ws_l = reinterpret_cast<float *>(base + w.l_offset);
    }
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.lse_out = lse_out;
    a.err = err_word;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.max_context_len = mp.max_len;
    a.partition_tokens = mp.partition;
    a.max_parts = mp.max_parts;
    a.query_start = query_start;
    a.total_q = total_q;
    a.max_q_len = max_q_len;
    a.first_wait_polls = pkv::test_wait_polls();
    // the flag covers query_start too; fixed partitions wait first thing
    a.defer_dep_wait = (mp.balanced && (flags & PKV_TABLES_READY)) ? 2 : 0;
    const cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    const cudaError_t e = mp.balanced ? pkv::launch_decode_balanced_multi(a, mp.bal, stream)
                                      : pkv::launch_decode_multi(a, mp.row_blocks, stream);
    if (e == cudaErrorInvalidValue) return PKV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int paged_decode_attention_multi(void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, const int32_t *query_start,
                                 int num_seqs, int total_q, int max_q_len,
                                 int max_blocks_per_seq, int64_t num_blocks, float scale,
                                 int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                 int max_context_len, int partition_tokens, void *workspace,
                                 size_t workspace_bytes, float *lse_out, int32_t *err_word,
                                 void *cuda_stream) {
    return paged_decode_attention_multi_ex(out, q, k_cache, v_cache, block_tables, context_lens,
                                           query_start, num_seqs, total_q, max_q_len,
                                           max_blocks_per_seq, num_blocks, scale, n_q_heads,
                                           n_kv_heads, head_dim, block_size, max_context_len,
                                           partition_tokens, workspace, workspace_bytes, lse_out,
                                           err_word, cuda_stream, 0);
}

int paged_decode_workspace_clear(void *workspace, size_t workspace_bytes, void *cuda_stream) {
    if (workspace_bytes == 0) return PKV_OK;
    if (!workspace) return PKV_ERR_INVALID_ARG;
    const size_t n = workspace_bytes < pkv::kBalancedCounterBytes ? workspace_bytes
                                                                  : pkv::kBalancedCounterBytes;
    return cudaMemsetAsync(workspace, 0, n, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

int paged_kv_get_error(const int32_t *err_word, void *cuda_stream, int32_t *bits_out) {
    if (!err_word) return PKV_ERR_INVALID_ARG;
    int32_t host = 0;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemcpyAsync(&host, err_word, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    if (bits_out) *bits_out = host;
    return host == 0 ? PKV_OK : PKV_ERR_INDEX;
}

int paged_copy_in(void *dst, const void *src, size_t bytes, void *cuda_stream) {
    if (bytes == 0) return PKV_OK;
    if (!dst || !src || !aligned(dst, 16) || !aligned(src, 16) || bytes % 16 != 0)
        return PKV_ERR_INVALID_ARG;
    return pkv::launch_copy_in(dst, src, bytes, static_cast<cudaStream_t>(cuda_stream)) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

int paged_kv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src, const int32_t *dst,
                         const int32_t *tokens, int num_copies, int n_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, int32_t *err_word,
                         void *cuda_stream) {
    if (num_copies < 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 ||
        block_size <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_copies == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src || !dst || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(src, 4) || !aligned(dst, 4) || (tokens && !aligned(tokens, 4)) ||
        (err_word && !aligned(err_word, 4)))
        return PKV_ERR_INVALID_ARG;
    const cudaError_t e =
        pkv::launch_copy_blocks(k_cache, v_cache, src, dst, tokens, num_copies, n_kv_heads,
                                head_dim, block_size, num_blocks, err_word,
                                static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

const char *paged_kv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported head_dim, block_size or group size";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_INDEX: return "device flagged a bad index";
        case PKV_ERR_OUT_OF_BLOCKS: return "no free block in the pool";
        default: return "unknown status";
    }
}

}  // extern "C"
