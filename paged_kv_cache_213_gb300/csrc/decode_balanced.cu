// decode_balanced.cu -- paged decode attention with the work split evenly
// over warps (the default tensor-core path): plan and launch of the kernel in
// balanced_kernel.cuh for one query token per sequence, fp16 or E4M3 caches.
//
// Method: "Distributed LLM Inference Serving Platform", sections 2-3 (block
// table gather) and 5.1 (attention over every block of a sequence's table),
// GQA from section 1; online softmax and the log-sum-exp combination of
// partial results from FlashAttention-2 (section 14 references).
#include "balanced_kernel.cuh"

namespace pkv {

bool balanced_supported(int num_seqs, int head_dim, int group, int block_size,
                        long long cache_rows) {
    return num_seqs >= 1 && num_seqs <= kMaxSeqsBalanced && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8) && block_size % kMmaTile == 0 &&
           cache_rows < (1LL << 31);
}

bool balanced_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int max_len,
                   BalancedPlan *plan, bool kv_fp8) {
    const int G = n_q_heads / n_kv_heads;
    const int sms = sm_count_cached();
    if (sms <= 0) return false;
    // Few (sequence, KV head) segments: each is long and every warp range
    // lies inside one, so more warps only cut the segments into more pieces
    // (more records, release fences and merges).  Eight warps per SM, as one
    // CTA, then beat twelve (LLaMA-3-8B-shaped layer, 256 segments: 44.5 ->
    // 40.2 us; 32k contexts, 64 segments: 187 -> 175 us).  Many short
    // segments are seldom cut and gain from the extra warps (Mistral mix,
    // 1024 segments: 45 -> 53 us at eight), and so does the E4M3 path, which
    // is issue-bound.
    const bool few = !kv_fp8 && static_cast<long long>(num_seqs) * n_kv_heads <= 2LL * sms;
    const int warps = few ? kWLarge : kWSmall;
    int per_sm = 0;
#define PKV_BAL_OCC(D_, G_)                                                                \
    if (head_dim == D_ && G == G_)                                                           \
        per_sm = kv_fp8 ? bal_ctas_per_sm<D_, G_, true, kWSmall, false>(num_seqs)           \
                        : (few ? bal_ctas_per_sm<D_, G_, false, kWLarge, false>(num_seqs)   \
                               : bal_ctas_per_sm<D_, G_, false, kWSmall, false>(num_seqs));
    PKV_BAL_OCC(128, 1)
    PKV_BAL_OCC(128, 2)
    PKV_BAL_OCC(128, 4)
    PKV_BAL_OCC(128, 8)
    PKV_BAL_OCC(64, 1)
    PKV_BAL_OCC(64, 2)
    PKV_BAL_OCC(64, 4)
    PKV_BAL_OCC(64, 8)
#undef PKV_BAL_OCC
    if (per_sm > 0 && few && per_sm * warps > kWLarge) per_sm = kWLarge / warps > 0 ? kWLarge / warps : 1;
    return finish_bal_plan(sms, per_sm, warps, num_seqs, n_kv_heads, head_dim, G, max_len, plan);
}

cudaError_t launch_decode_balanced(const DecodeArgs &a, const BalancedPlan &plan,
                                   cudaStream_t stream) {
    CUtensorMap tk{}, tv{};
    if (!make_bal_maps(a, &tk, &tv)) return cudaErrorNotSupported;
    const int g = a.n_q_heads / a.n_kv_heads;
#define PKV_BAL_CASE(D_, G_)                                                                   \
    if (a.head_dim == D_ && g == G_)                                                            \
        return a.kv_fp8 ? launch_bal_t<D_, G_, true, kWSmall, false>(a, plan, tk, tv, stream)   \
                        : (plan.warps == kWLarge                                                \
                               ? launch_bal_t<D_, G_, false, kWLarge, false>(a, plan, tk, tv, stream) \
                               : launch_bal_t<D_, G_, false, kWSmall, false>(a, plan, tk, tv, stream));
    PKV_BAL_CASE(128, 1)
    PKV_BAL_CASE(128, 2)
    PKV_BAL_CASE(128, 4)
    PKV_BAL_CASE(128, 8)
    PKV_BAL_CASE(64, 1)
    PKV_BAL_CASE(64, 2)
    PKV_BAL_CASE(64, 4)
    PKV_BAL_CASE(64, 8)
#undef PKV_BAL_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
