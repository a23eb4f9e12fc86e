// decode_balanced_multi.cu -- multi-token (causal) paged attention on the
// balanced split: plan and launch of the kernel in balanced_kernel.cuh with
// the (query token, head) rows of each sequence's n_b new tokens as the M
// rows of its segments, n_b * (n_q_heads / n_kv_heads) <= 16.
//
// Method: "Roadmap: vLLM-style serving features for TornadoVM batched
// decode", Deferred list (batch-prefill verify of draft tokens; multi-token
// chunked prefill) and "Distributed LLM Inference Serving Platform", section
// 9.2 (chunked prefill), over the block-table gather of that page's sections
// 2, 3 and 5.1.
#include "balanced_kernel.cuh"

namespace pkv {

bool balanced_multi_supported(int num_seqs, int max_q_len, int head_dim, int group,
                              int block_size) {
    return num_seqs >= 1 && num_seqs <= kMaxSeqsMultiBalanced && max_q_len >= 1 &&
           static_cast<long long>(max_q_len) * group <= 16 && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8) && block_size % kMmaTile == 0;
}

bool balanced_multi_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int max_len,
                         BalancedPlan *plan) {
    const int G = n_q_heads / n_kv_heads;
    const int sms = sm_count_cached();
    if (sms <= 0) return false;
    // the decode split's rule: one 8-warp CTA per SM for few long segments,
    // 4-warp CTAs (as many as fit) for many short ones
    const bool few = static_cast<long long>(num_seqs) * n_kv_heads <= 2LL * sms;
    const int warps = few ? kWLarge : kWSmall;
    int per_sm = 0;
#define PKV_BALM_OCC(D_, G_)                                                          \
    if (head_dim == D_ && G == G_)                                                      \
        per_sm = few ? bal_ctas_per_sm<D_, G_, false, kWLarge, true>(num_seqs)        \
                     : bal_ctas_per_sm<D_, G_, false, kWSmall, true>(num_seqs);
    PKV_BALM_OCC(128, 1)
    PKV_BALM_OCC(128, 2)
    PKV_BALM_OCC(128, 4)
    PKV_BALM_OCC(128, 8)
    PKV_BALM_OCC(64, 1)
    PKV_BALM_OCC(64, 2)
    PKV_BALM_OCC(64, 4)
    PKV_BALM_OCC(64, 8)
#undef PKV_BALM_OCC
    if (per_sm > 0 && few && per_sm * warps > kWLarge) per_sm = 1;
    return finish_bal_plan(sms, per_sm, warps, num_seqs, n_kv_heads, head_dim, 16, max_len, plan);
}

cudaError_t launch_decode_balanced_multi(const DecodeArgs &a, const BalancedPlan &plan,
                                         cudaStream_t stream) {
    if (a.kv_fp8 || !a.query_start) return cudaErrorInvalidValue;
    CUtensorMap tk{}, tv{};
    if (!make_bal_maps(a, &tk, &tv)) return cudaErrorNotSupported;
    const int g = a.n_q_heads / a.n_kv_heads;
#define PKV_BALM_CASE(D_, G_)                                                               \
    if (a.head_dim == D_ && g == G_)                                                         \
        return plan.warps == kWLarge                                                         \
                   ? launch_bal_t<D_, G_, false, kWLarge, true>(a, plan, tk, tv, stream)     \
                   : launch_bal_t<D_, G_, false, kWSmall, true>(a, plan, tk, tv, stream);
    PKV_BALM_CASE(128, 1)
    PKV_BALM_CASE(128, 2)
    PKV_BALM_CASE(128, 4)
    PKV_BALM_CASE(128, 8)
    PKV_BALM_CASE(64, 1)
    PKV_BALM_CASE(64, 2)
    PKV_BALM_CASE(64, 4)
    PKV_BALM_CASE(64, 8)
#undef PKV_BALM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
