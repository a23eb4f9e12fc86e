// static_scratch.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// Some callers hold only the buffers they were handed: an operator running
// inside a host framework's plugin interface that passes tensors in and out
// but exposes no allocator, or a foreign-language binding with no access to
// a CUDA allocator.  They cannot provide the split-K workspace that
// paged_decode_attention needs for long contexts.  This entry point uses a
// fixed-size scratch array that lives in the library's own device memory
// instead, and otherwise runs the same kernels.
//
// Layout of the array: the first kBalancedCounterBytes hold the balanced
// split's per-segment arrival counters, and the balanced kernel's partial
// records follow them, as in a caller's workspace.  A fixed-partition plan
// puts its partial sums after the counter region too, so that it never
// overwrites the counters.  Before each balanced launch the call clears the
// counter region on the caller's stream (cudaMemsetAsync allocates nothing),
// so a previous call that timed out leaves no stale counts behind.
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace {

// Scratch for split-K partial results.  Every GPU on which this library is
// loaded holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_pkv_scratch[PKV_NOALLOC_SCRATCH_BYTES];

static_assert(pkv::kBalancedCounterBytes % 256 == 0, "the partials after the counters stay aligned");
static_assert(pkv::kBalancedCounterBytes < PKV_NOALLOC_SCRATCH_BYTES, "room after the counters");

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_pkv_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address has to be asked
// for, once per device, with that device current.
int scratch_address(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int paged_decode_attention_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
    int max_blocks_per_seq, int64_t num_blocks, float scale, int n_q_heads, int n_kv_heads,
    int head_dim, int block_size, int max_context_len, int partition_tokens, float *lse_out,
    int32_t *err_word, void *cuda_stream) {
    int P = 0;
    size_t need = 0;
    int rc = paged_decode_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                               max_blocks_per_seq, max_context_len, partition_tokens, &P, &need);
    if (rc != PKV_OK) return rc;
    // a balanced plan's need already starts with the counter region; a
    // fixed-partition plan's partials go after it
    const size_t offset = (P > 0 && need > 0) ? pkv::kBalancedCounterBytes : 0;
    if (need > static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES) - offset) return PKV_ERR_WORKSPACE;
    if (need == 0 || num_seqs == 0)
        return paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens,
                                      num_seqs, max_blocks_per_seq, num_blocks, scale, n_q_heads,
                                      n_kv_heads, head_dim, block_size, max_context_len, P,
                                      nullptr, 0, lse_out, err_word, cuda_stream);
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != PKV_OK) return rc;
    if (P == 0 &&
        cudaMemsetAsync(scratch, 0, pkv::kBalancedCounterBytes,
                        static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                  max_blocks_per_seq, num_blocks, scale, n_q_heads, n_kv_heads,
                                  head_dim, block_size, max_context_len, P,
                                  static_cast<unsigned char *>(scratch) + offset, need, lse_out,
                                  err_word, cuda_stream);
}
