// append.cu -- slot-mapped append of the new token's K/V into the block pool.
//
// Method: "Distributed LLM Inference Serving Platform", section 5.1: the K and
// V vectors of a token are written directly into the physical PagedAttention
// block assigned to it (a fresh block when the tail block is full -- the
// caller's block manager chooses the slot; this kernel only writes).
// One thread moves one 16-byte vector of K and one of V: coalesced along
// head_dim, bit-exact.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pagedkv.h"
#include "pkv_internal.h"
#include "e4m3_quant.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                  const int64_t *__restrict__ slots, uint4 *__restrict__ k_cache,
                  uint4 *__restrict__ v_cache, long long total, int n_kv_heads, int chunks,
                  int block_size, long long num_slots, int32_t *err) {
    allow_dependent_launch();  // the attention kernel may get scheduled meanwhile
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int c = static_cast<int>(idx % chunks);
    const long long r = idx / chunks;
    const int j = static_cast<int>(r % n_kv_heads);
    const long long i = r / n_kv_heads;
    const long long s = slots[i];
    if (s < 0) return;  // padding token
    if (s >= num_slots) {
        if (c == 0 && j == 0) flag_error(err, PKV_ERRBIT_SLOT);
        return;
    }
    const long long block = s / block_size;
    const long long row = s % block_size;
    const long long dst = ((block * n_kv_heads + j) * block_size + row) * chunks + c;
    k_cache[dst] = k_new[idx];
    v_cache[dst] = v_new[idx];
}

}  // namespace

// One 16-byte piece per thread, every piece in flight at once: from mapped
// host memory the copy costs about one round trip over the host link.
__global__ void __launch_bounds__(256)
    copy_in_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, long long n) {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

cudaError_t launch_copy_in(void *dst, const void *src, size_t bytes, cudaStream_t stream) {
    const long long n = static_cast<long long>(bytes / 16);
    if (n == 0) return cudaSuccess;
    const long long blocks = (n + 255) / 256;
    copy_in_kernel<<<static_cast<unsigned>(blocks < 65535 ? blocks : 65535), 256, 0, stream>>>(
        static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n);
    return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs &a, cudaStream_t stream) {
    const int chunks = a.head_dim / 8;
    const long long total = static_cast<long long>(a.num_tokens) * a.n_kv_heads * chunks;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    append_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(a.k_new), static_cast<const uint4 *>(a.v_new), a.slot_mapping,
        static_cast<uint4 *>(a.k_cache), static_cast<uint4 *>(a.v_cache), total, a.n_kv_heads,
        chunks, a.block_size, a.num_blocks * a.block_size, a.err);
    return cudaGetLastError();
}

}  // namespace pkv

// Copy-on-write block copy ("Distributed LLM Inference Serving Platform",
// Lab 1 worked solution: the fresh tail block receives the shared tail's
// tokens).  One thread moves one 16-byte vector of K and one of V.
namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                       const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                       const int32_t *__restrict__ tokens, int num_copies, int n_kv_heads,
                       int chunks, int block_size, long long num_blocks, int32_t *err) {
    const long long per_copy = static_cast<long long>(n_kv_heads) * block_size * chunks;
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= per_copy * num_copies) return;
    const int i = static_cast<int>(idx / per_copy);
    const long long r = idx % per_copy;  // (head, row, chunk) inside the block
    const int row = static_cast<int>((r / chunks) % block_size);
    const int s = src[i];
    const int d = dst[i];
    const int n = tokens ? tokens[i] : block_size;
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks || n < 0 || n > block_size) {
        if (r == 0) flag_error(err, PKV_ERRBIT_SLOT);
        return;
    }
    if (row >= n) return;
    const long long block_vecs = per_copy;  // uint4 per (block, all heads)
    k_cache[d * block_vecs + r] = k_cache[s * block_vecs + r];
    v_cache[d * block_vecs + r] = v_cache[s * block_vecs + r];
}

}  // namespace

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *src,
                               const int32_t *dst, const int32_t *tokens, int num_copies,
                               int n_kv_heads, int head_dim, int block_size, long long num_blocks,
                               int32_t *err, cudaStream_t stream) {
    const int chunks = head_dim / 8;
    const long long total = static_cast<long long>(num_copies) * n_kv_heads * block_size * chunks;
    if (total == 0) return cudaSuccess;
    const long long blocks = (total + 255) / 256;
    copy_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), src, dst, tokens,
        num_copies, n_kv_heads, chunks, block_size, num_blocks, err);
    return cudaGetLastError();
}

}  // namespace pkv

// FP8 KV cache append (the quantized KV cache the "Roadmap: vLLM-style
// serving features for TornadoVM batched decode" page lists as future work):
// each value is stored as E4M3(x / scale) by quantize16 (e4m3_quant.cuh).
// One thread turns 16 fp16 values of K and of V (two 16-byte loads each) into
// one 16-byte store.
namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    append_f8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     const int64_t *__restrict__ slots, uint4 *__restrict__ k_cache,
                     uint4 *__restrict__ v_cache, long long total, int n_kv_heads, int chunks,
                     int block_size, long long num_slots, float k_scale, float v_scale,
                     int32_t *err) {
    allow_dependent_launch();  // the attention kernel may get scheduled meanwhile
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int c = static_cast<int>(idx % chunks);  // 16-value chunk of the row
    const long long r = idx / chunks;
    const int j = static_cast<int>(r % n_kv_heads);
    const long long i = r / n_kv_heads;
    const long long s = slots[i];
    if (s < 0) return;  // padding token
    if (s >= num_slots) {
        if (c == 0 && j == 0) flag_error(err, PKV_ERRBIT_SLOT);
        return;
    }
    const long long block = s / block_size;
    const long long row = s % block_size;
    const long long dst = ((block * n_kv_heads + j) * block_size + row) * chunks + c;
    k_cache[dst] = quantize16(k_new[2 * idx], k_new[2 * idx + 1], k_scale);
    v_cache[dst] = quantize16(v_new[2 * idx], v_new[2 * idx + 1], v_scale);
}

}  // namespace

cudaError_t launch_append_f8(const AppendArgs &a, float k_scale, float v_scale,
                             cudaStream_t stream) {
    const int chunks = a.head_dim / 16;
    const long long total = static_cast<long long>(a.num_tokens) * a.n_kv_heads * chunks;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    append_f8_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(a.k_new), static_cast<const uint4 *>(a.v_new), a.slot_mapping,
        static_cast<uint4 *>(a.k_cache), static_cast<uint4 *>(a.v_cache), total, a.n_kv_heads,
        chunks, a.block_size, a.num_blocks * a.block_size, k_scale, v_scale, a.err);
    return cudaGetLastError();
}

}  // namespace pkv
