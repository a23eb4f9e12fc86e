// decode_multi.cu -- multi-token (causal) paged attention: several new tokens
// of each sequence attend over its paged K/V in one call (speculative-decoding
// verify of draft tokens, chunked prefill).
//
// Method: "Roadmap: vLLM-style serving features for TornadoVM batched decode",
// Deferred list (batch-prefill verify of draft tokens; multi-token chunked
// prefill) and "Distributed LLM Inference Serving Platform", section 9.2
// (chunked prefill), over the block-table gather of that page's sections 2,
// 3 and 5.1.  Sequence b owns the query rows [query_start[b],
// query_start[b+1]) of q: its last n_b cached tokens, so query token i sits at
// position L_b - n_b + i and attends the tokens [0, L_b - n_b + i].
//
// Work: one CTA per (sequence b, KV head j, group of up to 4 blocks of 16
// query rows, KV partition), one warp per row block.  The 16 rows of a block
// are (query token, head) pairs -- row R = i * G + h of the sequence's
// n_b * G rows for KV head j -- and form the M dimension of mma.m16n8k16;
// each row has its own causal limit.  K/V tiles of 16 tokens arrive by TMA
// into a 4-stage ring that every warp of the CTA reads, so a tile is fetched
// once per group of row blocks.  One partition writes the output directly;
// several write partial (m, l, acc) states that a second kernel merges by
// log-sum-exp.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "mma_tile_multi.cuh"
#include "pagedkv.h"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kStagesM = 4;
constexpr float kLn2m = 0.69314718055994531f;

template <int D>
struct MultiCfg : MmaCfg<D> {
    static constexpr int STAGE_BYTES = 2 * MmaCfg<D>::TILE_BYTES;
    static constexpr int SMEM = 1024 + kStagesM * STAGE_BYTES;
};

constexpr int kMaxMultiWarps = 4;

template <int D, int G>
__global__ void __launch_bounds__(32 * kMaxMultiWarps)
    decode_multi_kernel(const __grid_constant__ DecodeArgs a,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, int row_groups) {
    using C = MultiCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kStagesM];
    __shared__ int s_ok[kStagesM];
    const uint32_t raw_s = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);

    const int tid = threadIdx.x;
    const int nwarps = blockDim.x >> 5;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int part = blockIdx.x;
    const int j = blockIdx.y / row_groups;
    const int rg = blockIdx.y % row_groups;  // this CTA's group of row blocks
    const int rb = rg * nwarps + warp;       // this warp's row block
    const int b = blockIdx.z;
    const int H = a.n_q_heads;
    const int Hk = a.n_kv_heads;
    const int bs = a.block_size;
    grid_dependency_wait();

    const int q0 = a.query_start[b];
    const int n = a.query_start[b + 1] - q0;
    int L = a.context_lens[b];
    const long long cap_ll = static_cast<long long>(a.max_blocks_per_seq) * bs;
    const int cap = static_cast<int>(cap_ll < a.max_context_len ? cap_ll : a.max_context_len);
    if (L < 0 || L > cap || n < 0 || n > L || n > a.max_q_len || q0 < 0 || q0 + n > a.total_q) {
        if (tid == 0 && part == 0 && blockIdx.y == 0) flag_error(a.err, PKV_ERRBIT_CONTEXT);
        return;
    }
    const int nrb = (n * G + 15) / 16;  // row blocks of this sequence
    if (rg * nwarps >= nrb) return;      // no query rows in this CTA (uniform)
    const bool warp_rows = rb < nrb;     // warps past the last block only help with barriers
    const int R0 = rb * 16;
    // query rows of this lane: r_lo = R0 + g, r_hi = R0 + g + 8
    const int r_lo = R0 + g, r_hi = R0 + g + 8;
    const bool has_lo = r_lo < n * G, has_hi = r_hi < n * G;
    const int i_lo = r_lo / G, i_hi = r_hi / G;
    const int h_lo = j * G + r_lo % G, h_hi = j * G + r_hi % G;
    // causal limits (exclusive) in absolute token positions
    const int lim_lo = has_lo ? L - n + i_lo + 1 : 0;
    const int lim_hi = has_hi ? L - n + i_hi + 1 : 0;
    // tokens any row of the CTA needs: up to its last query token
    const int rb_last = min(nrb - 1, rg * nwarps + nwarps - 1);
    const int i_last = min(n - 1, (rb_last * 16 + 15) / G);
    const int end = L - n + i_last + 1;
    const int P = a.partition_tokens;
    const int t_begin = part * P;
    const int t_end = min(end, t_begin + P);
    if (t_begin >= end) return;  // no row of the CTA reads this partition (uniform)
    const int ntiles = (t_end - t_begin + kMmaTile - 1) / kMmaTile;

    const __half *qb = static_cast<const __half *>(a.q);
    uint32_t qlo[C::NP][4], qhi[C::NP][4];
    load_q_frag<D>(qlo, qb + (static_cast<size_t>(q0 + (has_lo ? i_lo : 0)) * H + h_lo) * D,
                   has_lo, tq);
    load_q_frag<D>(qhi, qb + (static_cast<size_t>(q0 + (has_hi ? i_hi : 0)) * H + h_hi) * D,
                   has_hi, tq);

    const int32_t *bt = a.block_tables + static_cast<size_t>(b) * a.max_blocks_per_seq;
    auto issue = [&](int k) {  // thread 0
        const int st = k % kStagesM;
        const int tok0 = t_begin + k * kMmaTile;
        const int id = bt[tok0 / bs];
        const bool ok = id >= 0 && id < a.num_blocks;
        if (!ok) flag_error(a.err, PKV_ERRBIT_BLOCK_ID);
        s_ok[st] = ok;
        mbar_arrive_expect_tx(&full_bar[st], ok ? 2 * C::TILE_BYTES : 0);
        if (ok) {
            unsigned char *kdst = smem + st * C::STAGE_BYTES;
            unsigned char *vdst = kdst + C::TILE_BYTES;
            const int row = (id * Hk + j) * bs + (tok0 % bs);
#pragma unroll
            for (int bx = 0; bx < C::BOXES; ++bx) {
                tma_load_2d(kdst + bx * C::BOX_BYTES, &tmap_k, bx * 64, row, &full_bar[st]);
                tma_load_2d(vdst + bx * C::BOX_BYTES, &tmap_v, bx * 64, row, &full_bar[st]);
            }
        }
    };
    if (tid == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        for (int s = 0; s < kStagesM; ++s) mbar_init(&full_bar[s], 1);
        fence_barrier_init();
        for (int k = 0; k < ntiles && k < kStagesM; ++k) issue(k);
    }
    __syncthreads();

    float o[C::NB_D][4];
#pragma unroll
    for (int nb = 0; nb < C::NB_D; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
    float m_lo = -INFINITY, l_lo = 0.f, m_hi = -INFINITY, l_hi = 0.f;
    int k = 0;
    for (; k < ntiles; ++k) {
        const int st = k % kStagesM;
        const bool ok = mbar_wait_bounded(&full_bar[st], (k / kStagesM) & 1);
        if (__syncthreads_or(!ok)) break;
        if (warp_rows && s_ok[st]) {
            const int tok0 = t_begin + k * kMmaTile;
            unsigned char *ks = smem + st * C::STAGE_BYTES;
            mma_tile_multi<D>(ks, ks + C::TILE_BYTES, min(kMmaTile, L - tok0),
                              max(0, min(kMmaTile, lim_lo - tok0)),
                              max(0, min(kMmaTile, lim_hi - tok0)), qlo, qhi, a.scale_log2, o,
                              m_lo, l_lo, m_hi, l_hi, lane);
        }
        __syncthreads();  // every warp is done with stage st
        if (tid == 0 && k + kStagesM < ntiles) issue(k + kStagesM);
    }
    if (k < ntiles) {  // a copy never arrived: flag, drain what is in flight
        if (tid == 0) {
            flag_error(a.err, PKV_ERRBIT_TIMEOUT);
            for (int kk = k; kk < ntiles && kk < k + kStagesM; ++kk)
                mbar_wait_bounded(&full_bar[kk % kStagesM], (kk / kStagesM) & 1);
        }
        return;
    }
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);

    auto emit = [&](bool has, int i, int h, float m, float l, int c0) {
        if (!has) return;
        const size_t row = static_cast<size_t>(q0 + i) * H + h;  // (query row, head)
        if (a.max_parts == 1) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __half2 *dst = reinterpret_cast<__half2 *>(static_cast<__half *>(a.out) + row * D);
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb)
                dst[nb * 4 + tq] = __floats2half2_rn(o[nb][c0] * inv, o[nb][c0 + 1] * inv);
            if (tq == 0 && a.lse_out) a.lse_out[row] = l > 0.f ? (m + log2f(l)) * kLn2m : -INFINITY;
            return;
        }
        const size_t r = row * a.max_parts + part;
        float2 *acc = reinterpret_cast<float2 *>(a.ws_acc + r * D);
#pragma unroll
        for (int nb = 0; nb < C::NB_D; ++nb) acc[nb * 4 + tq] = make_float2(o[nb][c0], o[nb][c0 + 1]);
        if (tq == 0) {
            a.ws_m[r] = l > 0.f ? m : -INFINITY;
            a.ws_l[r] = l;
        }
    };
    if (!warp_rows) return;
    emit(has_lo, i_lo, h_lo, m_lo, l_lo, 0);
    emit(has_hi, i_hi, h_hi, m_hi, l_hi, 2);
}

// One warp per (query row, head): merge the row's partitions by log-sum-exp.
template <int D>
__global__ void __launch_bounds__(256) multi_merge_kernel(const DecodeArgs a) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int H = a.n_q_heads;
    if (warp >= a.total_q * H) return;
    const int rq = warp / H;
    // the sequence of query row rq: the last b with query_start[b] <= rq
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.query_start[mid] <= rq) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int q0 = a.query_start[b];
    const int n = a.query_start[b + 1] - q0;
    const int L = a.context_lens[b];
    const long long cap_ll = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    const int cap = static_cast<int>(cap_ll < a.max_context_len ? cap_ll : a.max_context_len);
    // rows of a sequence the partition kernel flagged stay unwritten
    if (rq - q0 >= n || n > L || L < 0 || L > cap || n > a.max_q_len || q0 + n > a.total_q) return;
    const int lim = L - n + (rq - q0) + 1;
    const int parts = min(a.max_parts, (lim + a.partition_tokens - 1) / a.partition_tokens);
    const size_t r0 = static_cast<size_t>(warp) * a.max_parts;
    float M = -INFINITY;
    for (int p = 0; p < parts; ++p) M = fmaxf(M, a.ws_m[r0 + p]);
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    if (M != -INFINITY) {
        for (int p = 0; p < parts; ++p) {
            const float mp = a.ws_m[r0 + p];
            if (mp == -INFINITY) continue;
            const float w = exp2f(mp - M);
            lsum = fmaf(w, a.ws_l[r0 + p], lsum);
            const float *src = a.ws_acc + (r0 + p) * D;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, src[lane + 32 * e], acc[e]);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __half *dst = static_cast<__half *>(a.out) + static_cast<size_t>(warp) * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) dst[lane + 32 * e] = __float2half_rn(acc[e] * inv);
    if (lane == 0 && a.lse_out) a.lse_out[warp] = lsum > 0.f ? (M + log2f(lsum)) * kLn2m : -INFINITY;
}

template <int D, int G>
cudaError_t launch_multi_t(const DecodeArgs &a, int row_blocks, const CUtensorMap &tk,
                           const CUtensorMap &tv, cudaStream_t stream) {
    auto kern = decode_multi_kernel<D, G>;
    const int smem = MultiCfg<D>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // one warp per row block, up to kMaxMultiWarps row blocks per CTA
    const int nw = row_blocks < kMaxMultiWarps ? row_blocks : kMaxMultiWarps;
    const int row_groups = (row_blocks + nw - 1) / nw;
    const long long y = static_cast<long long>(a.n_kv_heads) * row_groups;
    if (y > 65535 || a.num_seqs > 65535) return cudaErrorInvalidValue;
    dim3 grid(a.max_parts, static_cast<unsigned>(y), a.num_seqs);
    e = launch_pdl(kern, grid, dim3(32 * nw), static_cast<size_t>(smem), stream, a, tk, tv,
                   row_groups);
    if (e != cudaSuccess || a.max_parts == 1) return e;
    const long long warps = static_cast<long long>(a.total_q) * a.n_q_heads;
    const long long blocks = (warps * 32 + 255) / 256;
    multi_merge_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

int multi_row_blocks(int max_q_len, int group) { return (max_q_len * group + 15) / 16; }

cudaError_t launch_decode_multi(const DecodeArgs &a, int row_blocks, cudaStream_t stream) {
    const long long rows = a.num_blocks * a.n_kv_heads * static_cast<long long>(a.block_size);
    CUtensorMap tk, tv;
    if (!make_cache_map(&tk, a.k_cache, rows, a.head_dim) ||
        !make_cache_map(&tv, a.v_cache, rows, a.head_dim))
        return cudaErrorNotSupported;
    const int g = a.n_q_heads / a.n_kv_heads;
#define PKV_MULTI_CASE(D_, G_) \
    if (a.head_dim == D_ && g == G_) return launch_multi_t<D_, G_>(a, row_blocks, tk, tv, stream);
    PKV_MULTI_CASE(128, 1)
    PKV_MULTI_CASE(128, 2)
    PKV_MULTI_CASE(128, 4)
    PKV_MULTI_CASE(128, 8)
    PKV_MULTI_CASE(64, 1)
    PKV_MULTI_CASE(64, 2)
    PKV_MULTI_CASE(64, 4)
    PKV_MULTI_CASE(64, 8)
#undef PKV_MULTI_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
