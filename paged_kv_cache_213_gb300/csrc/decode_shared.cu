// decode_shared.cu -- the shared-prefix pass of prefix-aware decode attention.
//
// Sequences that share their leading physical blocks (forked completions of
// one prompt, requests with a cached common prefix) form a group: the caller
// lists the groups as consecutive ranges of sequences with the number of
// prefix tokens they share.  This kernel reads each shared K/V tile ONCE per
// chunk of members and computes its contribution for all of their queries: a
// CTA of up to 4 warps consumes every tile staged by TMA, each warp owns 16
// query rows -- both halves of the m16n8k16 row tile -- i.e. 16/G members of
// the group.  It leaves, per (member, query head, partition of the prefix), a
// partial softmax state (m, l, acc) that the balanced kernel folds into the
// member's private suffix by log-sum-exp.
//
// Method: "Distributed LLM Inference Serving Platform", section 2 (prompt
// blocks shared by parallel completions with a reference count) and Lab 1
// (forkSequence); attention per sections 3 and 5.1 of that page; the split
// of one softmax into partial states merged by log-sum-exp follows
// FlashAttention-2 (section 14 references).  E4M3 caches ("Roadmap:
// vLLM-style serving features for TornadoVM batched decode", KV-cache list:
// quantized FP8 KV cache) are widened in the tile math; their partial sums
// keep the E4M3 tile math's register order and v_scale units, as the suffix
// pass expects.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "mma_tile.cuh"
#include "pagedkv.h"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"
#include "shared_prefix.cuh"

namespace pkv {
namespace {

constexpr int kWS = 4;  // most warps per CTA (the launch uses only those with rows)
// Stages of the CTA-wide ring: fp16 tiles; E4M3 tiles (half the bytes, so
// twice the stages keep as many bytes in flight).  70B-shaped batch, E4M3,
// the whole prefix-aware call, back to back / isolated: 4 stages 72.8 / 84.0
// us, 6 stages 82.9 / 78.6 us, 8 stages 73.2 / 77.1 us.
#ifndef PKV_SHARED_STAGES
#define PKV_SHARED_STAGES 4
#endif
#ifndef PKV_SHARED_STAGES_F8
#define PKV_SHARED_STAGES_F8 8
#endif

template <int D, bool F8>
struct ShCfg : MmaCfg<D> {
    static constexpr int STAGES = F8 ? PKV_SHARED_STAGES_F8 : PKV_SHARED_STAGES;
    // one tile of one cache: fp16 TMA boxes, or one box of E4M3 codes
    static constexpr int KV_BYTES = F8 ? kMmaTile * D : MmaCfg<D>::TILE_BYTES;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;  // multiple of 1024
    static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
};

template <int D, int G, bool F8>
__global__ void __launch_bounds__(kWS * 32)
    decode_shared_kernel(const __grid_constant__ DecodeArgs a,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v) {
    using C = ShCfg<D, F8>;
    constexpr int kStagesS = C::STAGES;
    constexpr int MPW = 16 / G;  // members per warp
    const int nwarps = blockDim.x >> 5;
    const int MPC = nwarps * MPW;  // members per CTA chunk
    const int nthreads = blockDim.x;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kStagesS];
    __shared__ int s_ok[kStagesS];
    __shared__ int s_min_len;
    const uint32_t raw_s = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int H = a.n_q_heads;
    const int Hk = a.n_kv_heads;
    const int bs = a.block_size;
    const int gi = blockIdx.x / a.sh_chunks;
    const int chunk = blockIdx.x % a.sh_chunks;
    const int j = blockIdx.y;
    const int part = blockIdx.z;
    if (gi >= a.num_groups) return;
    if (tid == 0) {
        s_min_len = INT_MAX;
        for (int fb = 0; fb < kStagesS; ++fb) mbar_init(&full_bar[fb], 1);
        fence_barrier_init();
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    // The context lengths and block tables into L2, spread over the CTAs,
    // while the kernel before may still run (a prefetch reads nothing stale),
    // then the wait for it before anything it may have written is read.
    if (warp == 0) {
        const size_t cta = blockIdx.x + static_cast<size_t>(gridDim.x) *
                                            (blockIdx.y + static_cast<size_t>(gridDim.y) * blockIdx.z);
        const size_t ctas = static_cast<size_t>(gridDim.x) * gridDim.y * gridDim.z;
        const size_t len_lines = (static_cast<size_t>(a.num_seqs) * sizeof(int32_t) + 127) / 128;
        const size_t tab_lines =
            (static_cast<size_t>(a.num_seqs) * a.max_blocks_per_seq * sizeof(int32_t) + 127) / 128;
        for (size_t ln = cta * 32 + lane; ln < len_lines + tab_lines; ln += ctas * 32)
            prefetch_l2(ln < len_lines
                            ? reinterpret_cast<const char *>(a.context_lens) + ln * 128
                            : reinterpret_cast<const char *>(a.block_tables) + (ln - len_lines) * 128);
    }
    // Everything before this grid in the stream is complete after the wait,
    // so the suffix pass that follows may be scheduled as this grid's CTAs
    // retire: it reads nothing this grid writes before its own dependency
    // wait, and what it reads before that wait (lengths, tables, the private
    // K/V) was written before this grid started.  With sh_tables_ready the
    // kernel before writes no lengths, tables or groups, so the group's
    // bounds and shortest member are read before the wait.
    if (!a.sh_tables_ready) {
        grid_dependency_wait();
        allow_dependent_launch();
    }
    const int first = a.group_offsets[gi];
    const int count = a.group_offsets[gi + 1] - first;
    const int m0 = chunk * MPC;
    if (count < 2 || m0 >= count) {  // CTA-uniform
        // an exit counts as this CTA's trigger: wait first, so that the
        // suffix pass's early reads never run ahead of the kernel before
        if (a.sh_tables_ready) grid_dependency_wait();
        return;
    }
    const int nm = min(MPC, count - m0);

    // shared tiles of the group (the same rule as the private-suffix kernel)
    __syncthreads();
    for (int i = tid; i < count; i += nthreads) atomicMin(&s_min_len, shared_len_of(a, first + i));
    __syncthreads();
    if (a.sh_tables_ready) {  // q and the caches may come from the kernel before
        grid_dependency_wait();
        allow_dependent_launch();
    }
    const int St = shared_tiles(a, gi, s_min_len);
    const int PT = a.sh_part_tiles;
    const int t0 = part * PT;
    const int n = max(0, min(St, t0 + PT) - t0);

    // query rows of this warp: row r -> member m0 + MPW*warp + r/G, head r%G
    const int ml_lo = warp * MPW + g / G;
    const int ml_hi = warp * MPW + (g + 8) / G;
    const bool has_lo = ml_lo < nm;
    const bool has_hi = ml_hi < nm;
    const int b_lo = first + m0 + (has_lo ? ml_lo : 0);
    const int b_hi = first + m0 + (has_hi ? ml_hi : 0);
    const int h_lo = j * G + g % G;
    const int h_hi = j * G + (g + 8) % G;
    const __half *qb = static_cast<const __half *>(a.q);
    uint32_t qlo[C::NP][4], qhi[C::NP][4];
    load_q_frag<D>(qlo, qb + (static_cast<size_t>(b_lo) * H + h_lo) * D, has_lo, tq);
    load_q_frag<D>(qhi, qb + (static_cast<size_t>(b_hi) * H + h_hi) * D, has_hi, tq);

    const int32_t *bt_lead = a.block_tables + static_cast<size_t>(first) * a.max_blocks_per_seq;
    auto issue = [&](int i) {  // thread 0
        const int st = i % kStagesS;
        const int tok0 = (t0 + i) * kMmaTile;
        const int id = bt_lead[tok0 / bs];
        const bool ok = id >= 0 && id < a.num_blocks;
        if (!ok) flag_error(a.err, PKV_ERRBIT_BLOCK_ID);
        s_ok[st] = ok;
        mbar_arrive_expect_tx(&full_bar[st], ok ? 2 * C::KV_BYTES : 0);
        if (ok) {
            unsigned char *kdst = smem + st * C::STAGE_BYTES;
            unsigned char *vdst = kdst + C::KV_BYTES;
            const int row = (id * Hk + j) * bs + (tok0 % bs);
            if constexpr (F8) {  // one swizzled box per cache
                tma_load_2d(kdst, &tmap_k, 0, row, &full_bar[st]);
                tma_load_2d(vdst, &tmap_v, 0, row, &full_bar[st]);
            } else {
#pragma unroll
                for (int bx = 0; bx < C::BOXES; ++bx) {
                    tma_load_2d(kdst + bx * C::BOX_BYTES, &tmap_k, bx * 64, row, &full_bar[st]);
                    tma_load_2d(vdst + bx * C::BOX_BYTES, &tmap_v, bx * 64, row, &full_bar[st]);
                }
            }
        }
    };
    if (tid == 0)
        for (int i = 0; i < n && i < kStagesS; ++i) issue(i);

    float o[C::NB_D][4];
#pragma unroll
    for (int nb = 0; nb < C::NB_D; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
    float m_lo = -INFINITY, l_lo = 0.f, m_hi = -INFINITY, l_hi = 0.f;
    int i = 0;
    bool timed_out = false;
    for (; i < n; ++i) {
        const int st = i % kStagesS;
        const bool ok = mbar_wait_bounded(&full_bar[st], (i / kStagesS) & 1);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        if (s_ok[st]) {  // a bad block id leaves this tile out (flagged above)
            const unsigned char *ks = smem + st * C::STAGE_BYTES;
            mma_tile_2rows<D, F8>(ks, ks + C::KV_BYTES, qlo, qhi, a.scale_log2, o, m_lo, l_lo,
                                  m_hi, l_hi, lane);
        }
        __syncthreads();  // every warp is done with stage st
        if (tid == 0 && i + kStagesS < n) issue(i + kStagesS);
    }
    if (timed_out) {
        if (tid == 0) {
            flag_error(a.err, PKV_ERRBIT_TIMEOUT);
            for (int k = i; k < n && k < i + kStagesS; ++k)
                mbar_wait_bounded(&full_bar[k % kStagesS], (k / kStagesS) & 1);
        }
        return;
    }
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    // partial state of (member, head, this partition); empty partitions give m = -inf
    const int parts = a.sh_parts;
    if (has_lo) {
        const size_t r = (static_cast<size_t>(b_lo) * H + h_lo) * parts + part;
        float2 *acc = reinterpret_cast<float2 *>(a.sh_acc + r * D);
#pragma unroll
        for (int nb = 0; nb < C::NB_D; ++nb) acc[nb * 4 + tq] = make_float2(o[nb][0], o[nb][1]);
        if (tq == 0) {
            a.sh_m[r] = n > 0 ? m_lo : -INFINITY;
            a.sh_l[r] = l_lo;
        }
    }
    if (has_hi) {
        const size_t r = (static_cast<size_t>(b_hi) * H + h_hi) * parts + part;
        float2 *acc = reinterpret_cast<float2 *>(a.sh_acc + r * D);
#pragma unroll
        for (int nb = 0; nb < C::NB_D; ++nb) acc[nb * 4 + tq] = make_float2(o[nb][2], o[nb][3]);
        if (tq == 0) {
            a.sh_m[r] = n > 0 ? m_hi : -INFINITY;
            a.sh_l[r] = l_hi;
        }
    }
}

template <int D, int G, bool F8>
cudaError_t launch_shared_t(const DecodeArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t stream) {
    using C = ShCfg<D, F8>;
    const size_t smem = 1024 + C::PIPE_BYTES;
    auto kern = decode_shared_kernel<D, G, F8>;
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(a.num_groups * a.sh_chunks, a.n_kv_heads, a.sh_parts);
    // programmatic dependent launch: the CTAs may start while the kernel
    // before drains; they wait for it (griddepcontrol.wait) before reading
    return launch_pdl(kern, grid, dim3(a.sh_warps * 32), smem, stream, a, tk, tv);
}

template <int D, int G, bool F8>
int shared_ctas_per_sm_t(int warps) {
    using C = ShCfg<D, F8>;
    auto kern = decode_shared_kernel<D, G, F8>;
    const size_t smem = 1024 + C::PIPE_BYTES;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, warps * 32, smem) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace

int shared_members_per_warp(int group) { return 16 / group; }
int shared_max_warps() { return kWS; }

int shared_ctas_per_sm(int head_dim, int group, int warps, bool kv_fp8) {
#define PKV_SH_OCC(D_, G_)                                                               \
    if (head_dim == D_ && group == G_)                                                     \
        return kv_fp8 ? shared_ctas_per_sm_t<D_, G_, true>(warps)                          \
                      : shared_ctas_per_sm_t<D_, G_, false>(warps);
    PKV_SH_OCC(128, 1)
    PKV_SH_OCC(128, 2)
    PKV_SH_OCC(128, 4)
    PKV_SH_OCC(128, 8)
    PKV_SH_OCC(64, 1)
    PKV_SH_OCC(64, 2)
    PKV_SH_OCC(64, 4)
    PKV_SH_OCC(64, 8)
#undef PKV_SH_OCC
    return 0;
}

cudaError_t launch_decode_shared(const DecodeArgs &a, cudaStream_t stream) {
    const long long rows = a.num_blocks * a.n_kv_heads * static_cast<long long>(a.block_size);
    CUtensorMap tk, tv;
    if (a.kv_fp8 ? (!make_cache_map_e4m3(&tk, a.k_cache, rows, a.head_dim) ||
                    !make_cache_map_e4m3(&tv, a.v_cache, rows, a.head_dim))
                 : (!make_cache_map(&tk, a.k_cache, rows, a.head_dim) ||
                    !make_cache_map(&tv, a.v_cache, rows, a.head_dim)))
        return cudaErrorNotSupported;
    const int g = a.n_q_heads / a.n_kv_heads;
#define PKV_SH_CASE(D_, G_)                                                         \
    if (a.head_dim == D_ && g == G_)                                                 \
        return a.kv_fp8 ? launch_shared_t<D_, G_, true>(a, tk, tv, stream)           \
                        : launch_shared_t<D_, G_, false>(a, tk, tv, stream);
    PKV_SH_CASE(128, 1)
    PKV_SH_CASE(128, 2)
    PKV_SH_CASE(128, 4)
    PKV_SH_CASE(128, 8)
    PKV_SH_CASE(64, 1)
    PKV_SH_CASE(64, 2)
    PKV_SH_CASE(64, 4)
    PKV_SH_CASE(64, 8)
#undef PKV_SH_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
