// decode.cu -- paged decode attention: one CTA per (sequence, KV head,
// partition of the context), K/V block tiles streamed into shared memory by
// the bulk-copy (TMA) engine through a ring of mbarrier-tracked stages, the
// GQA query group's logits and the P.V accumulate on the CUDA cores in fp32,
// warp-shuffle reductions for the dot products, and a log-sum-exp merge
// kernel for sequences split over several partitions.
//
// Method: "Distributed LLM Inference Serving Platform", sections 2-3 (block
// table gather) and 5.1 (attention over all blocks of a sequence's table);
// grouped-query attention from section 1 of the same page.  The online
// softmax and the partition merge follow FlashAttention-2 (cited in section
// 14 of that page) and its flash-decoding split.
#include <cuda_fp16.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kTile = 16;      // tokens per pipeline stage
constexpr int kThreads = 128;  // 4 warps
constexpr float kLn2 = 0.69314718055994531f;

template <int D, int G>
struct Cfg {
    static constexpr int CH = D / 8;             // 16-byte chunks in one K/V row
    static constexpr int RG = kThreads / CH;     // row groups (threads sharing a chunk)
    static constexpr int RPT = kTile / RG;       // rows of a tile per thread
    static constexpr int TILE_BYTES = kTile * D * 2;
    static constexpr int STAGES = (D >= 128) ? 4 : 8;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
    static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
    static constexpr int RED_BYTES = (RG * G * D + 3 * RG * G + 2 * G) * 4;
    static constexpr int UNION_BYTES =
        ((PIPE_BYTES > RED_BYTES ? PIPE_BYTES : RED_BYTES) + 127) / 128 * 128;
    static_assert(RG * CH == kThreads && RPT * RG == kTile, "thread layout");
};

// Context length of sequence b after validation.  Out-of-range values are
// flagged (when `flag`) and clamped so that every index stays in bounds.
__device__ __forceinline__ int checked_len(const DecodeArgs &a, int b, bool flag) {
    const int L = a.context_lens[b];
    const long long cap_ll = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    const int cap = static_cast<int>(cap_ll < a.max_context_len ? cap_ll : a.max_context_len);
    if (L < 0 || L > cap) {
        if (flag) flag_error(a.err, PKV_ERRBIT_CONTEXT);
        return L < 0 ? 0 : cap;
    }
    return L;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads)
    decode_partition_kernel(const DecodeArgs a) {
    using C = Cfg<D, G>;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint64_t full_bar[C::STAGES];
    int32_t *s_blk = reinterpret_cast<int32_t *>(smem + C::UNION_BYTES);

    const int b = blockIdx.x;
    const int j = blockIdx.y;
    const int part = blockIdx.z;
    const int tid = threadIdx.x;
    const int c = tid % C::CH;   // chunk of head_dim owned by this thread
    const int rg = tid / C::CH;  // its row group: rows rg, rg + RG, ...
    const int H = a.n_q_heads;
    const int Hk = a.n_kv_heads;
    const int bs = a.block_size;
    const int P = a.partition_tokens;

    const int L = checked_len(a, b, j == 0 && part == 0);
    const int n_parts = (L + P - 1) / P;
    if (part >= (n_parts > 1 ? n_parts : 1)) return;
    const int t_begin = part * P;
    const int t_end = min(L, t_begin + P);
    const int n_tok = max(t_end - t_begin, 0);
    const int n_tiles = (n_tok + kTile - 1) / kTile;
    const int lb0 = t_begin / bs;
    const int n_blk = (n_tok + bs - 1) / bs;

    // Physical block ids of this partition, checked against the pool.
    const int32_t *bt_row = a.block_tables + static_cast<size_t>(b) * a.max_blocks_per_seq;
    for (int i = tid; i < n_blk; i += kThreads) {
        int32_t id = bt_row[lb0 + i];
        if (id < 0 || id >= a.num_blocks) {
            flag_error(a.err, PKV_ERRBIT_BLOCK_ID);
            id = -1;
        }
        s_blk[i] = id;
    }
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&full_bar[s], 1);
        fence_barrier_init();
    }

    // The query group of KV head j, in log2 units (scale * log2 e folded in).
    float qf[G][8];
    {
        const __half *qb = static_cast<const __half *>(a.q) +
                           (static_cast<size_t>(b) * H + static_cast<size_t>(j) * G) * D + c * 8;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint4 v = *reinterpret_cast<const uint4 *>(qb + static_cast<size_t>(h) * D);
            unpack8(v, qf[h]);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[h][e] *= a.scale_log2;
        }
    }
    __syncthreads();

    const __half *kcache = static_cast<const __half *>(a.k_cache);
    const __half *vcache = static_cast<const __half *>(a.v_cache);
    const size_t head_elems = static_cast<size_t>(bs) * D;  // one (block, head) row set

    // Thread 0: start the copies of tile i into its stage.
    auto issue = [&](int i) {
        const int s = i % C::STAGES;
        unsigned char *kdst = smem + s * C::STAGE_BYTES;
        unsigned char *vdst = kdst + C::TILE_BYTES;
        const int tok0 = t_begin + i * kTile;
        if (bs >= kTile) {
            const int id = s_blk[tok0 / bs - lb0];
            if (id >= 0) {
                const size_t off = (static_cast<size_t>(id) * Hk + j) * head_elems +
                                   static_cast<size_t>(tok0 % bs) * D;
                mbar_arrive_expect_tx(&full_bar[s], 2 * C::TILE_BYTES);
                bulk_copy_g2s(kdst, kcache + off, C::TILE_BYTES, &full_bar[s]);
                bulk_copy_g2s(vdst, vcache + off, C::TILE_BYTES, &full_bar[s]);
            } else {
                mbar_arrive_expect_tx(&full_bar[s], 0);
            }
        } else {
            // several whole blocks per tile (block_size 1, 2, 4 or 8)
            const int per = kTile / bs;
            const uint32_t seg = static_cast<uint32_t>(bs) * D * 2;
            uint32_t total = 0;
            for (int k = 0; k < per; ++k) {
                const int t = tok0 + k * bs;
                if (t < t_end && s_blk[t / bs - lb0] >= 0) total += 2 * seg;
            }
            mbar_arrive_expect_tx(&full_bar[s], total);
            for (int k = 0; k < per; ++k) {
                const int t = tok0 + k * bs;
                if (t >= t_end) break;
                const int id = s_blk[t / bs - lb0];
                if (id < 0) continue;
                const size_t off = (static_cast<size_t>(id) * Hk + j) * head_elems;
                bulk_copy_g2s(kdst + k * seg, kcache + off, seg, &full_bar[s]);
                bulk_copy_g2s(vdst + k * seg, vcache + off, seg, &full_bar[s]);
            }
        }
    };

    float m[G], l[G], acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    }

    const int prefetch = n_tiles < C::STAGES ? n_tiles : C::STAGES;
    if (tid == 0)
        for (int i = 0; i < prefetch; ++i) issue(i);
    int issued = prefetch;

    int i = 0;
    bool timed_out = false;
    for (; i < n_tiles; ++i) {
        const int s = i % C::STAGES;
        const bool ok = mbar_wait_bounded(&full_bar[s], (i / C::STAGES) & 1);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        // every thread is done with tile i-1: refill its stage
        if (i >= 1 && i - 1 + C::STAGES < n_tiles) {
            if (tid == 0) issue(i - 1 + C::STAGES);
            ++issued;
        }

        const unsigned char *ks = smem + s * C::STAGE_BYTES;
        const unsigned char *vs = ks + C::TILE_BYTES;
        const int tok0 = t_begin + i * kTile;

        float sc[C::RPT][G];
#pragma unroll
        for (int rr = 0; rr < C::RPT; ++rr) {
            const int row = rg + rr * C::RG;
            const uint4 kv = *reinterpret_cast<const uint4 *>(ks + (row * D + c * 8) * 2);
            float kf[8];
            unpack8(kv, kf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float d0 = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) d0 = fmaf(qf[h][e], kf[e], d0);
                sc[rr][h] = d0;
            }
        }
        // dot products: sum over the CH lanes that hold one row
#pragma unroll
        for (int off = C::CH / 2; off >= 1; off >>= 1)
#pragma unroll
            for (int rr = 0; rr < C::RPT; ++rr)
#pragma unroll
                for (int h = 0; h < G; ++h)
                    sc[rr][h] += __shfl_xor_sync(0xffffffffu, sc[rr][h], off);

        bool valid[C::RPT];
        float vf[C::RPT][8];
#pragma unroll
        for (int rr = 0; rr < C::RPT; ++rr) {
            const int row = rg + rr * C::RG;
            const int t = tok0 + row;
            valid[rr] = t < t_end && s_blk[t / bs - lb0] >= 0;
            const uint4 vv = *reinterpret_cast<const uint4 *>(vs + (row * D + c * 8) * 2);
            unpack8(vv, vf[rr]);
        }
        // online softmax over this thread's rows, then P.V
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mx = -INFINITY;
#pragma unroll
            for (int rr = 0; rr < C::RPT; ++rr)
                if (valid[rr]) mx = fmaxf(mx, sc[rr][h]);
            if (mx > m[h]) {
                const float corr = exp2f(m[h] - mx);
                l[h] *= corr;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] *= corr;
                m[h] = mx;
            }
#pragma unroll
            for (int rr = 0; rr < C::RPT; ++rr) {
                if (!valid[rr]) continue;  // never multiply rows outside [0, L)
                const float p = exp2f(sc[rr][h] - m[h]);
                l[h] += p;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(p, vf[rr][e], acc[h][e]);
            }
        }
    }

    if (timed_out) {
        if (tid == 0) {
            flag_error(a.err, PKV_ERRBIT_TIMEOUT);
            // let the copies still in flight land before the buffers are reused
            for (int k = i; k < issued; ++k)
                mbar_wait_bounded(&full_bar[k % C::STAGES], (k / C::STAGES) & 1);
        }
    }
    __syncthreads();

    // Merge the RG row groups' running states (log-sum-exp) through shared memory.
    float *red_acc = reinterpret_cast<float *>(smem);  // [RG][G][D]
    float *red_m = red_acc + C::RG * G * D;            // [RG][G]
    float *red_l = red_m + C::RG * G;                  // [RG][G]
    float *red_w = red_l + C::RG * G;                  // [RG][G]
    float *red_tot = red_w + C::RG * G;                // [G]
    float *red_M = red_tot + G;                        // [G]
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float4 *dst = reinterpret_cast<float4 *>(red_acc + (rg * G + h) * D + c * 8);
        dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
        if (c == 0) {
            red_m[rg * G + h] = m[h];
            red_l[rg * G + h] = l[h];
        }
    }
    __syncthreads();
    if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
        for (int r = 0; r < C::RG; ++r) M = fmaxf(M, red_m[r * G + h]);
        float tot = 0.f;
        for (int r = 0; r < C::RG; ++r) {
            const float w = (M == -INFINITY) ? 0.f : exp2f(red_m[r * G + h] - M);
            red_w[r * G + h] = w;
            tot = fmaf(w, red_l[r * G + h], tot);
        }
        red_tot[h] = tot;
        red_M[h] = M;
    }
    __syncthreads();

    const bool single = n_parts <= 1;
    const size_t bh0 = static_cast<size_t>(b) * H + static_cast<size_t>(j) * G;
    for (int o = tid; o < G * D; o += kThreads) {
        const int h = o / D;
        const int e = o % D;
        float A = 0.f;
#pragma unroll
        for (int r = 0; r < C::RG; ++r) A = fmaf(red_w[r * G + h], red_acc[(r * G + h) * D + e], A);
        const size_t bh = bh0 + h;
        if (single) {
            const float tot = red_tot[h];
            static_cast<__half *>(a.out)[bh * D + e] = __float2half_rn(tot > 0.f ? A / tot : 0.f);
        } else {
            a.ws_acc[(bh * a.max_parts + part) * D + e] = A;
        }
    }
    if (tid < G) {
        const size_t bh = bh0 + tid;
        const float tot = red_tot[tid];
        const float M = red_M[tid];
        if (single) {
            if (a.lse_out) a.lse_out[bh] = tot > 0.f ? (M + log2f(tot)) * kLn2 : -INFINITY;
        } else {
            a.ws_m[bh * a.max_parts + part] = M;
            a.ws_l[bh * a.max_parts + part] = tot;
        }
    }
}

// One warp per (sequence, query head) split over more than one partition:
//   M = max_i m_i,  out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const DecodeArgs a) {
    constexpr int E = D / 32;
    const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) / 32);
    const int lane = threadIdx.x % 32;
    const int H = a.n_q_heads;
    if (warp >= a.num_seqs * H) return;
    const int b = warp / H;
    const int L = checked_len(a, b, false);
    const int P = a.partition_tokens;
    const int n_parts = (L + P - 1) / P;
    if (n_parts <= 1) return;
    const size_t bh = static_cast<size_t>(warp);
    const float *pm = a.ws_m + bh * a.max_parts;
    const float *pl = a.ws_l + bh * a.max_parts;

    float M = -INFINITY;
    for (int i = lane; i < n_parts; i += 32) M = fmaxf(M, pm[i]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    __half *out = static_cast<__half *>(a.out) + bh * D + lane * E;
    if (M == -INFINITY) {
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] = __float2half_rn(0.f);
        if (lane == 0 && a.lse_out) a.lse_out[bh] = -INFINITY;
        return;
    }
    float tot = 0.f;
    for (int i = lane; i < n_parts; i += 32) tot = fmaf(exp2f(pm[i] - M), pl[i], tot);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);

    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    for (int i = 0; i < n_parts; ++i) {
        const float w = exp2f(pm[i] - M);
        const float *src = a.ws_acc + (bh * a.max_parts + i) * D + lane * E;
        if constexpr (E == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src);
            o[0] = fmaf(w, v.x, o[0]);
            o[1] = fmaf(w, v.y, o[1]);
            o[2] = fmaf(w, v.z, o[2]);
            o[3] = fmaf(w, v.w, o[3]);
        } else {
            const float2 v = *reinterpret_cast<const float2 *>(src);
            o[0] = fmaf(w, v.x, o[0]);
            o[1] = fmaf(w, v.y, o[1]);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = __float2half_rn(o[e] / tot);
    if (lane == 0 && a.lse_out) a.lse_out[bh] = (M + log2f(tot)) * kLn2;
}

template <int D, int G>
cudaError_t launch_simt_t(const DecodeArgs &a, cudaStream_t stream) {
    using C = Cfg<D, G>;
    const int ids = (a.partition_tokens / a.block_size + 3) / 4 * 4;
    const size_t smem = C::UNION_BYTES + static_cast<size_t>(ids) * 4;
    auto kern = decode_partition_kernel<D, G>;
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(a.num_seqs, a.n_kv_heads, a.max_parts);
    kern<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_simt(const DecodeArgs &a, cudaStream_t stream) {
    const int g = a.n_q_heads / a.n_kv_heads;
#define PKV_CASE(D_, G_) \
    if (a.head_dim == D_ && g == G_) return launch_simt_t<D_, G_>(a, stream);
    PKV_CASE(128, 1)
    PKV_CASE(128, 2)
    PKV_CASE(128, 4)
    PKV_CASE(128, 8)
    PKV_CASE(64, 1)
    PKV_CASE(64, 2)
    PKV_CASE(64, 4)
    PKV_CASE(64, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge(const DecodeArgs &a, cudaStream_t stream) {
    const long long warps = static_cast<long long>(a.num_seqs) * a.n_q_heads;
    const int blocks = static_cast<int>((warps * 32 + 255) / 256);
    if (a.head_dim == 128)
        lse_merge_kernel<128><<<blocks, 256, 0, stream>>>(a);
    else
        lse_merge_kernel<64><<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

// Kernel choice: the tensor-core kernel whenever it applies (block size a
// multiple of 16); PKV_DECODE_KERNEL=simt or =mma in the environment forces
// one of the partition-grid kernels (read once per process).
int kernel_override() {
    static std::once_flag once;
    static int mode = 0;
    std::call_once(once, [] {
        const char *e = std::getenv("PKV_DECODE_KERNEL");
        if (e && std::strcmp(e, "simt") == 0) mode = 1;
        if (e && std::strcmp(e, "mma") == 0) mode = 2;
        if (e && std::strcmp(e, "warp") == 0) mode = 3;
        if (e && std::strcmp(e, "pipe") == 0) mode = 4;
    });
    return mode;
}

int test_wait_polls() {
    const char *e = std::getenv("PKV_TEST_WAIT_POLLS");
    if (!e || !*e) return -1;
    const int v = std::atoi(e);
    return v < 0 ? -1 : v;
}

bool decode_supported(int head_dim, int group) {
    return (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    const int mode = kernel_override();
    const bool mma_ok = decode_mma_supported(a);
    if (mode == 2 && !mma_ok) return cudaErrorInvalidValue;
    const cudaError_t e =
        (mma_ok && mode != 1) ? launch_decode_mma(a, stream) : launch_simt(a, stream);
    if (e != cudaSuccess || a.max_parts <= 1) return e;
    return launch_merge(a, stream);
}

WorkspaceLayout workspace_layout(int num_seqs, int n_q_heads, int head_dim, int max_parts) {
    WorkspaceLayout w{};
    const size_t rows = static_cast<size_t>(num_seqs) * n_q_heads * max_parts;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    w.acc_offset = 0;
    w.m_offset = up(rows * head_dim * sizeof(float));
    w.l_offset = w.m_offset + up(rows * sizeof(float));
    w.total = w.l_offset + up(rows * sizeof(float));
    return w;
}

}  // namespace pkv
