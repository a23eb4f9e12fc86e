// decode_mma.cu -- paged decode attention with the GQA query group on the
// tensor cores.
//
// One CTA per (sequence, KV head, partition), 4 warps.  Each warp owns every
// 4th 16-token tile of the partition and a private 2-stage ring in shared
// memory: its lane 0 loads the K and V tiles of a block with 2-D TMA copies
// (128-byte swizzle, so the fragment loads below are free of bank
// conflicts), and the warp computes
//   S = Q K^T     mma.m16n8k16, M = query heads of the group (padded to 16),
//                 N = 8 tokens, K = head_dim (16 per step)
//   online softmax on S in fp32 (exp2 domain), P rounded to fp16
//   O += P V      mma.m16n8k16, M = heads, N = 8 head_dim columns, K = 16 tokens
// The C fragment of S is exactly the A fragment of P, so P never leaves the
// registers.  The four warps' running states are merged through shared
// memory at the end, as in the CUDA-core kernel.
//
// Method: "Distributed LLM Inference Serving Platform", sections 2-3 (block
// table gather) and 5.1 (attention over all blocks of a sequence); GQA from
// section 1 of that page; online softmax and the partition split from
// FlashAttention-2 (its section 14 references).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"
#include "mma_tile.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kTile = kMmaTile;
constexpr int kWarps = 4;
constexpr int kStages = 2;  // per warp
constexpr int kThreadsMma = kWarps * 32;
constexpr float kLn2f = 0.69314718055994531f;

template <int D>
struct GridCfg : MmaCfg<D> {
    static constexpr int STAGE_BYTES = 2 * MmaCfg<D>::TILE_BYTES;  // K then V
    static constexpr int PIPE_BYTES = kWarps * kStages * STAGE_BYTES;
};

__device__ __forceinline__ int checked_len_mma(const DecodeArgs &a, int b, bool flag) {
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
__global__ void __launch_bounds__(kThreadsMma)
    decode_mma_kernel(const __grid_constant__ DecodeArgs a,
                      const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
    using C = GridCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kWarps][kStages];
    // 1024-byte aligned base: the 128-byte swizzle pattern repeats every 1 KiB
    const uint32_t raw_s = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
    int32_t *s_blk = reinterpret_cast<int32_t *>(smem + C::PIPE_BYTES);

    const int b = blockIdx.x;
    const int j = blockIdx.y;
    const int part = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;   // query head of the group (rows >= G are padding)
    const int tq = lane & 3;
    const int H = a.n_q_heads;
    const int Hk = a.n_kv_heads;
    const int bs = a.block_size;
    const int P = a.partition_tokens;

    const int L = checked_len_mma(a, b, j == 0 && part == 0);
    const int n_parts = (L + P - 1) / P;
    if (part >= (n_parts > 1 ? n_parts : 1)) return;
    const int t_begin = part * P;
    const int t_end = min(L, t_begin + P);
    const int n_tok = max(t_end - t_begin, 0);
    const int n_tiles = (n_tok + kTile - 1) / kTile;
    const int lb0 = t_begin / bs;
    const int n_blk = (n_tok + bs - 1) / bs;

    const int32_t *bt_row = a.block_tables + static_cast<size_t>(b) * a.max_blocks_per_seq;
    for (int i = tid; i < n_blk; i += kThreadsMma) {
        int32_t id = bt_row[lb0 + i];
        if (id < 0 || id >= a.num_blocks) {
            flag_error(a.err, PKV_ERRBIT_BLOCK_ID);
            id = -1;
        }
        s_blk[i] = id;
    }
    if (tid == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        for (int w = 0; w < kWarps; ++w)
            for (int s = 0; s < kStages; ++s) mbar_init(&full_bar[w][s], 1);
        fence_barrier_init();
    }

    // Q fragments (A operand of S = Q K^T).  Thread (g, tq) owns, per row,
    // the 16-byte pieces p = 0..NP-1 at column 64*(p/2) + 8*(2*tq + p%2):
    // MMA k-step 2p+sub uses words 2*sub (k = 2tq, 2tq+1) and 2*sub+1
    // (k = 2tq+8, 2tq+9) of piece p, for Q and K alike.
    uint32_t qa[C::NP][4];
    load_q_frag<D>(qa,
                   static_cast<const __half *>(a.q) +
                       (static_cast<size_t>(b) * H + static_cast<size_t>(j) * G + (g < G ? g : 0)) * D,
                   g < G, tq);
    __syncthreads();

    unsigned char *my_stages = smem + warp * kStages * C::STAGE_BYTES;
    // Lane 0 of the warp: start the TMA loads of tile i into stage slot.
    auto issue = [&](int i, int slot) {
        unsigned char *kdst = my_stages + slot * C::STAGE_BYTES;
        unsigned char *vdst = kdst + C::TILE_BYTES;
        const int tok0 = t_begin + i * kTile;
        const int id = s_blk[tok0 / bs - lb0];
        uint64_t *bar = &full_bar[warp][slot];
        if (id >= 0) {
            const int row = (id * Hk + j) * bs + (tok0 % bs);
            mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
#pragma unroll
            for (int bx = 0; bx < C::BOXES; ++bx) {
                tma_load_2d(kdst + bx * C::BOX_BYTES, &tmap_k, bx * 64, row, bar);
                tma_load_2d(vdst + bx * C::BOX_BYTES, &tmap_v, bx * 64, row, bar);
            }
        } else {
            mbar_arrive_expect_tx(bar, 0);
        }
    };

    float o[C::NB_D][4];
#pragma unroll
    for (int n = 0; n < C::NB_D; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run = -INFINITY;
    float l_run = 0.f;

    const int my_tiles = n_tiles > warp ? (n_tiles - warp + kWarps - 1) / kWarps : 0;
    if (lane == 0)
        for (int k = 0; k < kStages && k < my_tiles; ++k) issue(warp + k * kWarps, k);
    int issued = my_tiles < kStages ? my_tiles : kStages;

    int k = 0;
    bool timed_out = false;
    for (; k < my_tiles; ++k) {
        const int i = warp + k * kWarps;
        const int slot = k % kStages;
        const bool ok = mbar_wait_bounded(&full_bar[warp][slot], (k / kStages) & 1);
        if (__any_sync(0xffffffffu, !ok)) {  // the whole warp leaves together
            timed_out = true;
            break;
        }
        unsigned char *ks = my_stages + slot * C::STAGE_BYTES;
        unsigned char *vs = ks + C::TILE_BYTES;
        const int tok0 = t_begin + i * kTile;
        int n_valid = min(kTile, t_end - tok0);
        if (s_blk[tok0 / bs - lb0] < 0) n_valid = 0;
        mma_tile<D>(ks, vs, n_valid, qa, a.scale_log2, o, m_run, l_run, lane);
        __syncwarp();
        if (k + kStages < my_tiles) {
            if (lane == 0) issue(i + kStages * kWarps, slot);
            ++issued;
        }
    }
    if (timed_out && lane == 0) {
        flag_error(a.err, PKV_ERRBIT_TIMEOUT);
        for (int kk = k; kk < issued; ++kk)
            mbar_wait_bounded(&full_bar[warp][kk % kStages], (kk / kStages) & 1);
    }
    // per-head sum over the 4 threads that share head g
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    __syncthreads();

    // merge the four warps' states (log-sum-exp) through shared memory
    float *red_o = reinterpret_cast<float *>(smem);  // [kWarps][G][D]
    float *red_m = red_o + kWarps * G * D;           // [kWarps][G]
    float *red_l = red_m + kWarps * G;               // [kWarps][G]
    float *red_w = red_l + kWarps * G;               // [kWarps][G]
    float *red_tot = red_w + kWarps * G;             // [G]
    float *red_M = red_tot + G;                      // [G]
    if (g < G) {
#pragma unroll
        for (int n = 0; n < C::NB_D; ++n)
            *reinterpret_cast<float2 *>(red_o + (warp * G + g) * D + n * 8 + 2 * tq) =
                make_float2(o[n][0], o[n][1]);
        if (tq == 0) {
            red_m[warp * G + g] = m_run;
            red_l[warp * G + g] = l_run;
        }
    }
    __syncthreads();
    if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * G + h]);
        float tot = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            const float wt = (M == -INFINITY) ? 0.f : exp2f(red_m[w * G + h] - M);
            red_w[w * G + h] = wt;
            tot = fmaf(wt, red_l[w * G + h], tot);
        }
        red_tot[h] = tot;
        red_M[h] = M;
    }
    __syncthreads();

    const bool single = n_parts <= 1;
    const size_t bh0 = static_cast<size_t>(b) * H + static_cast<size_t>(j) * G;
    for (int oi = tid; oi < G * D; oi += kThreadsMma) {
        const int h = oi / D;
        const int e = oi % D;
        float A = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) A = fmaf(red_w[w * G + h], red_o[(w * G + h) * D + e], A);
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
            if (a.lse_out) a.lse_out[bh] = tot > 0.f ? (M + log2f(tot)) * kLn2f : -INFINITY;
        } else {
            a.ws_m[bh * a.max_parts + part] = M;
            a.ws_l[bh * a.max_parts + part] = tot;
        }
    }
}

template <int D, int G>
cudaError_t launch_mma_t(const DecodeArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                         cudaStream_t stream) {
    using C = GridCfg<D>;
    const int ids = (a.partition_tokens / a.block_size + 3) / 4 * 4;
    const size_t smem = 1024 + C::PIPE_BYTES + static_cast<size_t>(ids) * 4;
    auto kern = decode_mma_kernel<D, G>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        1024 + C::PIPE_BYTES + 2048 * 4);
    });
    if (attr_err != cudaSuccess) return attr_err;
    dim3 grid(a.num_seqs, a.n_kv_heads, a.max_parts);
    kern<<<grid, kThreadsMma, smem, stream>>>(a, tk, tv);
    return cudaGetLastError();
}

}  // namespace

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view [rows = num_blocks * n_kv_heads * block_size][head_dim] of a cache,
// boxes of 16 rows x 64 columns, 128-byte swizzle.
bool make_cache_map(CUtensorMap *m, const void *base, long long rows, int D) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[2] = {64, kTile};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_cache_map_e4m3(CUtensorMap *m, const void *base, long long rows, int D) {
    auto fn = encode_fn();
    if (!fn || (D != 64 && D != 128)) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(D)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(D), kTile};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool decode_mma_supported(const DecodeArgs &a) {
    const int g = a.n_q_heads / a.n_kv_heads;
    const long long rows = a.num_blocks * a.n_kv_heads * static_cast<long long>(a.block_size);
    return (a.head_dim == 64 || a.head_dim == 128) && (g == 1 || g == 2 || g == 4 || g == 8) &&
           a.block_size % kTile == 0 && rows < (1LL << 31);
}

cudaError_t launch_decode_mma(const DecodeArgs &a, cudaStream_t stream) {
    const long long rows = a.num_blocks * a.n_kv_heads * static_cast<long long>(a.block_size);
    CUtensorMap tk, tv;
    if (!make_cache_map(&tk, a.k_cache, rows, a.head_dim) ||
        !make_cache_map(&tv, a.v_cache, rows, a.head_dim))
        return cudaErrorNotSupported;
    const int g = a.n_q_heads / a.n_kv_heads;
#define PKV_MMA_CASE(D_, G_) \
    if (a.head_dim == D_ && g == G_) return launch_mma_t<D_, G_>(a, tk, tv, stream);
    PKV_MMA_CASE(128, 1)
    PKV_MMA_CASE(128, 2)
    PKV_MMA_CASE(128, 4)
    PKV_MMA_CASE(128, 8)
    PKV_MMA_CASE(64, 1)
    PKV_MMA_CASE(64, 2)
    PKV_MMA_CASE(64, 4)
    PKV_MMA_CASE(64, 8)
#undef PKV_MMA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
