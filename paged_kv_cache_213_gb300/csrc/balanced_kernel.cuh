// balanced_kernel.cuh -- paged attention with the work split evenly over
// warps: the kernel of the default tensor-core path, included by
// decode_balanced.cu (one query token per sequence) and
// decode_balanced_multi.cu (several causal query tokens per sequence).
//
// The work of one call is the list of (KV head j, sequence b, 16-token tile t)
// units, ordered j, then b, then t: T units in all.  The W warps of the grid
// (4 or 8 per CTA, the grid sized to fill every SM once) take consecutive
// ranges of U = max(4, ceil(T / W)) units each, so every working warp moves the
// same number of K/V bytes whatever the mix of context lengths.  A warp streams its range
// through its own ring of TMA-loaded tiles, carrying the online-softmax state
// of the current (b, j) "segment".  A segment that ends inside the range is
// written out directly.  A segment cut by range boundaries leaves one partial
// result (m, l, acc) per warp; each such warp then bumps the segment's arrival
// counter, and the warp that arrives last merges all partials by log-sum-exp,
// writes the output and resets the counter to zero -- there is no second
// kernel.  The counters live at the start of the caller's workspace, which
// must therefore be zero-filled before its first use; every call leaves them
// zero again, and an arrival that proves a counter did not start at zero
// flags PKV_ERRBIT_WORKSPACE.
//
// The 16 rows of a segment's mma.m16n8k16 are its query rows.  For decode
// (MT = false) they are the G query heads of KV head j (rows past G are
// zero).  For multi-token attention (MT = true) they are the (query token i,
// head h) pairs R = i * G + h of the sequence's n_b <= 16 / G new tokens;
// token i sits at position L_b - n_b + i and sees the tokens up to it, so
// every row carries its own causal limit, and the last token, which sees all
// L_b tokens, sets the segment's tile count as in decode.
//
// Method: "Distributed LLM Inference Serving Platform", sections 2-3 (block
// table gather) and 5.1 (attention over every block of a sequence's table),
// GQA from section 1; online softmax and the log-sum-exp combination of
// partial results from FlashAttention-2 (section 14 references).  The causal
// rows follow "Roadmap: vLLM-style serving features for TornadoVM batched
// decode", Deferred list (batch-prefill verify of draft tokens, multi-token
// chunked prefill).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <map>
#include <mutex>

#include "mma_tile.cuh"
#include "mma_tile_multi.cuh"
#include "pagedkv.h"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"
#include "shared_prefix.cuh"
#include "tile_cursor.cuh"

namespace pkv {
namespace {

// Warps per CTA (each an independent worker): 4, three CTAs per SM; or 8,
// one CTA per SM, for batches of few long segments (balanced_plan).
constexpr int kWSmall = 4;
constexpr int kWLarge = 8;
// Ring stages per warp: fp16 tiles with 4-warp CTAs (three per SM) and with
// 8-warp CTAs (one per SM), E4M3 tiles, and the multi-token kernel.
#ifndef PKV_BAL_STAGES
#define PKV_BAL_STAGES 2
#endif
#ifndef PKV_BAL_STAGES_LARGE
#define PKV_BAL_STAGES_LARGE 2
#endif
#ifndef PKV_BAL_STAGES_F8
#define PKV_BAL_STAGES_F8 2
#endif
#ifndef PKV_BAL_STAGES_MT
#define PKV_BAL_STAGES_MT 2
#endif
constexpr int kMaxSeqsBalanced = 2048;
constexpr int kMaxSeqsMultiBalanced = 1024;  // multi-token: larger Q slots
constexpr int kMaxWorkers = kBalancedMaxWorkers;  // size of the counter region
constexpr int kMinUnits = 4;        // fewest units a working warp takes
// In the suffix pass of the prefix-aware call the private parts are short
// (forked completions: a block or two), and each output waits for the shared
// pass; one short segment per warp spreads those fold-ins over more warps.
constexpr int kMinUnitsSuffix = 2;
// With eight warps per CTA (long segments, most of them cut), the split
// counts every segment start as this many extra units.  A warp whose range
// holds a segment's first tile is the one that releases the cut piece before
// it, mid-loop (a GPU-scope release while its loads are in flight), and it
// loads the segment's Q rows, so it gets less to stream.  Measured on GB300
// (back to back, LLaMA-3-8B-shaped layer / 32k contexts): 1 unit 32.1 /
// 162.7 us, 2 units 31.6 / 161.4, 3 units 31.5 / 162.3, 4 units 31.4 / 160.0.
constexpr int kCutUnits = 4;
constexpr float kLn2b = 0.69314718055994531f;

template <int D, int G, bool F8, int kW, bool MT>
struct BalCfg : MmaCfg<D> {
    static constexpr int STAGES = MT ? PKV_BAL_STAGES_MT
                                     : (F8 ? PKV_BAL_STAGES_F8
                                           : (kW == kWLarge ? PKV_BAL_STAGES_LARGE : PKV_BAL_STAGES));
    static constexpr int ROWS = MT ? 16 : G;      // query rows of a segment
    static constexpr int Q_BYTES = ROWS * D * 2;  // one Q slot
    // one tile of one cache in the ring: fp16 (TMA boxes) or E4M3 bytes
    static constexpr int KV_BYTES = F8 ? kMmaTile * D : MmaCfg<D>::TILE_BYTES;
    static constexpr int SLOT_BYTES = 2 * KV_BYTES;  // K tile, V tile
    static constexpr int WARP_BYTES = STAGES * SLOT_BYTES;  // multiple of 1024
    // Multi-token: a warp's Q slots follow its ring, so that the whole region
    // (a multiple of 1024 bytes) can stage partial records in a merge.
    static constexpr int REGION_BYTES = WARP_BYTES + (MT ? STAGES * Q_BYTES : 0);
    static constexpr int PIPE_BYTES = kW * REGION_BYTES;
    static constexpr int QS_BYTES = MT ? 0 : kW * STAGES * Q_BYTES;
};

// Workspace: int counters[kMaxWorkers] at offset 0 (whatever the plan, so
// that a workspace reused by another plan still starts zeroed), then one
// record per (worker, slot 0/1): acc [rows][D], m [rows], l [rows] (fp32),
// padded to a multiple of 16 bytes so that a record is one bulk copy.
__host__ __device__ constexpr size_t rec_bytes(int rows, int D) {
    return (static_cast<size_t>(rows) * (D + 2) * 4 + 15) / 16 * 16;
}
constexpr size_t kRecBase = kBalancedCounterBytes;
__host__ __device__ inline size_t bal_ws_bytes(int workers, int rows, int D) {
    return kRecBase + static_cast<size_t>(workers) * 2 * rec_bytes(rows, D);
}

__device__ __forceinline__ int clamped_len(const DecodeArgs &a, int b, bool flag) {
    const int L = a.context_lens[b];
    const long long cap_ll = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    const int cap = static_cast<int>(cap_ll < a.max_context_len ? cap_ll : a.max_context_len);
    if (L < 0 || L > cap) {
        if (flag) flag_error(a.err, PKV_ERRBIT_CONTEXT);
        return L < 0 ? 0 : cap;
    }
    return L;
}

// Multi-token: the length that sets sequence b's tiles, or 0 (no work) when
// it has no query rows or its rows are malformed (then flagged and left
// unwritten): n_b > L_b, n_b > max_q_len, n_b * G > 16, rows outside
// [0, total_q), or L_b outside [0, min(table capacity, max_context_len)].
template <int G>
__device__ __forceinline__ int multi_len(const DecodeArgs &a, int b, bool flag) {
    const int L = a.context_lens[b];
    const int q0 = a.query_start[b];
    const int q1 = a.query_start[b + 1];
    const int n = q1 - q0;
    const long long cap_ll = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    const int cap = static_cast<int>(cap_ll < a.max_context_len ? cap_ll : a.max_context_len);
    if (L < 0 || L > cap || n < 0 || n > L || n > a.max_q_len || n * G > 16 || q0 < 0 ||
        q1 > a.total_q) {
        if (flag) flag_error(a.err, PKV_ERRBIT_CONTEXT);
        return 0;
    }
    return n == 0 ? 0 : L;
}

// Launch bounds: three 4-warp CTAs or one 8-warp CTA per SM, so that the
// 8-warp kernel may use the registers one CTA per SM leaves it (178 against
// the 150 the compiler picks otherwise, 13 % fewer instructions;
// LLaMA-3-8B-shaped layer, back to back with PKV_TABLES_READY: 32.4 -> 31.9 us).
template <int D, int G, bool F8, int kW, bool MT>
__global__ void __launch_bounds__(kW * 32, kW == kWSmall ? 3 : 1)
    decode_balanced_kernel(const __grid_constant__ DecodeArgs a,
                           const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const int workers) {
    using C = BalCfg<D, G, F8, kW, MT>;
    constexpr int R = C::ROWS;
    constexpr int kS = C::STAGES;
    constexpr int kThreadsB = kW * 32;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kW][kS];
    __shared__ uint64_t merge_bar[kW];
    __shared__ int s_ok[kW][kS];
    __shared__ int s_scan[kW];
    __shared__ int s_scan_nz[kW];
    const uint32_t raw_s = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
    unsigned char *qslots = smem + C::PIPE_BYTES;
    int *s_pre = reinterpret_cast<int *>(qslots + C::QS_BYTES);  // [B + 1]
    int *s_len = s_pre + a.num_seqs + 1;                          // [B]
    int *s_skip = s_len + a.num_seqs;  // [B] tiles left to the shared-prefix pass
    int *s_nz = s_skip + a.num_seqs;   // [B + 1] sequences with tiles before b
    int *s_qs = s_nz + a.num_seqs + 1; // multi-token: [B + 1] query_start

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int B = a.num_seqs;
    const int H = a.n_q_heads;
    const int Hk = a.n_kv_heads;
    const int bs = a.block_size;
    char *ws = reinterpret_cast<char *>(a.ws_acc);
    int *counters = reinterpret_cast<int *>(ws);
    // barriers and tensor-map prefetch first: they overlap the loads below
    if (tid == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        for (int w = 0; w < kW; ++w) {
            for (int s = 0; s < kS; ++s) mbar_init(&full_bar[w][s], 1);
            mbar_init(&merge_bar[w], 1);
        }
        fence_barrier_init();
    }
    // The context lengths and block tables into L2, spread over the CTAs,
    // while the kernel before may still be running: a prefetch cannot read
    // stale data (L2 is where the GPU's memory is coherent), so it may come
    // before the dependency wait; the loads after it then hit L2.
    if (warp == 0) {
        const size_t len_lines = (static_cast<size_t>(B) * sizeof(int32_t) + 127) / 128;
        const size_t tab_lines =
            (static_cast<size_t>(B) * a.max_blocks_per_seq * sizeof(int32_t) + 127) / 128;
        for (size_t ln = static_cast<size_t>(blockIdx.x) * 32 + lane; ln < len_lines + tab_lines;
             ln += static_cast<size_t>(gridDim.x) * 32)
            prefetch_l2(ln < len_lines
                            ? reinterpret_cast<const char *>(a.context_lens) + ln * 128
                            : reinterpret_cast<const char *>(a.block_tables) + (ln - len_lines) * 128);
    }
    // the previous kernel in the stream (e.g. the append) is done; after the
    // shared-prefix pass, only the reads of its partials have to wait.  Once
    // this grid has waited, everything before it in the stream is complete,
    // so the next kernel may be scheduled as this grid's CTAs retire (it too
    // waits for this grid before reading what this grid writes).
    if (!a.defer_dep_wait) {
        grid_dependency_wait();
        allow_dependent_launch();
    } else if (a.defer_dep_wait == 1) {
        // After the shared-prefix pass, which let this grid launch only after
        // its own dependency wait: everything before that pass is complete,
        // and what this grid writes (out, lse, workspace) a dependent reads
        // only after its own wait.  So the next kernel may be scheduled now,
        // as this grid's idle CTAs retire (70B-shaped batch, back to back:
        // fp16 58.2 -> 57.9 us, E4M3 78.3 -> 73.5 us).
        allow_dependent_launch();
    }

    // --- tile prefix over sequences: contiguous chunk per thread, then a scan
    const int chunk = (B + kThreadsB - 1) / kThreadsB;
    const int c0 = min(B, tid * chunk);
    const int c1 = min(B, c0 + chunk);
    for (int b = c0; b < c1; ++b) {
        if constexpr (MT) {
            s_len[b] = multi_len<G>(a, b, blockIdx.x == 0);
            s_qs[b] = a.query_start[b];
        } else {
            s_len[b] = clamped_len(a, b, blockIdx.x == 0);
            // fused append: a token of an empty sequence has no newest position
            if (!F8 && a.fuse_append && blockIdx.x == 0 && s_len[b] == 0 &&
                a.append_slots[b] >= 0)
                flag_error(a.err, PKV_ERRBIT_APPEND);
        }
        s_skip[b] = 0;
    }
    if constexpr (MT) {
        if (tid == kThreadsB - 1) s_qs[B] = a.query_start[B];
    }
    if (!MT && a.num_groups > 0) {
        __syncthreads();
        // members of a prefix-shared group leave the shared tiles to that pass
        for (int gi = tid; gi < a.num_groups; gi += kThreadsB) {
            const int f = max(0, min(B, a.group_offsets[gi]));
            const int e = max(f, min(B, a.group_offsets[gi + 1]));
            if (e - f < 2) continue;
            int mn = INT_MAX;
            for (int b = f; b < e; ++b) mn = min(mn, s_len[b]);
            const int st = shared_tiles(a, gi, mn);
            for (int b = f; b < e; ++b) s_skip[b] = st;
        }
        __syncthreads();
    }
    // tiles per sequence and sequences with tiles, both prefix-summed
    auto tiles_of = [&](int b) { return (s_len[b] + kMmaTile - 1) / kMmaTile - s_skip[b]; };
    int local = 0, local_nz = 0;
    for (int b = c0; b < c1; ++b) {
        const int tb = tiles_of(b);
        local += tb;
        local_nz += tb > 0;
    }
    int incl = local, incl_nz = local_nz;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        const int v_nz = __shfl_up_sync(0xffffffffu, incl_nz, off);
        if (lane >= off) {
            incl += v;
            incl_nz += v_nz;
        }
    }
    if (lane == 31) {
        s_scan[warp] = incl;
        s_scan_nz[warp] = incl_nz;
    }
    __syncthreads();
    int base = 0, base_nz = 0;
    for (int w = 0; w < warp; ++w) {
        base += s_scan[w];
        base_nz += s_scan_nz[w];
    }
    int run = base + incl - local, run_nz = base_nz + incl_nz - local_nz;
    for (int b = c0; b < c1; ++b) {
        s_pre[b] = run;
        s_nz[b] = run_nz;
        const int tb = tiles_of(b);
        run += tb;
        run_nz += tb > 0;
    }
    if (tid == kThreadsB - 1) {
        s_pre[B] = base + incl;
        s_nz[B] = base_nz + incl_nz;
    }
    __syncthreads();

    // Sequences without private tiles (sequences spread over the CTAs): empty
    // ones get out = 0, lse = -inf; the others are the shared pass's result
    // (E4M3: its partial sums are in the tile math's register order, in units
    // of v_scale).  (Multi-token: a sequence without tiles has no query rows,
    // or is flagged.)
    for (int b = blockIdx.x; !MT && b < B; b += gridDim.x) {
        if (s_pre[b + 1] != s_pre[b]) continue;
        grid_dependency_wait();  // the shared pass's partials are complete
        __half *ob = static_cast<__half *>(a.out) + static_cast<size_t>(b) * H * D;
        for (int i = tid; i < H * D; i += kThreadsB) {
            const int h = i / D;
            float M = -INFINITY, Ls = 0.f, A = 0.f;
            if (s_skip[b] > 0) {
                const size_t r0 = (static_cast<size_t>(b) * H + h) * a.sh_parts;
                for (int pp = 0; pp < a.sh_parts; ++pp) M = fmaxf(M, a.sh_m[r0 + pp]);
                for (int pp = 0; pp < a.sh_parts && M != -INFINITY; ++pp) {
                    const float mp = a.sh_m[r0 + pp];
                    if (mp == -INFINITY) continue;
                    const float wgt = exp2f(mp - M);
                    Ls = fmaf(wgt, a.sh_l[r0 + pp], Ls);
                    A = fmaf(wgt, a.sh_acc[(r0 + pp) * D + (F8 ? f8_acc_index(i % D) : i % D)], A);
                }
            }
            ob[i] = __float2half_rn(Ls > 0.f ? A * a.v_scale / Ls : 0.f);
            if (a.lse_out && i % D == 0)
                a.lse_out[static_cast<size_t>(b) * H + h] = Ls > 0.f ? (M + log2f(Ls)) * kLn2b : -INFINITY;
        }
    }

    // --- this warp's range of units.  The split is even over "virtual"
    // units: each segment (b, j) with tiles is kCut units, then its tiles.
    // Unit x of segment number s (in j, b order) sits at virtual position
    // x + kCut * (s + 1); warp w takes the units whose positions fall in
    // [w * U, (w + 1) * U).  kCut = 0: the plain even split.
    constexpr int kCut = kW == kWLarge ? kCutUnits : 0;
    const int w = blockIdx.x * kW + warp;
    const int TB = s_pre[B];
    const int T = Hk * TB;
    const int NZ = s_nz[B];
    const long long VTB = TB + static_cast<long long>(kCut) * NZ;
    const long long VT = Hk * VTB;
    // at least kMinUnits units per warp: short segments then stay whole
    const int U = static_cast<int>(max(static_cast<long long>(a.num_groups > 0 ? kMinUnitsSuffix
                                                                               : kMinUnits),
                                       (VT + workers - 1) / workers));
    auto real_at = [&](long long v) -> int {  // the first unit at or after position v
        if (v >= VT) return T;
        const int j = static_cast<int>(v / VTB);
        const int r = static_cast<int>(v - j * VTB);
        int lo = 0, hi = B - 1;  // the last sequence whose segment starts at or before r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pre[mid] + kCut * s_nz[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const int off = r - (s_pre[lo] + kCut * s_nz[lo]);
        const int x0 = j * TB + s_pre[lo];
        return off < kCut ? x0 : x0 + off - kCut;
    };
    // virtual position of the first unit of segment (b, j), and of the unit before it
    auto vpos0 = [&](int b, int j) {
        return j * TB + s_pre[b] + kCut * (j * NZ + s_nz[b] + 1);
    };
    const int w0 = real_at(static_cast<long long>(w) * U);
    const int n = real_at(static_cast<long long>(w + 1) * U) - w0;
    if (n <= 0) return;  // no CTA-wide barriers below

    unsigned char *my_pipe = smem + warp * C::REGION_BYTES;
    unsigned char *my_q = MT ? my_pipe + C::WARP_BYTES : qslots + warp * kS * C::Q_BYTES;
    Cursor pc = locate(w0, s_pre, B);  // producer cursor
    Cursor cc = pc;                        // consumer cursor
    int prev_seg_p = -1;

    // Block ids of the range, 32 tiles at a time: lane i holds the id of tile
    // 32c + i, for the chunk c being issued (ids_cur) and the next (ids_next),
    // so no table load sits on the issue path.
    auto load_ids = [&](int chunk_no) -> int {
        const int kk = chunk_no * 32 + lane;
        if (kk >= n) return -1;
        const Cursor c = locate(w0 + kk, s_pre, B);
        return a.block_tables[static_cast<size_t>(c.b) * a.max_blocks_per_seq +
                              ((c.t + s_skip[c.b]) * kMmaTile) / bs];
    };
    int ids_cur = load_ids(0);
    int ids_next = load_ids(1);

    // Fused append (fp16 decode only): per ring slot, this lane's 16-byte
    // piece of the newest token's K row (lanes < D/8) or V row (the next D/8
    // lanes), its slot and the tile's block id, fetched when a segment's last
    // tile is issued and used when that tile is consumed.
    constexpr bool kFuse = !MT && !F8;
    constexpr int kU8 = D / 8;  // 16-byte pieces per row
    uint4 app_piece[kS];
    long long app_slot[kS];
    int app_id[kS];
#pragma unroll
    for (int s = 0; s < kS; ++s) {
        app_piece[s] = make_uint4(0u, 0u, 0u, 0u);
        app_slot[s] = -1;
        app_id[s] = -1;
    }
    auto is_last_tile = [&](const Cursor &c) { return c.t == s_pre[c.b + 1] - s_pre[c.b] - 1; };

    // All lanes call (the cursor bookkeeping is warp-uniform); lane 0 issues.
    auto issue = [&](int k) {
        const int slot = k % kS;
        const int seg = pc.j * B + pc.b;
        const bool newseg = seg != prev_seg_p;
        prev_seg_p = seg;
        if (k > 0 && (k & 31) == 0) {
            ids_cur = ids_next;
            ids_next = load_ids((k >> 5) + 1);
        }
        const int id = __shfl_sync(0xffffffffu, ids_cur, k & 31);
        if (kFuse && a.fuse_append && is_last_tile(pc)) {
            const size_t row = static_cast<size_t>(pc.b) * Hk + pc.j;
            uint4 piece = make_uint4(0u, 0u, 0u, 0u);
            if (lane < 2 * kU8)
                piece = __ldg(static_cast<const uint4 *>(lane < kU8 ? a.append_k : a.append_v) +
                              row * kU8 + (lane % kU8));
            const long long sl = a.append_slots[pc.b];
#pragma unroll
            for (int s = 0; s < kS; ++s)
                if (s == slot) {
                    app_piece[s] = piece;
                    app_slot[s] = sl;
                    app_id[s] = id;
                }
        }
        if (lane == 0) {
            uint64_t *bar = &full_bar[warp][slot];
            const int tok0 = (pc.t + s_skip[pc.b]) * kMmaTile;
            const bool ok = id >= 0 && id < a.num_blocks;
            if (!ok) flag_error(a.err, PKV_ERRBIT_BLOCK_ID);
            s_ok[warp][slot] = ok;
            // the segment's query rows: the G heads, or G heads of each query token
            const int qn = MT ? s_qs[pc.b + 1] - s_qs[pc.b] : 1;
            const uint32_t bytes =
                (ok ? 2 * C::KV_BYTES : 0) + (newseg ? static_cast<uint32_t>(qn) * G * D * 2 : 0);
            mbar_arrive_expect_tx(bar, bytes);
            if (ok) {
                unsigned char *kdst = my_pipe + slot * C::SLOT_BYTES;
                unsigned char *vdst = kdst + C::KV_BYTES;
                const int row = (id * Hk + pc.j) * bs + (tok0 % bs);
                if constexpr (F8) {  // one swizzled box each, widened by the tile math
                    tma_load_2d(kdst, &tmap_k, 0, row, bar);
                    tma_load_2d(vdst, &tmap_v, 0, row, bar);
                } else {
#pragma unroll
                    for (int bx = 0; bx < C::BOXES; ++bx) {
                        tma_load_2d(kdst + bx * C::BOX_BYTES, &tmap_k, bx * 64, row, bar);
                        tma_load_2d(vdst + bx * C::BOX_BYTES, &tmap_v, bx * 64, row, bar);
                    }
                }
            }
            if (newseg) {
                const size_t q_row0 = MT ? static_cast<size_t>(s_qs[pc.b]) : static_cast<size_t>(pc.b);
                for (int i = 0; i < qn; ++i)  // row R = i * G + h of the slot
                    bulk_copy_g2s(my_q + slot * C::Q_BYTES + i * G * D * 2,
                                  static_cast<const __half *>(a.q) +
                                      ((q_row0 + i) * H + static_cast<size_t>(pc.j) * G) * D,
                                  G * D * 2, bar);
            }
        }
        advance(pc, s_pre, B);
    };

    if (a.defer_dep_wait == 2) {  // the append has written the caches
        grid_dependency_wait();
        allow_dependent_launch();
    }
    const int pro = n < kS ? n : kS;
    for (int k = 0; k < pro; ++k) issue(k);
    int issued = pro;

    // Running state.  Decode: row g (head g < G) in o[][0..1], m_run, l_run.
    // Multi-token: row g in o[][0..1], m_run, l_run and row g + 8 in
    // o[][2..3], m_hi, l_hi, each with its causal limit (exclusive, in tokens).
    float o[C::NB_D][4];
    uint32_t qa[C::NP][4];
    uint32_t qh[C::NP][4];
    float m_run = -INFINITY, l_run = 0.f, m_hi = -INFINITY, l_hi = 0.f;
    int lim_lo = 0, lim_hi = 0;
    int cur_seg = -1, pb = 0, pj = 0, piece_t0 = 0, last_t = 0, piece_no = 0;

    constexpr size_t REC = rec_bytes(R, D);
    auto rec = [&](int wk, int slot) { return ws + kRecBase + (static_cast<size_t>(wk) * 2 + slot) * REC; };
    const int gg = g < G ? g : 0;

    // Output row of head gg of segment (b, j): o / l in fp16, lse.
    auto write_out = [&](int b, int j, float fm, float fl) {
        if (g >= G) return;
        const size_t bh = static_cast<size_t>(b) * H + static_cast<size_t>(j) * G + g;
        if (s_skip[b] > 0) {  // fold in the shared-prefix partial states (same register order)
            grid_dependency_wait();  // complete and visible once the shared pass is done
            const size_t r0 = bh * a.sh_parts;
            float M = fm;
#pragma unroll 4
            for (int pp = 0; pp < a.sh_parts; ++pp) M = fmaxf(M, a.sh_m[r0 + pp]);
            const float so = M == -INFINITY ? 0.f : exp2f(fm - M);  // 0: no private part
            fl *= so;
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb) {
                o[nb][0] *= so;
                o[nb][1] *= so;
            }
#pragma unroll 4
            for (int pp = 0; pp < a.sh_parts; ++pp) {
                const float mp = a.sh_m[r0 + pp];
                const float lp = a.sh_l[r0 + pp];
                const float2 *src = reinterpret_cast<const float2 *>(a.sh_acc + (r0 + pp) * D);
                float2 v[C::NB_D];
#pragma unroll
                for (int nb = 0; nb < C::NB_D; ++nb) v[nb] = src[nb * 4 + tq];
                if (mp == -INFINITY) continue;
                const float sn = exp2f(mp - M);
                fl = fmaf(lp, sn, fl);
#pragma unroll
                for (int nb = 0; nb < C::NB_D; ++nb) {
                    o[nb][0] = fmaf(v[nb].x, sn, o[nb][0]);
                    o[nb][1] = fmaf(v[nb].y, sn, o[nb][1]);
                }
            }
            fm = M;
        }
        const float inv = fl > 0.f ? a.v_scale / fl : 0.f;  // v_scale = 1 for fp16 caches
        if constexpr (F8) {  // columns 32c + 8tq .. + 7 (the E4M3 tile math's order)
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(a.out) + bh * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
                dst[4 * c + tq] = make_uint4(
                    pack_half2(o[4 * c][0] * inv, o[4 * c + 1][0] * inv),
                    pack_half2(o[4 * c + 2][0] * inv, o[4 * c + 3][0] * inv),
                    pack_half2(o[4 * c][1] * inv, o[4 * c + 1][1] * inv),
                    pack_half2(o[4 * c + 2][1] * inv, o[4 * c + 3][1] * inv));
        } else {
            __half2 *dst = reinterpret_cast<__half2 *>(static_cast<__half *>(a.out) + bh * D);
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb)
                dst[nb * 4 + tq] = __floats2half2_rn(o[nb][0] * inv, o[nb][1] * inv);
        }
        if (tq == 0 && a.lse_out) a.lse_out[bh] = fl > 0.f ? (fm + log2f(fl)) * kLn2b : -INFINITY;
    };

    // Multi-token: output rows g (o[][0..1]) and g + 8 (o[][2..3]) of segment
    // (b, j), those of them that are query rows: row R is query token R / G
    // of the sequence, head j * G + R % G.
    auto write_out_mt = [&](int b, int j, float fm, float fl, float fmh, float flh) {
        const int q0 = s_qs[b];
        const int rows = (s_qs[b + 1] - q0) * G;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = g + 8 * half;
            if (r >= rows) continue;
            const float m = half ? fmh : fm;
            const float l = half ? flh : fl;
            const size_t row = static_cast<size_t>(q0 + r / G) * H + static_cast<size_t>(j) * G + r % G;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __half2 *dst = reinterpret_cast<__half2 *>(static_cast<__half *>(a.out) + row * D);
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb)
                dst[nb * 4 + tq] = __floats2half2_rn(o[nb][2 * half] * inv, o[nb][2 * half + 1] * inv);
            if (tq == 0 && a.lse_out) a.lse_out[row] = l > 0.f ? (m + log2f(l)) * kLn2b : -INFINITY;
        }
    };

    // Cut segments this warp arrived last on, merged once its ring is idle.
    int pend_n = 0, pend_b[2], pend_j[2], pend_x0[2], pend_nt[2];

    // Writes the finished piece [piece_t0, last_t] of segment (pb, pj).
    auto flush = [&]() {
        float lt = l_run;
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        float lth = 0.f;
        if constexpr (MT) {
            lth = l_hi;
            lth += __shfl_xor_sync(0xffffffffu, lth, 1);
            lth += __shfl_xor_sync(0xffffffffu, lth, 2);
        }
        const int nt = s_pre[pb + 1] - s_pre[pb];
        if (piece_t0 == 0 && last_t == nt - 1) {  // the whole segment: write it out
            if constexpr (MT) write_out_mt(pb, pj, m_run, lt, m_hi, lth);
            else write_out(pb, pj, m_run, lt);
            ++piece_no;
            return;
        }
        // a cut segment: publish this piece as a record, then count the arrivals
        char *r = rec(w, piece_no == 0 ? 0 : 1);
        if (MT || g < G) {
            float2 *acc = reinterpret_cast<float2 *>(r) + static_cast<size_t>(g) * (D / 2);
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb) acc[nb * 4 + tq] = make_float2(o[nb][0], o[nb][1]);
            if (tq == 0) {
                reinterpret_cast<float *>(r)[R * D + g] = m_run;
                reinterpret_cast<float *>(r)[R * D + R + g] = lt;
            }
            if constexpr (MT) {  // row g + 8
                float2 *acch = acc + 8 * (D / 2);
#pragma unroll
                for (int nb = 0; nb < C::NB_D; ++nb) acch[nb * 4 + tq] = make_float2(o[nb][2], o[nb][3]);
                if (tq == 0) {
                    reinterpret_cast<float *>(r)[R * D + g + 8] = m_hi;
                    reinterpret_cast<float *>(r)[R * D + R + g + 8] = lth;
                }
            }
        }
        __syncwarp();  // the record's stores, all lanes, before lane 0's release
        const int x0 = pj * s_pre[B] + s_pre[pb];  // the segment's units [x0, x0 + nt)
        const int wf = vpos0(pb, pj) / U;          // the warps holding its pieces
        const int wl = (vpos0(pb, pj) + nt - 1) / U;
        // lane 1 counts: lane 0 issues the ring's TMA loads, and a release by
        // the lane that issued them could wait for them to land
        int old = 0;
        if (lane == 1) {
            old = atomic_add_acq_rel_gpu(&counters[wf], 1);
            if (counter_not_zeroed(old, wl - wf)) {
                flag_error(a.err, PKV_ERRBIT_WORKSPACE);
                atomic_exch_relaxed_gpu(&counters[wf], kCounterPoison);
            }
        }
        old = __shfl_sync(0xffffffffu, old, 1);
        __syncwarp();  // lane 1's acquire before lane 0's bulk copies of the records
        ++piece_no;
        if (old == wl - wf) {  // arrived last: merge later, when the ring is idle
            pend_b[pend_n] = pb;
            pend_j[pend_n] = pj;
            pend_x0[pend_n] = x0;
            pend_nt[pend_n] = nt;
            ++pend_n;
        }
    };

    // Merge all records of a cut segment: bulk-copy them into this warp's
    // (idle) region, combine by log-sum-exp, write the output, reset the counter.
    uint32_t merge_phase = 0;
    auto merge = [&](int b, int j, int x0, int nt) -> bool {
        // the acquiring atomic (lane 0) made the other warps' records visible;
        // order them before the bulk copies (async proxy) that read them
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const int v0 = vpos0(b, j);
        const int wf = v0 / U;
        const int wl = (v0 + nt - 1) / U;
        // the piece in warp wf is its first iff the unit before x0 (at
        // position v0 - kCut - 1) lies before warp wf's positions
        const bool wf_starts_here = x0 == 0 || static_cast<long long>(wf) * U > v0 - kCut - 1;
        constexpr int cap = static_cast<int>(C::REGION_BYTES / REC);
        static_assert(cap >= 1, "a warp's region must hold a merge record");
        float M = -INFINITY, Lsum = 0.f, Mh = -INFINITY, Lh = 0.f;
#pragma unroll
        for (int nb = 0; nb < C::NB_D; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
        for (int first = wf; first <= wl; first += cap) {
            const int cnt = min(cap, wl - first + 1);
            if (lane == 0) {
                mbar_arrive_expect_tx(&merge_bar[warp], static_cast<uint32_t>(cnt * REC));
                for (int i = 0; i < cnt; ++i) {
                    const int wk = first + i;
                    const int slot = (wk == wf && !wf_starts_here) ? 1 : 0;
                    bulk_copy_g2s(my_pipe + i * REC, rec(wk, slot), static_cast<uint32_t>(REC),
                                  &merge_bar[warp]);
                }
            }
            const bool ok = mbar_wait_bounded(&merge_bar[warp], merge_phase & 1);
            ++merge_phase;
            if (__any_sync(0xffffffffu, !ok)) return false;
            for (int i = 0; i < cnt; ++i) {
                const float *rf = reinterpret_cast<const float *>(my_pipe + i * REC);
#pragma unroll
                for (int half = 0; half < (MT ? 2 : 1); ++half) {
                    const int row = MT ? g + 8 * half : gg;
                    const float mi = rf[R * D + row];
                    if (mi == -INFINITY) continue;  // a piece of skipped blocks only
                    const float li = rf[R * D + R + row];
                    float &Mr = half ? Mh : M;
                    float &Lr = half ? Lh : Lsum;
                    const float Mn = fmaxf(Mr, mi);
                    const float so = exp2f(Mr - Mn);  // 0 while Mr = -inf
                    const float sn = exp2f(mi - Mn);
                    Lr = Lr * so + li * sn;
                    const float2 *acc = reinterpret_cast<const float2 *>(rf) + static_cast<size_t>(row) * (D / 2);
#pragma unroll
                    for (int nb = 0; nb < C::NB_D; ++nb) {
                        const float2 v = acc[nb * 4 + tq];
                        o[nb][2 * half] = o[nb][2 * half] * so + v.x * sn;
                        o[nb][2 * half + 1] = o[nb][2 * half + 1] * so + v.y * sn;
                    }
                    Mr = Mn;
                }
            }
            __syncwarp();  // before the next round overwrites the staged records
        }
        // ready for the next call: back from n to 0 (a poisoned count stays >= n)
        if (lane == 0) red_add_relaxed_gpu(&counters[wf], -(wl - wf + 1));
        if constexpr (MT) write_out_mt(b, j, M, Lsum, Mh, Lh);
        else write_out(b, j, M, Lsum);
        return true;
    };

    int k = 0;
    bool timed_out = false;
    for (; k < n; ++k) {
        const int slot = k % kS;
        const bool ok = (k == 0 && a.first_wait_polls >= 0)
                            ? mbar_wait_polls(&full_bar[warp][slot], 0, a.first_wait_polls)
                            : mbar_wait_bounded(&full_bar[warp][slot], (k / kS) & 1);
        if (__any_sync(0xffffffffu, !ok)) {
            timed_out = true;
            break;
        }
        const int seg = cc.j * B + cc.b;
        if (seg != cur_seg) {
            if (cur_seg >= 0) flush();
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
            const __half *qs = reinterpret_cast<const __half *>(my_q + slot * C::Q_BYTES);
            if constexpr (MT) {
                m_hi = -INFINITY;
                l_hi = 0.f;
                const int qn = s_qs[cc.b + 1] - s_qs[cc.b];
                const int Lb = s_len[cc.b];
                const bool has_lo = g < qn * G, has_hi = g + 8 < qn * G;
                lim_lo = has_lo ? Lb - qn + g / G + 1 : 0;
                lim_hi = has_hi ? Lb - qn + (g + 8) / G + 1 : 0;
                load_q_frag<D>(qa, qs + g * D, has_lo, tq);
                load_q_frag<D>(qh, qs + (g + 8) * D, has_hi, tq);
            } else {
                load_q_frag<D>(qa, qs + (g < G ? g : 0) * D, g < G, tq);
            }
            cur_seg = seg;
            pb = cc.b;
            pj = cc.j;
            piece_t0 = cc.t;
        }
        last_t = cc.t;
        unsigned char *ks = my_pipe + slot * C::SLOT_BYTES;
        unsigned char *vs = ks + C::KV_BYTES;
        const int tok0 = (cc.t + s_skip[cc.b]) * kMmaTile;
        const int n_valid = s_ok[warp][slot] ? min(kMmaTile, s_len[cc.b] - tok0) : 0;
        if (kFuse && a.fuse_append && is_last_tile(cc)) {
            uint4 piece = make_uint4(0u, 0u, 0u, 0u);
            long long sl = -1;
            int tile_id = -1;
#pragma unroll
            for (int s = 0; s < kS; ++s)
                if (s == slot) {
                    piece = app_piece[s];
                    sl = app_slot[s];
                    tile_id = app_id[s];
                }
            if (sl >= 0) {
                const int L = s_len[cc.b];
                const long long newest = static_cast<long long>(tile_id) * bs + (L - 1) % bs;
                if (sl == newest && n_valid > 0) {
                    // row L - 1 of the staged tile takes the new token (the
                    // 128B-swizzled layout of the TMA boxes, 64 columns each)
                    const int r = L - 1 - tok0;
                    if (lane < 2 * kU8) {
                        const int u = lane % kU8;
                        unsigned char *tile = lane < kU8 ? ks : vs;
                        *reinterpret_cast<uint4 *>(tile + (u >> 3) * C::BOX_BYTES + swz(r, u & 7)) =
                            piece;
                    }
                    fence_proxy_async_smem();  // before a later TMA write of this slot
                    __syncwarp();
                } else if (sl != newest && lane == 0) {
                    flag_error(a.err, PKV_ERRBIT_APPEND);
                }
                // the append itself: the token's rows into its cache slot
                if (sl < a.num_blocks * bs) {
                    if (lane < 2 * kU8) {
                        const long long dst =
                            ((sl / bs) * Hk + cc.j) * static_cast<long long>(bs) + sl % bs;
                        uint4 *cache = static_cast<uint4 *>(const_cast<void *>(
                            lane < kU8 ? a.k_cache : a.v_cache));
                        cache[dst * kU8 + (lane % kU8)] = piece;
                    }
                } else if (lane == 0 && cc.j == 0) {
                    flag_error(a.err, PKV_ERRBIT_SLOT);
                }
            }
        }
        if constexpr (MT) {
            mma_tile_multi<D>(ks, vs, n_valid, min(n_valid, max(0, lim_lo - tok0)),
                              min(n_valid, max(0, lim_hi - tok0)), qa, qh, a.scale_log2, o,
                              m_run, l_run, m_hi, l_hi, lane);
        } else {
            mma_tile<D, F8>(ks, vs, n_valid, qa, a.scale_log2, o, m_run, l_run, lane);
        }
        __syncwarp();
        if (k + kS < n) {
            issue(k + kS);
            ++issued;
        }
        advance(cc, s_pre, B);
    }
    if (timed_out) {
        if (lane == 0) {
            flag_error(a.err, PKV_ERRBIT_TIMEOUT);
            for (int kk = k; kk < issued; ++kk)
                mbar_wait_bounded(&full_bar[warp][kk % kS], (kk / kS) & 1);
        }
        return;
    }
    if (cur_seg >= 0) flush();
    // every tile is consumed: the ring is free for the merges
    for (int i = 0; i < pend_n; ++i) {
        if (!merge(pend_b[i], pend_j[i], pend_x0[i], pend_nt[i])) {
            if (lane == 0) flag_error(a.err, PKV_ERRBIT_TIMEOUT);
            return;
        }
    }
}

template <int D, int G, bool F8, int kW, bool MT>
size_t bal_smem(int B) {
    using C = BalCfg<D, G, F8, kW, MT>;
    return 1024 + C::PIPE_BYTES + C::QS_BYTES + (4 * static_cast<size_t>(B) + 2) * 4 +
           (MT ? (static_cast<size_t>(B) + 1) * 4 : 0);
}

template <int D, int G, bool F8, int kW, bool MT>
int bal_ctas_per_sm(int B) {
    static std::mutex mu;
    static std::map<size_t, int> cache;
    const size_t smem = bal_smem<D, G, F8, kW, MT>(B);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(smem);
    if (it != cache.end()) return it->second;
    auto kern = decode_balanced_kernel<D, G, F8, kW, MT>;
    // the limit: what the most sequences need, within what a CTA may have
    // (a batch whose arrays do not fit then gets no plan)
    const int max_seqs = MT ? kMaxSeqsMultiBalanced : kMaxSeqsBalanced;
    int dev = 0, optin = 0;
    cudaFuncAttributes fa{};
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaFuncGetAttributes(&fa, kern) != cudaSuccess)
        return 0;
    size_t limit = bal_smem<D, G, F8, kW, MT>(max_seqs);
    const size_t room = static_cast<size_t>(optin) - fa.sharedSizeBytes;
    if (limit > room) limit = room;
    if (smem > limit) return 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(limit)) != cudaSuccess)
        return 0;
    // the grid is sized to fill every SM once: ask for the whole carve-out
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kW * 32, smem) != cudaSuccess)
        return 0;
    cache[smem] = n;
    return n;
}

template <int D, int G, bool F8, int kW, bool MT>
cudaError_t launch_bal_t(const DecodeArgs &a, const BalancedPlan &plan, const CUtensorMap &tk,
                         const CUtensorMap &tv, cudaStream_t stream) {
    auto kern = decode_balanced_kernel<D, G, F8, kW, MT>;
    if (bal_ctas_per_sm<D, G, F8, kW, MT>(a.num_seqs) <= 0) return cudaErrorInvalidConfiguration;
    return launch_pdl(kern, dim3(plan.ctas), dim3(kW * 32), bal_smem<D, G, F8, kW, MT>(a.num_seqs),
                      stream, a, tk, tv, plan.workers);
}

int sm_count_cached() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess)
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    });
    return n;
}

// Grid of a balanced plan: per_sm CTAs of `warps` warps on every SM, fewer
// when the work is small (at least two tiles per warp on average), within
// the counter region.  rows: query rows per segment record.
bool finish_bal_plan(int sms, int per_sm, int warps, int num_seqs, int n_kv_heads, int head_dim,
                     int rows, int max_len, BalancedPlan *plan) {
    if (per_sm <= 0) return false;
    // units must fit 32-bit arithmetic: Hk * B * (tiles per sequence + the
    // split's extra units per segment)
    const long long t_max = static_cast<long long>(n_kv_heads) * num_seqs *
                            ((static_cast<long long>(max_len) + kMmaTile - 1) / kMmaTile);
    if (t_max + static_cast<long long>(kCutUnits) * n_kv_heads * num_seqs >= (1LL << 31))
        return false;
    long long ctas = static_cast<long long>(sms) * per_sm;
    const long long need = (t_max + 2 * warps - 1) / (2 * warps);  // >= 2 tiles per warp on average
    if (need < ctas) ctas = need;
    if (ctas * warps > kMaxWorkers) ctas = kMaxWorkers / warps;
    if (ctas < 1) ctas = 1;
    plan->ctas = static_cast<int>(ctas);
    plan->warps = warps;
    plan->workers = plan->ctas * warps;
    plan->ws_bytes = bal_ws_bytes(plan->workers, rows, head_dim);
    plan->kind = 0;
    return true;
}

bool make_bal_maps(const DecodeArgs &a, CUtensorMap *tk, CUtensorMap *tv) {
    const long long rows = a.num_blocks * a.n_kv_heads * static_cast<long long>(a.block_size);
    return a.kv_fp8 ? (make_cache_map_e4m3(tk, a.k_cache, rows, a.head_dim) &&
                       make_cache_map_e4m3(tv, a.v_cache, rows, a.head_dim))
                    : (make_cache_map(tk, a.k_cache, rows, a.head_dim) &&
                       make_cache_map(tv, a.v_cache, rows, a.head_dim));
}

}  // namespace
}  // namespace pkv
