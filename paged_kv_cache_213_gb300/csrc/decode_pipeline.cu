// decode_pipeline.cu -- paged decode attention for batches of many
// (sequence, KV head) segments (fp16 caches): one producer warp per CTA
// streams whole blocks of the cache (a group of KV heads of a 16-token tile)
// through a ring of TMA stages, and one consumer warp per KV head of the
// group attends over them.
//
// Work units are (head group hg, sequence b, 16-token tile t) in hg, b, t
// order: unit x covers tokens [16t, 16t + 16) of sequence b for the HK
// consecutive KV heads of group hg (all n_kv_heads heads, or a part), i.e.
// the K and V rows of those heads in one physical block (or in a 16-row slice
// of a larger block).  In the cache layout [num_blocks][n_kv_heads]
// [block_size][head_dim] they form one strided box, so one 3-D TMA load per
// 64-column half fetches a unit's K (and one its V): 64 KB per unit at 8
// heads and head_dim 128, a handful of copy instructions per unit.  Smaller
// groups make smaller stages, and more of them fit on an SM (as more CTAs).
//
// CTA c of the one-wave grid owns the contiguous units [c*U, (c+1)*U), U =
// ceil(units / CTAs), so every CTA moves the same number of bytes whatever the
// mix of context lengths.
//  - The producer warp walks the range in order: it waits for a free stage,
//    writes the unit's description, and loads the unit's K and V (and the
//    sequence's query rows, at the sequence's first unit in this range) into
//    the stage, all counted on the stage's "full" barrier.  Block ids come 32
//    at a time, one per lane, ahead of use.
//  - Consumer warp j takes head j of the group in every unit: it folds the
//    16 x head_dim K and V rows of that head into its online-softmax state of
//    segment (b, head)
//    (mma_tile.cuh) and arrives on the stage's "empty" barrier, which
//    completes when every head is done.  A warp therefore sees all of its
//    segment's tiles in this CTA, and no partial results are merged inside a
//    CTA.
//  - At the end of a sequence's units in the range the warp finalises:
//    sequences inside the range are written out (fp16 out, lse).  A sequence
//    cut by a range boundary (only the first and the last of a range) leaves
//    one record per (CTA, head) in the workspace with plain stores; once its
//    range is done the warp makes its records visible with one release,
//    counts them on the segments' counters, and where it arrived last merges
//    all records of the segment in CTA order, writes the output and resets
//    the counter.  No global round trip stalls a warp before its range is
//    done, so no warp holds the ring up.  The counters sit at the start of
//    the workspace and must be zero when the kernel starts (an arrival that
//    proves otherwise flags PKV_ERRBIT_WORKSPACE).  Every unit's rows
//    are summed in the same order on every run, so results are reproducible
//    bit for bit.
//
// Every wait is bounded: on a timeout the kernel flags PKV_ERRBIT_TIMEOUT,
// stops the CTA, waits (bounded) for the copies it has in flight and returns.
//
// Method: "Distributed LLM Inference Serving Platform", sections 2-3 (block
// table gather) and 5.1 (attention over every block of a sequence's table),
// GQA from section 1; online softmax and the log-sum-exp combination of
// partial results from FlashAttention-2 (section 14 references).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <mutex>

#include "mma_tile.cuh"
#include "pagedkv.h"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kMaxStages = 8;
constexpr int kMaxSeqsPipe = 2048;
constexpr int kSmemPerSm = 226 * 1024;  // shared memory the CTAs of one SM may take
constexpr int kMinUnitsPerCta = 4;      // smaller problems use fewer CTAs
constexpr float kLn2p = 0.69314718055994531f;

// HK: KV heads per unit (a group of consecutive heads; all of them, or a
// part so that the ring's stages are smaller and more of them fit an SM).
template <int D, int G, int HK>
struct PipeCfg : MmaCfg<D> {
    static constexpr int THREADS = (HK + 1) * 32;  // a consumer warp per head + the producer
    static constexpr int CTAS_PER_SM = 8 / HK;
    static constexpr int HALF_BYTES = HK * MmaCfg<D>::BOX_BYTES;    // 64 columns, every head
    static constexpr int KV_BYTES = MmaCfg<D>::BOXES * HALF_BYTES;  // K (or V) of a unit
    static constexpr int Q_BYTES = HK * G * D * 2;                  // the group's query rows
    static constexpr int STAGE_BYTES = (2 * KV_BYTES + Q_BYTES + 1023) / 1024 * 1024;
    // cross-CTA record of one head: acc [G][D], m [G], l [G], padded to 16 bytes
    static constexpr size_t REC = (static_cast<size_t>(G) * (D + 2) * 4 + 15) / 16 * 16;
    // a consumer's slice of a ring of at least two stages holds a record, so
    // that a merge round always stages one or more
    static_assert(2 * STAGE_BYTES / HK >= static_cast<int>(REC) + 16, "merge slice");
};

struct __align__(16) UnitMeta {
    int b;        // the sequence
    int hg;       // the head group
    int n_valid;  // rows of the tile that take part (0: a skipped block)
    int pad;
};

__device__ __forceinline__ int clamped_len_p(const DecodeArgs &a, int b, bool flag) {
    const int L = a.context_lens[b];
    const long long cap_ll = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    const int cap = static_cast<int>(cap_ll < a.max_context_len ? cap_ll : a.max_context_len);
    if (L < 0 || L > cap) {
        if (flag) flag_error(a.err, PKV_ERRBIT_CONTEXT);
        return L < 0 ? 0 : cap;
    }
    return L;
}

// Bounded wait for a barrier phase that also gives up when the CTA aborts.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity,
                                                   const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 0; it < kWaitLimitIters; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
    return false;
}

// The sequence holding unit index r (0 <= r < pre[B]): the largest b with
// pre[b] <= r; it has tiles.
__device__ __forceinline__ int seq_of(int r, const int *pre, int B) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <int D, int G, int HK>
__global__ void __launch_bounds__(PipeCfg<D, G, HK>::THREADS, PipeCfg<D, G, HK>::CTAS_PER_SM)
    decode_pipeline_kernel(const __grid_constant__ DecodeArgs a,
                           const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const int ns) {
    using C = PipeCfg<D, G, HK>;
    constexpr int kThreads = C::THREADS;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages];
    __shared__ uint64_t empty_bar[kMaxStages];
    __shared__ UnitMeta meta[kMaxStages];
    __shared__ uint64_t merge_bar[HK];  // a consumer's bulk copies of records
    __shared__ volatile int s_abort;
    __shared__ int s_scan[HK + 1];

    const uint32_t raw_s = smem_addr(smem_raw);
    unsigned char *ring = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
    int *s_pre = reinterpret_cast<int *>(ring + ns * C::STAGE_BYTES);  // [B + 1]
    int *s_len = s_pre + a.num_seqs + 1;                                // [B]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int B = a.num_seqs;
    const int H = a.n_q_heads;
    const int Hk = a.n_kv_heads;
    const int NG = Hk / HK;  // head groups
    const int bs = a.block_size;
    char *ws = reinterpret_cast<char *>(a.ws_acc);
    int *counters = reinterpret_cast<int *>(ws);

    if (tid == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], HK);
        }
        for (int w = 0; w < HK; ++w) mbar_init(&merge_bar[w], 1);
        fence_barrier_init();
        s_abort = 0;
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
    // the kernel before (e.g. the append) must be complete before anything it
    // may write is read; after this library's append only the caches are.
    // Once this grid has waited, everything before it in the stream is
    // complete, so the next kernel may be scheduled as this grid's CTAs
    // retire (it too waits for this grid before reading what it writes).
    if (a.defer_dep_wait != 2) {
        grid_dependency_wait();
        allow_dependent_launch();
    }

    // --- tiles per sequence, prefix-summed: contiguous chunk per thread, then a scan
    const int chunk = (B + kThreads - 1) / kThreads;
    const int c0 = min(B, tid * chunk);
    const int c1 = min(B, c0 + chunk);
    int local = 0;
    for (int b = c0; b < c1; ++b) {
        const int L = clamped_len_p(a, b, blockIdx.x == 0);
        s_len[b] = L;
        local += (L + kMmaTile - 1) / kMmaTile;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_scan[w];
    int run = base + incl - local;
    for (int b = c0; b < c1; ++b) {
        s_pre[b] = run;
        run += (s_len[b] + kMmaTile - 1) / kMmaTile;
    }
    if (tid == kThreads - 1) s_pre[B] = base + incl;
    __syncthreads();

    // Empty sequences (spread over the CTAs): out = 0, lse = -inf.
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        if (s_pre[b + 1] != s_pre[b]) continue;
        __half *ob = static_cast<__half *>(a.out) + static_cast<size_t>(b) * H * D;
        for (int i = tid; i < H * D; i += kThreads) ob[i] = __float2half_rn(0.f);
        if (a.lse_out)
            for (int h = tid; h < H; h += kThreads)
                a.lse_out[static_cast<size_t>(b) * H + h] = -INFINITY;
    }

    // --- this CTA's range of units
    const int T = s_pre[B];  // units per head group
    const int TT = NG * T;   // < 2^31 (checked by the planner)
    const int U = (TT + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int x0 = min(TT, static_cast<int>(blockIdx.x) * U);
    const int x1 = min(TT, x0 + U);
    const int n = x1 - x0;
    if (n <= 0) return;  // CTA-uniform; no CTA-wide barrier below

    if (warp == HK) {
        // =================== producer ===================
        // lane i holds the block id of unit 32c + i of the range, for the
        // chunk c being issued (ids_cur) and the next one (ids_next)
        auto load_ids = [&](int chunk_no) -> int {
            const int kk = chunk_no * 32 + lane;
            if (kk >= n) return -1;
            const int x = x0 + kk;
            const int r = x % T;
            const int b = seq_of(r, s_pre, B);
            return a.block_tables[static_cast<size_t>(b) * a.max_blocks_per_seq +
                                  ((r - s_pre[b]) * kMmaTile) / bs];
        };
        int ids_cur = load_ids(0);
        int ids_next = load_ids(1);
        int phg = x0 / T;                   // the head group of the unit being issued,
        int pb = seq_of(x0 % T, s_pre, B);  // its sequence
        int pt = x0 % T - s_pre[pb];        // and its tile
        int prev_key = -1;
        if (a.defer_dep_wait == 2) {  // the append has written the caches
            grid_dependency_wait();
            allow_dependent_launch();
        }
        int k = 0;
        bool failed = false;
        for (; k < n; ++k) {
            const int stage = k % ns;
            if (k >= ns) {  // unit k - ns held this stage: wait until every head is done with it
                const bool ok =
                    mbar_wait_or_abort(&empty_bar[stage], ((k / ns) - 1) & 1, &s_abort);
                if (__any_sync(0xffffffffu, !ok)) {
                    failed = !s_abort;
                    break;
                }
            }
            if (s_abort) break;
            if (k > 0 && (k & 31) == 0) {
                ids_cur = ids_next;
                ids_next = load_ids((k >> 5) + 1);
            }
            const int id = __shfl_sync(0xffffffffu, ids_cur, k & 31);
            const int key = phg * B + pb;
            const bool newseq = key != prev_key;
            prev_key = key;
            if (lane == 0) {
                const bool ok = id >= 0 && id < a.num_blocks;
                if (!ok) flag_error(a.err, PKV_ERRBIT_BLOCK_ID);
                const int tok0 = pt * kMmaTile;
                meta[stage].b = pb;
                meta[stage].hg = phg;
                meta[stage].n_valid = ok ? min(kMmaTile, s_len[pb] - tok0) : 0;
                uint64_t *bar = &full_bar[stage];
                // the description above is ordered before the arrival (release)
                mbar_arrive_expect_tx(bar, (ok ? 2 * C::KV_BYTES : 0) + (newseq ? C::Q_BYTES : 0));
                unsigned char *st = ring + stage * C::STAGE_BYTES;
                if (ok) {
#pragma unroll
                    for (int h = 0; h < C::BOXES; ++h) {
                        tma_load_3d(st + h * C::HALF_BYTES, &tmap_k, h * 64, tok0 % bs,
                                    id * Hk + phg * HK, bar);
                        tma_load_3d(st + C::KV_BYTES + h * C::HALF_BYTES, &tmap_v, h * 64, tok0 % bs,
                                    id * Hk + phg * HK, bar);
                    }
                }
                if (newseq)  // the segment's first unit here: the group's query rows too
                    bulk_copy_g2s(st + 2 * C::KV_BYTES,
                                  static_cast<const __half *>(a.q) +
                                      (static_cast<size_t>(pb) * H + static_cast<size_t>(phg) * HK * G) * D,
                                  C::Q_BYTES, bar);
            }
            if (++pt == s_pre[pb + 1] - s_pre[pb]) {  // next sequence with tiles
                pt = 0;
                do {
                    ++pb;
                } while (pb < B && s_pre[pb + 1] == s_pre[pb]);
                if (pb == B) {  // next head group
                    ++phg;
                    pb = 0;
                    while (pb < B && s_pre[pb + 1] == s_pre[pb]) ++pb;
                }
            }
        }
        if (lane == 0) {
            if (failed) {
                flag_error(a.err, PKV_ERRBIT_TIMEOUT);
                s_abort = 1;
            }
            // every copy issued must land before the CTA may exit
            for (int kk = k > ns ? k - ns : 0; kk < k; ++kk)
                mbar_wait_bounded(&full_bar[kk % ns], (kk / ns) & 1);
        }
        return;
    }

    // ============ consumers: warp j = head j of the unit's group ============
    const int j = warp;
    float o[C::NB_D][4];
    uint32_t qa[C::NP][4];
    float m_run = -INFINITY, l_run = 0.f;
    int cur_b = -1, cur_hg = -1;
    const int gg = g < G ? g : 0;
    const int cta = blockIdx.x;
    constexpr size_t REC = C::REC;
    auto rec = [&](int cc, int slot) {
        return ws + kBalancedCounterBytes + ((static_cast<size_t>(cc) * 2 + slot) * HK + j) * REC;
    };

    // Output row of query head (hg*HK + j)*G + g of sequence b: o / l in
    // fp16, and the lse.
    auto write_out = [&](int hg, int b, float fm, float fl) {
        if (g >= G) return;
        const size_t bh =
            static_cast<size_t>(b) * H + (static_cast<size_t>(hg) * HK + j) * G + g;
        const float inv = fl > 0.f ? 1.f / fl : 0.f;
        __half2 *dst = reinterpret_cast<__half2 *>(static_cast<__half *>(a.out) + bh * D);
#pragma unroll
        for (int nb = 0; nb < C::NB_D; ++nb)
            dst[nb * 4 + tq] = __floats2half2_rn(o[nb][0] * inv, o[nb][1] * inv);
        if (tq == 0 && a.lse_out) a.lse_out[bh] = fl > 0.f ? (fm + log2f(fl)) * kLn2p : -INFINITY;
    };

    // Segments cut by this range's boundaries whose record is stored but not
    // yet counted (at most the range's first and last).
    int pend_b[2], pend_hg[2], pend_n = 0;

    // The warp has seen every unit of segment (hg, b) in this range: write
    // its head's result out, or store it as this CTA's record of a cut
    // segment.
    auto finalize = [&](int hg, int b) {
        float fl = l_run;
        fl += __shfl_xor_sync(0xffffffffu, fl, 1);
        fl += __shfl_xor_sync(0xffffffffu, fl, 2);
        const int s0 = hg * T + s_pre[b];
        const int nt = s_pre[b + 1] - s_pre[b];
        if (s0 >= x0 && s0 + nt <= x1) {
            write_out(hg, b, m_run, fl);
            return;
        }
        // slot 0: the sequence started before this CTA's range; 1: it starts here
        char *r = rec(cta, s0 < x0 ? 0 : 1);
        if (g < G) {
            float2 *acc = reinterpret_cast<float2 *>(r) + static_cast<size_t>(g) * (D / 2);
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb) acc[nb * 4 + tq] = make_float2(o[nb][0], o[nb][1]);
            if (tq == 0) {
                reinterpret_cast<float *>(r)[G * D + g] = m_run;
                reinterpret_cast<float *>(r)[G * D + G + g] = fl;
            }
        }
        pend_b[pend_n] = b;
        pend_hg[pend_n++] = hg;
    };

    // Merges all records of cut segment (b, j) in CTA order (this CTA's
    // included), writes the output and resets the counter.  The records come
    // into this warp's slice of the ring (free once every consumer is past
    // its last unit) by bulk copies, a batch per round trip.  False on a
    // timeout.
    constexpr int kSliceAlign = 16;
    const int slice = (ns * C::STAGE_BYTES / HK) / kSliceAlign * kSliceAlign;
    const int per_batch = slice / static_cast<int>(REC);
    unsigned char *my_slice = ring + j * slice;
    uint32_t merge_phase = 0;
    auto merge = [&](int hg, int b) -> bool {
        const int s0 = hg * T + s_pre[b];
        const int nt = s_pre[b + 1] - s_pre[b];
        const int first = s0 / U;
        const int last = (s0 + nt - 1) / U;
        float M = -INFINITY, L = 0.f;
#pragma unroll
        for (int nb = 0; nb < C::NB_D; ++nb) o[nb][0] = o[nb][1] = 0.f;
        for (int f = first; f <= last; f += per_batch) {
            const int cnt = min(per_batch, last - f + 1);
            if (lane == 0) {
                mbar_arrive_expect_tx(&merge_bar[j], static_cast<uint32_t>(cnt * REC));
                for (int i = 0; i < cnt; ++i)
                    bulk_copy_g2s(my_slice + i * REC, rec(f + i, f + i == first ? 1 : 0),
                                  static_cast<uint32_t>(REC), &merge_bar[j]);
            }
            const bool ok = mbar_wait_bounded(&merge_bar[j], merge_phase & 1);
            ++merge_phase;
            if (__any_sync(0xffffffffu, !ok)) return false;
            for (int i = 0; i < cnt; ++i) {
                const float *rf = reinterpret_cast<const float *>(my_slice + i * REC);
                const float mi = rf[G * D + gg];
                if (mi == -INFINITY) continue;  // a piece of skipped blocks only
                const float li = rf[G * D + G + gg];
                const float Mn = fmaxf(M, mi);
                const float so = M == -INFINITY ? 0.f : exp2f(M - Mn);
                const float sn = exp2f(mi - Mn);
                L = L * so + li * sn;
                const float2 *acc = reinterpret_cast<const float2 *>(rf) + static_cast<size_t>(gg) * (D / 2);
#pragma unroll
                for (int nb = 0; nb < C::NB_D; ++nb) {
                    const float2 v = acc[nb * 4 + tq];
                    o[nb][0] = o[nb][0] * so + v.x * sn;
                    o[nb][1] = o[nb][1] * so + v.y * sn;
                }
                M = Mn;
            }
            __syncwarp();  // every lane's reads before the next batch lands
        }
        // ready for the next call: back from n to 0 (a poisoned count stays >= n)
        if (lane == 0) red_add_relaxed_gpu(&counters[first * HK + j], -(last - first + 1));
        write_out(hg, b, M, L);
        return true;
    };

    // After the range: count this warp's records on their segments' counters
    // (one release covers both) and merge the segments it arrived last on.
    auto publish = [&]() -> bool {
        if (pend_n == 0) return true;
        __syncwarp();  // every lane's record stores before lane 1's release
        int last_on = 0;  // bit i: arrived last on pending segment i
        if (lane == 1) {
            // one release fence for the records of both segments, then the
            // counts (their return values are independent)
            __threadfence();
            int old[2] = {0, 0};
            for (int i = 0; i < pend_n; ++i) {
                const int first = (pend_hg[i] * T + s_pre[pend_b[i]]) / U;
                old[i] = atomic_add_relaxed_gpu(&counters[first * HK + j], 1);
            }
            for (int i = 0; i < pend_n; ++i) {
                const int s0 = pend_hg[i] * T + s_pre[pend_b[i]];
                const int nt = s_pre[pend_b[i] + 1] - s_pre[pend_b[i]];
                const int last = (s0 + nt - 1) / U - s0 / U;
                if (old[i] == last) last_on |= 1 << i;
                if (counter_not_zeroed(old[i], last)) {
                    flag_error(a.err, PKV_ERRBIT_WORKSPACE);
                    const int first = s0 / U;
                    atomic_exch_relaxed_gpu(&counters[first * HK + j], kCounterPoison);
                }
            }
        }
        last_on = __shfl_sync(0xffffffffu, last_on, 1);
        if (!last_on) return true;
        // the other CTAs' records, visible after lane 1 saw their counts, are
        // read by bulk copies (the async proxy)
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        // and land where the ring's tiles were read through the generic proxy
        fence_proxy_async_smem();
        for (int i = 0; i < pend_n; ++i)
            if ((last_on & (1 << i)) && !merge(pend_hg[i], pend_b[i])) return false;
        return true;
    };

    bool failed = false;
    for (int k = 0; k < n; ++k) {
        const int stage = k % ns;
        const bool ok = (k == 0 && a.first_wait_polls >= 0)
                            ? mbar_wait_polls(&full_bar[stage], 0, a.first_wait_polls)
                            : mbar_wait_or_abort(&full_bar[stage], (k / ns) & 1, &s_abort);
        if (__any_sync(0xffffffffu, !ok)) {
            failed = true;
            break;
        }
        const UnitMeta mt = meta[stage];
        unsigned char *st = ring + stage * C::STAGE_BYTES;
        if (mt.b != cur_b || mt.hg != cur_hg) {  // the segment's first unit here (with the queries)
            if (cur_b >= 0) finalize(cur_hg, cur_b);
#pragma unroll
            for (int nb = 0; nb < C::NB_D; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
            cur_b = mt.b;
            cur_hg = mt.hg;
            load_q_frag<D>(qa, reinterpret_cast<const __half *>(st + 2 * C::KV_BYTES) +
                                   (j * G + gg) * D,
                           g < G, tq);
        }
        if (mt.n_valid > 0)
            mma_tile<D, false, C::HALF_BYTES>(st + j * MmaCfg<D>::BOX_BYTES,
                                              st + C::KV_BYTES + j * MmaCfg<D>::BOX_BYTES,
                                              mt.n_valid, qa, a.scale_log2, o, m_run, l_run, lane);
        __syncwarp();  // every lane's reads of the stage before it is released
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
    }
    if (failed && lane == 0) {
        if (!s_abort) flag_error(a.err, PKV_ERRBIT_TIMEOUT);
        s_abort = 1;
    }
    if (!failed && cur_b >= 0) finalize(cur_hg, cur_b);
    // every consumer is past its last unit: the ring is free for the merges
    // (a warp that gave up arrives here too)
    asm volatile("bar.sync 1, %0;" ::"r"(HK * 32) : "memory");
    if (!failed && !s_abort && !publish() && lane == 0) {
        flag_error(a.err, PKV_ERRBIT_TIMEOUT);
        s_abort = 1;
    }
}

template <int D, int G, int HK>
int pipe_stages(int B) {
    using C = PipeCfg<D, G, HK>;
    const long long budget = kSmemPerSm / C::CTAS_PER_SM - 1024 - (2LL * B + 1) * 4;
    long long s = budget / C::STAGE_BYTES;
    if (s > kMaxStages) s = kMaxStages;
    return static_cast<int>(s);
}

template <int D, int G, int HK>
size_t pipe_smem(int B, int ns) {
    using C = PipeCfg<D, G, HK>;
    return 1024 + static_cast<size_t>(ns) * C::STAGE_BYTES + (2 * static_cast<size_t>(B) + 1) * 4;
}

template <int D, int G, int HK>
bool pipe_attrs_ok() {
    static std::once_flag once;
    static bool ok = false;
    std::call_once(once, [] {
        auto kern = decode_pipeline_kernel<D, G, HK>;
        const size_t most = kSmemPerSm / PipeCfg<D, G, HK>::CTAS_PER_SM;
        ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(most)) == cudaSuccess &&
             cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    });
    return ok;
}

template <int D, int G, int HK>
cudaError_t launch_pipe_t(const DecodeArgs &a, const BalancedPlan &plan, const CUtensorMap &tk,
                          const CUtensorMap &tv, cudaStream_t stream) {
    if (!pipe_attrs_ok<D, G, HK>()) return cudaErrorInvalidConfiguration;
    const int ns = pipe_stages<D, G, HK>(a.num_seqs);
    if (ns < 2) return cudaErrorInvalidConfiguration;
    return launch_pdl(decode_pipeline_kernel<D, G, HK>, dim3(plan.ctas),
                      dim3(PipeCfg<D, G, HK>::THREADS), pipe_smem<D, G, HK>(a.num_seqs, ns), stream,
                      a, tk, tv, ns);
}

int sm_count_pipe() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess)
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    });
    return n;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_pipe() {
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

// 3-D view of a cache: x = head_dim column, y = row within a block, z =
// block * n_kv_heads + head.  A box of 64 columns x 16 rows x heads_per_box
// heads is one 64-column half of a unit (a head group of a 16-token tile),
// laid out in shared memory head by head, 2 KB each, with the 128-byte
// swizzle.
bool make_unit_map(CUtensorMap *m, const void *base, long long num_blocks, int n_kv_heads,
                   int heads_per_box, int block_size, int D) {
    auto fn = encode_fn_pipe();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(block_size),
                          static_cast<cuuint64_t>(num_blocks) * static_cast<cuuint64_t>(n_kv_heads)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(block_size) * static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kMmaTile),
                         static_cast<cuuint32_t>(heads_per_box)};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t pipe_rec_bytes(int G, int D) { return (static_cast<size_t>(G) * (D + 2) * 4 + 15) / 16 * 16; }

}  // namespace

bool pipeline_supported(int num_seqs, int n_kv_heads, int head_dim, int group, int block_size,
                        long long cache_rows) {
    return num_seqs >= 1 && num_seqs <= kMaxSeqsPipe && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8) && n_kv_heads >= 1 &&
           (n_kv_heads % 8 == 0 || n_kv_heads == 1 || n_kv_heads == 2 || n_kv_heads == 4) &&
           block_size % kMmaTile == 0 && cache_rows < (1LL << 31);
}

namespace {

// KV heads per unit: 4 when they divide n_kv_heads (two CTAs per SM, each
// with three 32 KB stages at head_dim 128: on the Mistral-shaped mix 40.5 us,
// against 43.7 us with 8 heads and 66.7 us with 2), else all of them.
// PKV_PIPE_HEADS (1, 2, 4 or 8) overrides it when it divides n_kv_heads.
int pipe_heads(int n_kv_heads) {
    static int env = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        const char *e = std::getenv("PKV_PIPE_HEADS");
        env = e ? std::atoi(e) : 0;
    });
    int hc = n_kv_heads % 4 == 0 ? 4 : n_kv_heads;
    if ((env == 1 || env == 2 || env == 4 || env == 8) && n_kv_heads % env == 0) hc = env;
    return hc;
}

}  // namespace

bool pipeline_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int max_len,
                   BalancedPlan *plan) {
    const int G = n_q_heads / n_kv_heads;
    const int sms = sm_count_pipe();
    if (sms <= 0 || n_kv_heads <= 0) return false;
    const int hc = pipe_heads(n_kv_heads);
    if (n_kv_heads % hc != 0) return false;
    const long long t_max = static_cast<long long>(num_seqs) * (n_kv_heads / hc) *
                            ((static_cast<long long>(max_len) + kMmaTile - 1) / kMmaTile);
    if (t_max >= (1LL << 31)) return false;  // unit indices are 32-bit
    // at least two stages must fit beside the per-sequence tables
    const long long stage = (2LL * (head_dim / 64) * hc * MmaCfg<128>::BOX_BYTES +
                             static_cast<long long>(hc) * G * head_dim * 2 + 1023) / 1024 * 1024;
    const long long budget = kSmemPerSm / (8 / hc) - 1024 - (2LL * num_seqs + 1) * 4;
    if (budget / stage < 2) return false;
    long long ctas = static_cast<long long>(sms) * (8 / hc);  // one wave
    const long long need = (t_max + kMinUnitsPerCta - 1) / kMinUnitsPerCta;
    if (need < ctas) ctas = need;
    if (ctas * hc > kBalancedMaxWorkers) ctas = kBalancedMaxWorkers / hc;
    if (ctas < 1) ctas = 1;
    plan->ctas = static_cast<int>(ctas);
    plan->warps = hc + 1;
    plan->workers = plan->ctas;
    plan->kind = 1;
    plan->heads = hc;
    plan->ws_bytes = kBalancedCounterBytes +
                     static_cast<size_t>(plan->ctas) * 2 * hc * pipe_rec_bytes(G, head_dim);
    return true;
}

cudaError_t launch_decode_pipeline(const DecodeArgs &a, const BalancedPlan &plan,
                                   cudaStream_t stream) {
    const int hc = plan.heads;
    CUtensorMap tk{}, tv{};
    if (!make_unit_map(&tk, a.k_cache, a.num_blocks, a.n_kv_heads, hc, a.block_size, a.head_dim) ||
        !make_unit_map(&tv, a.v_cache, a.num_blocks, a.n_kv_heads, hc, a.block_size, a.head_dim))
        return cudaErrorNotSupported;
    const int g = a.n_q_heads / a.n_kv_heads;
#define PKV_PIPE_CASE(D_, G_, HK_) \
    if (a.head_dim == D_ && g == G_ && hc == HK_) \
        return launch_pipe_t<D_, G_, HK_>(a, plan, tk, tv, stream);
#define PKV_PIPE_G(D_, HK_) \
    PKV_PIPE_CASE(D_, 1, HK_) PKV_PIPE_CASE(D_, 2, HK_) PKV_PIPE_CASE(D_, 4, HK_) PKV_PIPE_CASE(D_, 8, HK_)
    PKV_PIPE_G(128, 8)
    PKV_PIPE_G(128, 4)
    PKV_PIPE_G(128, 2)
    PKV_PIPE_G(128, 1)
    PKV_PIPE_G(64, 8)
    PKV_PIPE_G(64, 4)
    PKV_PIPE_G(64, 2)
    PKV_PIPE_G(64, 1)
#undef PKV_PIPE_G
#undef PKV_PIPE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
