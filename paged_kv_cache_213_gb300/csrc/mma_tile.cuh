// mma_tile.cuh -- the per-tile math of the tensor-core decode kernels: one
// warp, one 16-token K/V tile (TMA-loaded with 128-byte swizzle), the GQA
// query group as the M dimension of mma.m16n8k16.
//
//   S = Q K^T       M = query heads (padded to 16), N = 8 tokens, K = head_dim
//   online softmax  fp32, exp2 domain, running max / sum per head
//   O += P V        M = heads, N = 8 head_dim columns, K = 16 tokens
//
// Fragment ownership: lane = 4*g + tq.  g is the query head (row of A / C),
// tq picks columns.  For S = Q K^T the MMA k index is mapped to head_dim so
// that each thread reads whole 16-byte pieces: piece p (0 .. D/32-1) of a row
// is the 16 bytes at column 64*(p/2) + 8*(2*tq + p%2); MMA k-step 2p+sub takes
// its words 2*sub (k = 2tq, 2tq+1) and 2*sub+1 (k = 2tq+8, 2tq+9).  Q and K use
// the same map, so the dot products are unchanged.  The C fragment of S
// (tokens 2tq, 2tq+1 of each 8-token block) is exactly the A fragment of P.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>

#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kMmaTile = 16;  // tokens per tile

template <int D>
struct MmaCfg {
    static constexpr int BOXES = D / 64;           // 64-column TMA boxes per tile
    static constexpr int BOX_BYTES = kMmaTile * 128;  // 16 rows x 128 B
    static constexpr int TILE_BYTES = BOXES * BOX_BYTES;
    static constexpr int NP = D / 32;              // 16-byte pieces per row per thread
    static constexpr int NB_D = D / 8;             // 8-column output blocks
};

// Byte offset of 16-byte unit `unit` (0-7) of row `row` in a 128B-swizzled box.
__device__ __forceinline__ int swz(int row, int unit) { return row * 128 + ((unit ^ (row & 7)) << 4); }

// The fp16 pair of E4M3 codes in bytes 0 (low half) and 1 of `two`.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    const __half2_raw h =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Piece p (as above) of row t of an E4M3 K tile staged by TMA with the D-byte
// swizzle (D = 128: 128B, 16-byte unit u of row t at u ^ (t & 7); D = 64:
// 64B, at u ^ ((t >> 1) & 3)), widened to the four fp16 pairs that the same
// piece of an fp16 tile holds.  Every E4M3 code is exact in fp16.
template <int D>
__device__ __forceinline__ uint4 e4m3_piece(const unsigned char *ks, int t, int p, int tq) {
    const int u = 4 * (p >> 1) + tq;  // 16-byte unit of the piece; it starts 8 * (p & 1) in
    const int off = D == 128 ? swz(t, u) : t * 64 + ((u ^ ((t >> 1) & 3)) << 4);
    const uint2 w = *reinterpret_cast<const uint2 *>(ks + off + 8 * (p & 1));
    return make_uint4(e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16), e4m3x2_to_f16x2(w.y),
                      e4m3x2_to_f16x2(w.y >> 16));
}

// Byte offset of bytes [4c, 4c + 4) of row t of an E4M3 tile with the
// D-byte swizzle (see e4m3_piece); c < D / 4.
template <int D>
__device__ __forceinline__ int e4m3_word_off(int t, int c) {
    const int u = c >> 2;  // 16-byte unit
    return (D == 128 ? swz(t, u) : t * 64 + ((u ^ ((t >> 1) & 3)) << 4)) + 4 * (c & 3);
}

// Q fragments of head g from a row-major [.., D] fp16 row (global or shared).
template <int D>
__device__ __forceinline__ void load_q_frag(uint32_t (&qa)[MmaCfg<D>::NP][4], const __half *row,
                                            bool present, int tq) {
#pragma unroll
    for (int p = 0; p < MmaCfg<D>::NP; ++p) {
        const int col = (p >> 1) * 64 + (2 * tq + (p & 1)) * 8;
        if (present) {
            const uint4 v = *reinterpret_cast<const uint4 *>(row + col);
            qa[p][0] = v.x;
            qa[p][1] = v.y;
            qa[p][2] = v.z;
            qa[p][3] = v.w;
        } else {
            qa[p][0] = qa[p][1] = qa[p][2] = qa[p][3] = 0u;
        }
    }
}

// Where head_dim column `col` sits in a row of partial sums stored in
// register order (float2 number 4 * nb + tq holds o[nb][0], o[nb][1] of lane
// 4g + tq) by the E4M3 tile math: column 32c + 8tq + e is o[4c + e % 4][e / 4].
__host__ __device__ __forceinline__ int f8_acc_index(int col) {
    const int c = col >> 5, tq = (col >> 3) & 3, e = col & 7;
    return 2 * ((4 * c + (e & 3)) * 4 + tq) + (e >> 2);
}

// O += P V for an E4M3 V tile (D-byte swizzle): lane 4g + tq loads the
// 4-byte words at column 32c + 4g of rows 2tq, 2tq+1, 2tq+8, 2tq+9 and pairs
// their bytes, so byte i of each row pair feeds output block 4c + i, column g
// (the permuted column order described at mma_tile).  pa: the A fragment of P.
template <int D>
__device__ __forceinline__ void pv_e4m3(const unsigned char *vs, const uint32_t (&pa)[4],
                                        float (&o)[MmaCfg<D>::NB_D][4], int lane) {
    const int g = lane >> 2;
    const int tq = lane & 3;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        const int wc = 8 * c + g;  // 4-byte word of the row
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(vs + e4m3_word_off<D>(2 * tq, wc));
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(vs + e4m3_word_off<D>(2 * tq + 1, wc));
        const uint32_t w2 = *reinterpret_cast<const uint32_t *>(vs + e4m3_word_off<D>(2 * tq + 8, wc));
        const uint32_t w3 = *reinterpret_cast<const uint32_t *>(vs + e4m3_word_off<D>(2 * tq + 9, wc));
        const uint32_t lo01 = __byte_perm(w0, w1, 0x5140);  // byte 0 pair, byte 1 pair
        const uint32_t lo23 = __byte_perm(w0, w1, 0x7362);  // byte 2 pair, byte 3 pair
        const uint32_t hi01 = __byte_perm(w2, w3, 0x5140);
        const uint32_t hi23 = __byte_perm(w2, w3, 0x7362);
        mma_16816(o[4 * c + 0], pa, e4m3x2_to_f16x2(lo01), e4m3x2_to_f16x2(hi01));
        mma_16816(o[4 * c + 1], pa, e4m3x2_to_f16x2(lo01 >> 16), e4m3x2_to_f16x2(hi01 >> 16));
        mma_16816(o[4 * c + 2], pa, e4m3x2_to_f16x2(lo23), e4m3x2_to_f16x2(hi23));
        mma_16816(o[4 * c + 3], pa, e4m3x2_to_f16x2(lo23 >> 16), e4m3x2_to_f16x2(hi23 >> 16));
    }
}

// One tile: rows [0, n_valid) of the K tile `ks` and V tile `vs` take part;
// the V rows past n_valid are zeroed first (they may hold another sequence's
// data or NaN and must not reach P.V).  Updates the running state of head g.
//
// F8: both tiles hold E4M3 codes with the D-byte swizzle, widened in
// registers.  K goes piece by piece (e4m3_piece).  V needs, per lane, pairs
// of tokens (2tq, 2tq+1) and (2tq+8, 2tq+9) of one column: the lane loads
// 4-byte words of those four rows and pairs their bytes, so the output
// columns are permuted instead of V being transposed.  Output block 4c + i,
// column n, holds head_dim column 32c + 4n + i: o[4c + i][0] is column
// 32c + 8tq + i and o[4c + i][1] is column 32c + 8tq + 4 + i (f8_acc_index).
//
// HS: bytes from a 64-column box of an fp16 tile to the next one (the box
// holding columns 64 .. 127 at D = 128); MmaCfg<D>::BOX_BYTES when the tile's
// boxes are adjacent, larger when tiles of several heads are interleaved.
template <int D, bool F8 = false, int HS = MmaCfg<D>::BOX_BYTES>
__device__ __forceinline__ void mma_tile(const unsigned char *ks, unsigned char *vs, int n_valid,
                                         const uint32_t (&qa)[MmaCfg<D>::NP][4],
                                         float scale_log2, float (&o)[MmaCfg<D>::NB_D][4],
                                         float &m_run, float &l_run, int lane) {
    using C = MmaCfg<D>;
    const int g = lane >> 2;
    const int tq = lane & 3;
    if (n_valid < kMmaTile) {
        if constexpr (F8) {  // a row of codes is D contiguous bytes (swizzled within)
            for (int idx = n_valid * (D / 16) + lane; idx < kMmaTile * (D / 16); idx += 32)
                reinterpret_cast<uint4 *>(vs)[idx] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            const int per_row = C::BOXES * 8;
            for (int idx = lane; idx < (kMmaTile - n_valid) * per_row; idx += 32) {
                const int r = n_valid + idx / per_row;
                const int rem = idx % per_row;
                *reinterpret_cast<uint4 *>(vs + (rem >> 3) * HS + r * 128 +
                                           (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();  // before a later TMA write of these bytes
        __syncwarp();
    }

    // S = Q K^T for tokens 0-7 (nb = 0) and 8-15 (nb = 1)
    float sacc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
        sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
        const int t = nb * 8 + g;
#pragma unroll
        for (int p = 0; p < C::NP; ++p) {
            uint4 kw;
            if constexpr (F8)
                kw = e4m3_piece<D>(ks, t, p, tq);
            else
                kw = *reinterpret_cast<const uint4 *>(ks + (p >> 1) * HS +
                                                      swz(t, 2 * tq + (p & 1)));
            const uint32_t a0[4] = {qa[p][0], 0u, qa[p][1], 0u};
            mma_16816(sacc[nb], a0, kw.x, kw.y);
            const uint32_t a1[4] = {qa[p][2], 0u, qa[p][3], 0u};
            mma_16816(sacc[nb], a1, kw.z, kw.w);
        }
    }
    // online softmax of head g over tokens 2tq, 2tq+1, 8+2tq, 9+2tq
    float s[2][2];
    float mx = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tt = nb * 8 + 2 * tq + e;
            s[nb][e] = tt < n_valid ? sacc[nb][e] * scale_log2 : -INFINITY;
            mx = fmaxf(mx, s[nb][e]);
        }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
    float pv[2][2];
    float psum = 0.f;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            pv[nb][e] = (s[nb][e] == -INFINITY) ? 0.f : exp2f(s[nb][e] - m_new);
            psum += pv[nb][e];
        }
    l_run = l_run * corr + psum;
    m_run = m_new;
#pragma unroll
    for (int n = 0; n < C::NB_D; ++n) {
        o[n][0] *= corr;
        o[n][1] *= corr;
    }
    const uint32_t pa[4] = {pack_half2(pv[0][0], pv[0][1]), 0u, pack_half2(pv[1][0], pv[1][1]),
                            0u};
    if constexpr (F8) {
        pv_e4m3<D>(vs, pa, o, lane);
    } else {
        // O += P V: V fragments by transposed 8x8 loads, two 8-column blocks per load
        const int lm = lane >> 3;
        const int ri = lane & 7;
        const int vt = ((lm & 1) << 3) + ri;
#pragma unroll
        for (int qd = 0; qd < C::NB_D / 2; ++qd) {
            const int u = 2 * qd + (lm >> 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(r0, r1, r2, r3, vs + (u >> 3) * HS + swz(vt, u & 7));
            mma_16816(o[2 * qd], pa, r0, r1);
            mma_16816(o[2 * qd + 1], pa, r2, r3);
        }
    }
}

}  // namespace pkv

namespace pkv {

// Both halves of the 16-row A tile carry queries: row g ("lo") and row g+8
// ("hi") of lane 4g+tq, each with its own online-softmax state.  Used where
// one K/V tile serves several sequences' queries at once (shared prefixes).
// All 16 rows of the tile take part (a shared prefix is made of full tiles).
// F8: E4M3 tiles as in mma_tile, with the same permuted output columns.
template <int D, bool F8 = false>
__device__ __forceinline__ void mma_tile_2rows(const unsigned char *ks, const unsigned char *vs,
                                               const uint32_t (&qlo)[MmaCfg<D>::NP][4],
                                               const uint32_t (&qhi)[MmaCfg<D>::NP][4],
                                               float scale_log2, float (&o)[MmaCfg<D>::NB_D][4],
                                               float &m_lo, float &l_lo, float &m_hi, float &l_hi,
                                               int lane) {
    using C = MmaCfg<D>;
    const int g = lane >> 2;
    const int tq = lane & 3;
    float sacc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
        sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
        const int t = nb * 8 + g;
#pragma unroll
        for (int p = 0; p < C::NP; ++p) {
            uint4 kw;
            if constexpr (F8)
                kw = e4m3_piece<D>(ks, t, p, tq);
            else
                kw = *reinterpret_cast<const uint4 *>(ks + (p >> 1) * C::BOX_BYTES +
                                                      swz(t, 2 * tq + (p & 1)));
            const uint32_t a0[4] = {qlo[p][0], qhi[p][0], qlo[p][1], qhi[p][1]};
            mma_16816(sacc[nb], a0, kw.x, kw.y);
            const uint32_t a1[4] = {qlo[p][2], qhi[p][2], qlo[p][3], qhi[p][3]};
            mma_16816(sacc[nb], a1, kw.z, kw.w);
        }
    }
    float mxl = -INFINITY, mxh = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            sacc[nb][e] *= scale_log2;
            sacc[nb][2 + e] *= scale_log2;
            mxl = fmaxf(mxl, sacc[nb][e]);
            mxh = fmaxf(mxh, sacc[nb][2 + e]);
        }
    }
    mxl = fmaxf(mxl, __shfl_xor_sync(0xffffffffu, mxl, 1));
    mxl = fmaxf(mxl, __shfl_xor_sync(0xffffffffu, mxl, 2));
    mxh = fmaxf(mxh, __shfl_xor_sync(0xffffffffu, mxh, 1));
    mxh = fmaxf(mxh, __shfl_xor_sync(0xffffffffu, mxh, 2));
    const float mnl = fmaxf(m_lo, mxl);
    const float mnh = fmaxf(m_hi, mxh);
    const float cl = exp2f(m_lo - mnl);  // 0 while m = -inf
    const float ch = exp2f(m_hi - mnh);
    float pl[2][2], ph[2][2], sl = 0.f, sh = 0.f;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            pl[nb][e] = exp2f(sacc[nb][e] - mnl);
            ph[nb][e] = exp2f(sacc[nb][2 + e] - mnh);
            sl += pl[nb][e];
            sh += ph[nb][e];
        }
    l_lo = l_lo * cl + sl;
    l_hi = l_hi * ch + sh;
    m_lo = mnl;
    m_hi = mnh;
#pragma unroll
    for (int n = 0; n < C::NB_D; ++n) {
        o[n][0] *= cl;
        o[n][1] *= cl;
        o[n][2] *= ch;
        o[n][3] *= ch;
    }
    const uint32_t pa[4] = {pack_half2(pl[0][0], pl[0][1]), pack_half2(ph[0][0], ph[0][1]),
                            pack_half2(pl[1][0], pl[1][1]), pack_half2(ph[1][0], ph[1][1])};
    if constexpr (F8) {
        pv_e4m3<D>(vs, pa, o, lane);
    } else {
        const int lm = lane >> 3;
        const int ri = lane & 7;
        const int vt = ((lm & 1) << 3) + ri;
#pragma unroll
        for (int qd = 0; qd < C::NB_D / 2; ++qd) {
            const int u = 2 * qd + (lm >> 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(r0, r1, r2, r3, vs + (u >> 3) * C::BOX_BYTES + swz(vt, u & 7));
            mma_16816(o[2 * qd], pa, r0, r1);
            mma_16816(o[2 * qd + 1], pa, r2, r3);
        }
    }
}

}  // namespace pkv
