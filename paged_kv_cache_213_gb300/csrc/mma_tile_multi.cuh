// mma_tile_multi.cuh -- per-tile math of the multi-token (causal) kernel:
// one warp, one 16-token K/V tile, 16 query rows (query token x head pairs)
// as the M dimension of mma.m16n8k16.  Row g ("lo") and row g + 8 ("hi") of
// lane 4g + tq each carry their own online-softmax state and their own
// causal limit: token k of the tile takes part in row r's softmax iff
// k < nv_r.  Tile rows at or past nv_tile (past the context) are zeroed in
// V first, so that poisoned memory cannot reach P.V.
#pragma once

#include <cuda_fp16.h>

#include <cmath>

#include "mma_tile.cuh"
#include "pkv_ptx.cuh"

namespace pkv {

template <int D>
__device__ __forceinline__ void mma_tile_multi(const unsigned char *ks, unsigned char *vs,
                                               int nv_tile, int nv_lo, int nv_hi,
                                               const uint32_t (&qlo)[MmaCfg<D>::NP][4],
                                               const uint32_t (&qhi)[MmaCfg<D>::NP][4],
                                               float scale_log2, float (&o)[MmaCfg<D>::NB_D][4],
                                               float &m_lo, float &l_lo, float &m_hi,
                                               float &l_hi, int lane) {
    using C = MmaCfg<D>;
    const int g = lane >> 2;
    const int tq = lane & 3;
    if (nv_tile < kMmaTile) {
        const int per_row = C::BOXES * 8;
        for (int idx = lane; idx < (kMmaTile - nv_tile) * per_row; idx += 32) {
            const int r = nv_tile + idx / per_row;
            const int rem = idx % per_row;
            *reinterpret_cast<uint4 *>(vs + (rem >> 3) * C::BOX_BYTES + r * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // before a later TMA write of these bytes
        __syncwarp();
    }
    // S = Q K^T for tokens 0-7 (nb = 0) and 8-15 (nb = 1), rows g and g + 8
    float sacc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
        sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
        const int t = nb * 8 + g;
#pragma unroll
        for (int p = 0; p < C::NP; ++p) {
            const uint4 kw = *reinterpret_cast<const uint4 *>(ks + (p >> 1) * C::BOX_BYTES +
                                                              swz(t, 2 * tq + (p & 1)));
            const uint32_t a0[4] = {qlo[p][0], qhi[p][0], qlo[p][1], qhi[p][1]};
            mma_16816(sacc[nb], a0, kw.x, kw.y);
            const uint32_t a1[4] = {qlo[p][2], qhi[p][2], qlo[p][3], qhi[p][3]};
            mma_16816(sacc[nb], a1, kw.z, kw.w);
        }
    }
    // masked logits: token nb*8 + 2tq + e of rows g (lo) and g + 8 (hi)
    float sl[2][2], sh[2][2];
    float mxl = -INFINITY, mxh = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tt = nb * 8 + 2 * tq + e;
            sl[nb][e] = tt < nv_lo ? sacc[nb][e] * scale_log2 : -INFINITY;
            sh[nb][e] = tt < nv_hi ? sacc[nb][2 + e] * scale_log2 : -INFINITY;
            mxl = fmaxf(mxl, sl[nb][e]);
            mxh = fmaxf(mxh, sh[nb][e]);
        }
    mxl = fmaxf(mxl, __shfl_xor_sync(0xffffffffu, mxl, 1));
    mxl = fmaxf(mxl, __shfl_xor_sync(0xffffffffu, mxl, 2));
    mxh = fmaxf(mxh, __shfl_xor_sync(0xffffffffu, mxh, 1));
    mxh = fmaxf(mxh, __shfl_xor_sync(0xffffffffu, mxh, 2));
    const float mnl = fmaxf(m_lo, mxl);
    const float mnh = fmaxf(m_hi, mxh);
    const float cl = mnl == -INFINITY ? 1.f : exp2f(m_lo - mnl);
    const float ch = mnh == -INFINITY ? 1.f : exp2f(m_hi - mnh);
    float pl[2][2], ph[2][2], suml = 0.f, sumh = 0.f;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            pl[nb][e] = sl[nb][e] == -INFINITY ? 0.f : exp2f(sl[nb][e] - mnl);
            ph[nb][e] = sh[nb][e] == -INFINITY ? 0.f : exp2f(sh[nb][e] - mnh);
            suml += pl[nb][e];
            sumh += ph[nb][e];
        }
    l_lo = l_lo * cl + suml;
    l_hi = l_hi * ch + sumh;
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

}  // namespace pkv
