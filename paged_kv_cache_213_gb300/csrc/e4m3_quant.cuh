// e4m3_quant.cuh -- fp16 to E4M3 quantization of the FP8 KV cache, shared
// by the append kernel and the one-launch decode step so that both store the
// same codes.  Each value is stored as E4M3(x / scale): the quotient one
// correctly rounded fp32 division, the conversion round-to-nearest-even with
// finite overflow saturated to +-448 (cvt.rn.satfinite).  E4M3 with one scale
// per cache tensor is this library's reading of the quantized KV cache that
// "Roadmap: vLLM-style serving features for TornadoVM batched decode" lists
// in its KV-cache items.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace pkv {

// 16 fp16 values (lo: values 0-7, hi: 8-15) to 16 E4M3 codes, value i in byte i.
__device__ __forceinline__ uint4 quantize16(const uint4 &lo, const uint4 &hi, float scale) {
    const __half2 *h0 = reinterpret_cast<const __half2 *>(&lo);
    const __half2 *h1 = reinterpret_cast<const __half2 *>(&hi);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 a = i < 2 ? h0[2 * i] : h1[2 * i - 4];
        const __half2 b = i < 2 ? h0[2 * i + 1] : h1[2 * i - 3];
        const float2 fa = __half22float2(a);
        const float2 fb = __half22float2(b);
        const __nv_fp8x2_storage_t ca = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(fa.x, scale), __fdiv_rn(fa.y, scale)), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t cb = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(fb.x, scale), __fdiv_rn(fb.y, scale)), __NV_SATFINITE, __NV_E4M3);
        w[i] = static_cast<uint32_t>(ca) | (static_cast<uint32_t>(cb) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace pkv
