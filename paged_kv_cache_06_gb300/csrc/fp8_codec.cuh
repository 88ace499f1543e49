// E4M3 (FP8) encode and decode shared by the FP8 append and the fused FP8
// append + decode, so both store bit-identical codes.
//
// "PagedAttention" (deepconcepts.dev), section "Checking it on a real
// system", names FP8 KV as a way to change the bytes per token; the format
// used here is E4M3 with one float scale per KV head: code c stands for
// e4m3(c) * scale[head], and a new element x is stored as the nearest E4M3
// value (ties to even, saturating at 448) of the binary32 quotient x / scale.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace pkv {

// Two binary32 values to two E4M3 codes (round to nearest even, saturating);
// lo lands in the lower byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tmov.b16 %0, t;\n\t}"
        : "=h"(d)
        : "f"(hi), "f"(lo));
    return d;
}

// Eight fp16 values (one 16-byte vector) to eight codes (8 bytes).
__device__ __forceinline__ uint2 quantize8(uint4 x, float s) {
    const __half2* h = reinterpret_cast<const __half2*>(&x);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        w[i] = e4m3x2(__fdiv_rn(f.x, s), __fdiv_rn(f.y, s));
    }
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// Four codes (one 32-bit word, code 0 in the lowest byte) to four fp16
// values, exactly (every E4M3 value is an fp16 value): lo holds codes 0, 1,
// hi codes 2, 3.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Eight codes to eight fp16 values (one 16-byte vector).
__device__ __forceinline__ uint4 widen8(uint2 c) {
    uint4 r;
    widen4(c.x, r.x, r.y);
    widen4(c.y, r.z, r.w);
    return r;
}

}  // namespace pkv
