// dequant.cuh -- record-field conversions and shared-memory addressing used by the decode kernels
// that dequantize NVFP4 records into 16-bit MMA operand tiles.
//
// An NVFP4 value is an e2m1 code times the e4m3 scale of its 16-value block; the product has at
// most five significant bits and lies in [2^-10, 2688] (or is zero), so it is exact in f16 and in
// bf16 and every conversion below is exact.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace nvfp4mla {

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128B-swizzled tile of 128-byte
// rows (the canonical SWIZZLE_128B operand layout: 8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// e4m3 scale byte -> (s, s) as f16x2 (exact).
__device__ __forceinline__ __half2 scale_half2(uint32_t sbyte) {
    uint32_t h;
    const uint16_t in = static_cast<uint16_t>(sbyte | (sbyte << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    return *reinterpret_cast<__half2*>(&h);
}

// Eight e2m1 codes (one word, low nibble first) times a scale -> four f16x2 words (exact).
__device__ __forceinline__ uint4 dq8(uint32_t w, __half2 s2) {
    uint32_t h[4];
    asm("{\n"
        "  .reg .b8 a, b, c, d;\n"
        "  mov.b32 {a, b, c, d}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, a;\n"
        "  cvt.rn.f16x2.e2m1x2 %1, b;\n"
        "  cvt.rn.f16x2.e2m1x2 %2, c;\n"
        "  cvt.rn.f16x2.e2m1x2 %3, d;\n"
        "}\n"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&h[k]), s2);
        h[k] = *reinterpret_cast<const uint32_t*>(&p);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

// Four e4m3 codes -> two f16x2 words (exact).
__device__ __forceinline__ uint2 e4m3x4_to_f16(uint32_t w) {
    uint32_t a, b;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(a) : "h"(static_cast<uint16_t>(w)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b) : "h"(static_cast<uint16_t>(w >> 16)));
    return make_uint2(a, b);
}

// Byte q of each word of w, low word first.
__device__ __forceinline__ uint32_t gather_byte4(const uint4& w, int q) {
    const uint32_t sel = static_cast<uint32_t>(q) | (static_cast<uint32_t>(q + 4) << 4);
    return __byte_perm(__byte_perm(w.x, w.y, sel), __byte_perm(w.z, w.w, sel), 0x5410);
}

}  // namespace nvfp4mla
