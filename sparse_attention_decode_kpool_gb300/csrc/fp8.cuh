// The FP8 latent cache's codec on the device: OCP E4M3 codes with one power-of-two
// scale 2^k per token and 128-channel group (see dsa_quantize_latent in dsa.h). Shared
// by the cache encoder and the decode-time append, so both store the same bytes, and
// by the attention kernels that decode the cache.
#pragma once

#include "common.cuh"

namespace dsa {

// k for a group's largest magnitude (amax >= 0, finite): the smallest integer with
// amax <= 448 * 2^k, not below -126; 0 for an all-zero group.
__device__ __forceinline__ int fp8_scale_exp(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    if (bits == 0u) return 0;
    const int E = (int)(bits >> 23);
    if (E == 0) return -126;  // below 2^-126: the clamp
    const uint32_t mant = bits & 0x7fffffu;
    // amax = m * 2^e with m in [1, 2): amax <= 448 * 2^k  <=>  m * 2^(e-k) <= 1.75 * 2^8
    const int e = E - 127;
    const int k = mant <= 0x600000u ? e - 8 : e - 7;
    return k < -126 ? -126 : k;
}

// Two E4M3 codes (low byte first) times a power-of-two scale, as packed bf16: the
// E4M3 -> f16 conversion, the f16 -> f32 widening and the scaling are exact, and so
// is the bf16 rounding (an E4M3 value times 2^k has a 4-bit significand).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two, float scale) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)(two & 0xffffu)));
    float f0, f1;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f0) : "h"((unsigned short)(h2 & 0xffffu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(f1) : "h"((unsigned short)(h2 >> 16)));
    return pack_bf16x2(f0 * scale, f1 * scale);
}

// Two values to E4M3 codes (nearest, ties to even, saturating), low byte first.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// One warp encodes one 128-channel group: src (bf16, 16-byte aligned) -> 128 codes
// and the group's scale. Lane l takes channels 4l .. 4l+3.
__device__ __forceinline__ void fp8_encode_group(const uint16_t* src, uint8_t* codes, float* scale,
                                                 int lane) {
    const uint2 v = *reinterpret_cast<const uint2*>(src + lane * 4);
    const float f0 = bf16_lo(v.x), f1 = bf16_hi(v.x), f2 = bf16_lo(v.y), f3 = bf16_hi(v.y);
    float m = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int k = fp8_scale_exp(m);
    const float inv = __uint_as_float((uint32_t)(127 - k) << 23);  // 2^-k, exact
    const uint32_t c = e4m3x2(f0 * inv, f1 * inv) | (e4m3x2(f2 * inv, f3 * inv) << 16);
    *reinterpret_cast<uint32_t*>(codes + lane * 4) = c;
    if (lane == 0) *scale = __uint_as_float((uint32_t)(k + 127) << 23);
}

}  // namespace dsa
