// gemv_helpers.cuh -- element helpers of the small-M kernels (M <= 16): E2M1 code pairs
// to f16, mixed f16 x f16 -> f32 FMAs, the per-row power-of-two rescale that carries bf16
// x as fp16 (exact for every value within 2^31 of the row maximum, with an exact fp32
// residual for the rest), and the y store.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "common.cuh"

namespace nvfp4 {

// two codes (one byte, element 2i in the low nibble) -> f16x2
__device__ __forceinline__ uint32_t cvt2(uint32_t byte_in_low_bits) {
    uint32_t h;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n"
        : "=r"(h)
        : "r"(byte_in_low_bits));
    return h;
}

// p0 += lo(v) * lo(x); p1 += hi(v) * hi(x), fp16 products accumulated in fp32.
__device__ __forceinline__ void mfma2(float& p0, float& p1, uint32_t v, uint32_t x) {
    asm("{\n .reg .f16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %3;\n"
        " fma.rn.f32.f16 %0, a0, b0, %0;\n fma.rn.f32.f16 %1, a1, b1, %1;\n}\n"
        : "+f"(p0), "+f"(p1)
        : "r"(v), "r"(x));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// E4M3 byte -> f16x2 with the value in both halves (exact: E4M3 is a subset of f16).
__device__ __forceinline__ uint32_t e4m3_to_h2(uint32_t b) {
    const __half h = __float2half_rn(e4m3_to_f32(b));
    const uint32_t u = __half_as_ushort(h);
    return u | (u << 16);
}

__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
    const uint32_t m = code & 7u;
    const float v = m < 4u ? 0.5f * (float)m : (m == 7u ? 6.0f : (float)m - 2.0f);
    return (code & 8u) ? -v : v;
}

// W4A4 with the activation scale g fused into the small-M kernels: the 32 bf16 values of a
// lane's chunk of x (two 16-element blocks) are quantized to NVFP4 with g, as the
// quantizer would, and replaced by e2m1(code) * e4m3(scale).  bf16 holds those exactly (at
// most 5 significant bits, magnitudes in [2^-10, 2688]); g stays out of them and in y's
// scale.  quantize_chunk_codes also returns the chunk's encoding: codes[0..3] the 32 E2M1
// codes in the packed byte order (block 0: codes[0..1], block 1: codes[2..3]) and s2 the
// two block scale bytes (block 0 in the low byte).
__device__ __forceinline__ void quantize_chunk_codes(uint4 (&v)[4], float g, uint32_t (&codes)[4],
                                                     uint32_t& s2) {
    s2 = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float t[16];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t w[4] = {v[2 * h + q].x, v[2 * h + q].y, v[2 * h + q].z, v[2 * h + q].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                t[8 * q + 2 * j] = bf16_to_f32(w[j] & 0xFFFFu);
                t[8 * q + 2 * j + 1] = bf16_to_f32(w[j] >> 16);
            }
        }
        uint32_t lo, hi;
        const uint32_t s8 = quantize_block16(t, g, lo, hi);
        codes[2 * h] = lo;
        codes[2 * h + 1] = hi;
        s2 |= s8 << (8 * h);
        const float s = e4m3_to_f32(s8);
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            // elements 2j and 2j + 1: nibbles 2j, 2j + 1 of lo (j < 4) or hi
            const uint32_t w = j < 4 ? lo : hi;
            const float a = __fmul_rn(e2m1_to_f32((w >> (8 * (j & 3))) & 15u), s);
            const float b = __fmul_rn(e2m1_to_f32((w >> (8 * (j & 3) + 4)) & 15u), s);
            o[j] = (uint32_t)f32_to_bf16_rne(a) | ((uint32_t)f32_to_bf16_rne(b) << 16);
        }
        v[2 * h] = make_uint4(o[0], o[1], o[2], o[3]);
        v[2 * h + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

__device__ __forceinline__ void quantize_chunk_static(uint4 (&v)[4], float g) {
    uint32_t codes[4], s2;
    quantize_chunk_codes(v, g, codes, s2);
}

// exponent e with amax * 2^e in [2^14, 2^15) (0 for amax == 0)
__device__ __forceinline__ int chunk_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int E;
    frexpf(amax, &E);
    return 15 - E;
}

// exact v * 2^e for |e| <= 252, as two power-of-two factors of the same sign (the
// intermediate never leaves the range the final value is in); a chunk exponent lies in
// [-114, 148]
__device__ __forceinline__ float times_pow2(float v, int e) {
    const int e1 = e / 2, e2 = e - e / 2;
    return v * __int_as_float((e1 + 127) << 23) * __int_as_float((e2 + 127) << 23);
}

__device__ __forceinline__ uint32_t to_h2_scaled(uint32_t bf16x2, int e, bool& inexact) {
    const float a = times_pow2(bf16_to_f32(bf16x2 & 0xFFFFu), e);
    const float b = times_pow2(bf16_to_f32(bf16x2 >> 16), e);
    const __half ha = __float2half_rn(a), hb = __float2half_rn(b);
    inexact |= (__half2float(ha) != a) | (__half2float(hb) != b);
    return (uint32_t)__half_as_ushort(ha) | ((uint32_t)__half_as_ushort(hb) << 16);
}

// residual x' - fp16(x') of one bf16 element, exact in fp32
__device__ __forceinline__ float residual(uint32_t bf16bits, int e) {
    const float a = times_pow2(bf16_to_f32(bf16bits), e);
    return a - __half2float(__float2half_rn(a));
}

__device__ __forceinline__ void store_y(void* y, int64_t o, float v, int y_bf16) {
    if (y_bf16) static_cast<uint16_t*>(y)[o] = f32_to_bf16_rne(v);
    else static_cast<float*>(y)[o] = v;
}

}  // namespace nvfp4
