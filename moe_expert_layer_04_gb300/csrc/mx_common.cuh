// mx_common.cuh -- MXFP8 helpers shared by the quantiser and the MX GEMMs.
//
// Format: OCP Microscaling Formats (MX) v1.0 with FP8 E4M3 elements.  A
// block is 32 consecutive elements along the contraction; its E8M0 scale code
// c stands for X = 2^(c - 127).  E4M3 (OCP FP8): sign, 4 exponent bits with
// bias 7, 3 mantissa bits, no infinities, largest finite 448, subnormal
// quantum 2^-9.  A block is quantised with X = 2^(floor(log2 amax) - 8)
// (8 = exponent of E4M3's largest normal, clamped to [-127, 127]) and
// elements v / X rounded to the nearest E4M3 value, ties to even, saturating
// at 448.  ("DeepSeek-V4昇腾训练支持：基于 CANN 平台的TorchTitan-NPU + AutoFuse
// 极简训练优化实践", 性能结果与未来展望: FP8 training on MxFP8 compute.)
#pragma once

#include <cstdint>

namespace moe {

// Bytes per row of an MX scale matrix for a contraction of K elements: K / 32
// codes, padded to a multiple of 16 bytes (TMA rows).
__host__ __device__ inline int mx_sf_pitch(int K) { return ((K / 32) + 15) / 16 * 16; }

// floor(log2(a)) of a finite fp32 a > 0 (normal or subnormal), from its bits.
__device__ __forceinline__ int floor_log2_f32(float a) {
    const uint32_t b = __float_as_uint(a);
    const int e = (int)(b >> 23);
    if (e > 0) return e - 127;
    return (31 - __clz(b & 0x7FFFFFu)) - 149;
}

// E8M0 code of the scale of a block whose largest magnitude is amax.
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
    if (!(amax > 0.0f)) return 0u;
    int se = floor_log2_f32(amax) - 8;
    se = se < -127 ? -127 : (se > 127 ? 127 : se);
    return (uint32_t)(se + 127);
}

// 2^p for p in [-127, 127] (2^-127 is an fp32 subnormal).
__device__ __forceinline__ float exp2_int(int p) {
    return p >= -126 ? __uint_as_float((uint32_t)(p + 127) << 23) : __uint_as_float(0x00400000u);
}

// X = 2^(code - 127) and 1 / X.
__device__ __forceinline__ float mx_scale(uint32_t code) { return exp2_int((int)code - 127); }
__device__ __forceinline__ float mx_inv_scale(uint32_t code) { return exp2_int(127 - (int)code); }

// Quantises 32 fp32 values (one block) into 8 words of E4M3 codes (element i
// in byte i % 4 of word i / 4) and returns the block's E8M0 scale code.  The
// element codes come from the hardware conversion (cvt.rn.satfinite: nearest
// value, ties to even, magnitudes saturating at 448, the sign kept for values
// that round to zero), which is the rounding rule above.
__device__ __forceinline__ uint32_t mx_quantize_block(const float (&v)[32], uint32_t (&w)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t code = mx_scale_code(amax);
    const float inv = mx_inv_scale(code);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint16_t a, b;   // first operand -> high byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
            : "=h"(a) : "f"(v[4 * j + 1] * inv), "f"(v[4 * j] * inv));
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
            : "=h"(b) : "f"(v[4 * j + 3] * inv), "f"(v[4 * j + 2] * inv));
        w[j] = (uint32_t)a | ((uint32_t)b << 16);
    }
    return code;
}

}  // namespace moe
