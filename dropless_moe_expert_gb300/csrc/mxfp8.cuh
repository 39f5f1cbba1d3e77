// MXFP8 block quantiser and scale-atom addressing, shared by the
// quantisation kernels and the GEMM1 epilogue (which quantises h).
// Format and layout: see mxfp8.cu.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {
namespace mx {

// Scale byte e + 127 of a block whose largest magnitude is amax (>= 0): e is
// the smallest exponent with 448 * 2^e >= amax (for amax = m 2^E with
// 1 <= m < 2: E - 8, or E - 7 when m > 1.75); zero and fp32-subnormal maxima
// give e = -127.
__device__ __forceinline__ uint32_t scale_byte(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    const int be = static_cast<int>(bits >> 23);
    int e = be == 0 ? -127 : (be - 127) - 8 + ((bits & 0x7fffffu) > 0x600000u ? 1 : 0);
    e = max(e, -127);
    return static_cast<uint32_t>(e + 127);
}

// Four values (already divided by the block scale) -> four E4M3 codes,
// little-endian, rounded to nearest even.
__device__ __forceinline__ uint32_t pack4(float a, float b, float c, float d) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// 32 fp32 values -> 32 E4M3 codes packed little-endian in 8 words; returns
// the scale byte.
__device__ __forceinline__ uint32_t quant_block(const float (&v)[32], uint32_t (&packed)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t s = scale_byte(amax);
    const float inv = __uint_as_float((254u - s) << 23);  // 2^-(s-127), exact
#pragma unroll
    for (int w = 0; w < 8; ++w) packed[w] = pack4(v[4 * w] * inv, v[4 * w + 1] * inv, v[4 * w + 2] * inv, v[4 * w + 3] * inv);
    return s;
}

__device__ __forceinline__ size_t atom_word(int rb, int ks, int nslices, int i) {
    // byte offset of row i (0..127) of atom (rb, ks), as a 4-byte word index
    return (static_cast<size_t>(rb) * nslices + ks) * 128 + (i & 31) * 4 + (i >> 5);
}

}  // namespace mx
}  // namespace moe
