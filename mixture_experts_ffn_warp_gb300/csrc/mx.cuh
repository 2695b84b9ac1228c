// mx.cuh -- MXFP8 (E4M3 elements, one UE8M0 scale per 32-element block along K)
// helpers shared by the quantisers, the quantising permute and the MXFP8 GEMM.
//
// Scale rule: the smallest power of two 2^X with amax / 2^X <= 448 (E4M3's
// largest finite value): X = floor(log2 amax) - 8, plus 1 when amax's
// significand exceeds 1.75; clamped to [-127, 127]; the stored byte is X + 127
// (amax = 0 -> byte 0).  Elements are v / 2^X rounded to nearest even onto
// E4M3 with saturation (the hardware cvt.rn.satfinite conversion).
//
// Scale layouts:
//   row-major   scale[row][K/32]
//   tile layout the operand layout of the block-scaled MMA: for every 128-row
//               tile and every 128-element K block one 512-byte atom, byte
//               (m % 32) * 16 + (m / 32) * 4 + (kb % 4) for tile row m and
//               32-block kb; atoms ordered [tile][K/128].  Weights use
//               [expert][K/128][N/128] atoms with m = the output column n.
//               A tcgen05.cp.32x128b.warpx4 of one atom gives the MMA row m's
//               scales in TMEM lane m, column m / 32, byte = scale id.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {
namespace mx {

// UE8M0 exponent X of a block with maximum magnitude amax (finite, >= 0).
__device__ __forceinline__ int scale_exp(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int e = (int)((b >> 23) & 0xFF);
    if (e == 0) return -127;                       // zero or subnormal amax: clamp
    int X = e - 127 - 8 + ((b & 0x7FFFFF) > 0x600000 ? 1 : 0);   // significand > 1.75
    return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// 2^-X as a float, X in [-127, 126].
__device__ __forceinline__ float inv_pow2(int X) { return __uint_as_float((uint32_t)(127 - X) << 23); }

// Quantise 32 values to E4M3 with block exponent X; packs 32 bytes.
__device__ __forceinline__ void quantize32(const float (&v)[32], int X, uint4 &lo, uint4 &hi) {
    const float s = inv_pow2(X);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __nv_fp8x2_storage_t p0 =
            __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * s, v[4 * i + 1] * s), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t p1 =
            __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * s, v[4 * i + 3] * s), __NV_SATFINITE, __NV_E4M3);
        w[i] = (uint32_t)p0 | ((uint32_t)p1 << 16);
    }
    lo = make_uint4(w[0], w[1], w[2], w[3]);
    hi = make_uint4(w[4], w[5], w[6], w[7]);
}

// Quantise 8 values to E4M3 with block exponent X (a quarter of a block); packs 8 bytes.
__device__ __forceinline__ uint2 quantize8(const float (&v)[8], int X) {
    const float s = inv_pow2(X);
    uint32_t w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const __nv_fp8x2_storage_t p0 =
            __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * s, v[4 * i + 1] * s), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t p1 =
            __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * s, v[4 * i + 3] * s), __NV_SATFINITE, __NV_E4M3);
        w[i] = (uint32_t)p0 | ((uint32_t)p1 << 16);
    }
    return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ float amax32(const float (&v)[32]) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
    return a;
}

// Byte offset of (tile row m, 32-block kb) within the atoms of one tile.
__host__ __device__ __forceinline__ int64_t tile_sf_offset(int64_t tile, int kblocks128, int m, int kb) {
    return (tile * kblocks128 + kb / 4) * 512 + (m % 32) * 16 + (m / 32) * 4 + (kb % 4);
}

}  // namespace mx
}  // namespace moe
