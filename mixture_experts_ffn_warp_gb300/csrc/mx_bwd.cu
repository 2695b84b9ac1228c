// mx_bwd.cu -- the MXFP8 path's operands for the backward: dequantisation of
// MXFP8 rows (tile-layout scales) and of the pre-tiled expert weights to bf16.
//
// The backward of the MXFP8 forward is straight-through: every quantisation
// round trip has derivative identity ("Add MoE + expert-parallel Python API
// surface, PyTorch reference, and tests", Summary: quantization round-trips are
// straight-through).  Its GEMMs are therefore the bf16 backward's, run on the
// values the forward's block-scaled MMAs consumed: x, h and the weights as
// E4M3 code * 2^(scale - 127).  An E4M3 value times a power of two has at most
// 4 significant bits, so bf16 holds it exactly whenever its exponent is in
// bf16's range (|v| >= 2^-133); smaller values flush to zero, larger ones
// cannot occur (448 * 2^127 is the largest).
#include "common.cuh"
#include "mx.cuh"

namespace moe {
namespace {

constexpr int kDqWarps = 8;

// 2^X as a float for X in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int X) {
    return X >= -126 ? __uint_as_float((uint32_t)(X + 127) << 23) : __uint_as_float(0x00400000u);
}

// 8 E4M3 codes (two words) times 2^X -> 8 bf16 (one 16-byte word).
__device__ __forceinline__ uint4 dequant8(uint2 codes, float scale) {
    uint4 out;
    __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(&out);
    const uint32_t w[2] = {codes.x, codes.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> (16 * h)), __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r));
            o[2 * i + h] = __floats2bfloat162_rn(f.x * scale, f.y * scale);
        }
    }
    return out;
}

// Largest g with go[g] <= row, or -1 past the last group's end.
__device__ __forceinline__ int group_of_row(const int32_t *go, int G, int64_t row) {
    if (row >= go[G]) return -1;
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (go[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// One warp per row: each lane a 32-element block per step (32 code bytes in, 64 bf16
// bytes out) with the block's scale from the tile layout of the row's group.  Rows
// past the last group are written as zeros.
__global__ void __launch_bounds__(kDqWarps * 32)
dequantize_rows_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ tile_sf,
                       const int32_t *__restrict__ group_offsets, int G, const int32_t *__restrict__ mtile_start,
                       int64_t rows, int K, __nv_bfloat16 *__restrict__ out) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kDqWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int nb = K / 32;
    uint4 *dst = reinterpret_cast<uint4 *>(out + row * K);
    const int g = group_of_row(group_offsets, G, row);
    if (g < 0) {
        for (int b = lane; b < nb; b += 32)
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[4 * b + q] = make_uint4(0, 0, 0, 0);
        return;
    }
    const int64_t i = row - group_offsets[g];
    const int64_t tile = mtile_start[g] + i / 128;
    const int m = (int)(i % 128);
    const uint4 *src = reinterpret_cast<const uint4 *>(codes + row * K);
    for (int b = lane; b < nb; b += 32) {
        const uint4 lo = __ldg(src + 2 * b), hi = __ldg(src + 2 * b + 1);
        const float sc = pow2f((int)tile_sf[mx::tile_sf_offset(tile, K / 128, m, b)] - 127);
        dst[4 * b + 0] = dequant8(make_uint2(lo.x, lo.y), sc);
        dst[4 * b + 1] = dequant8(make_uint2(lo.z, lo.w), sc);
        dst[4 * b + 2] = dequant8(make_uint2(hi.x, hi.y), sc);
        dst[4 * b + 3] = dequant8(make_uint2(hi.z, hi.w), sc);
    }
}

// Weights: the inverse of the weight quantiser's layout.  Block (n-tile of 64, k-block
// of 32, expert e), one thread per column n: its 32 codes (two swizzled 16-byte chunks of
// row n % 128 of the 16 KB code block) and its scale byte, dequantised into a shared
// [32][64] tile, written back row by row as W[e][k][n] (N contiguous).
__global__ void __launch_bounds__(64)
dequantize_weights_kernel(const uint8_t *__restrict__ data, const uint8_t *__restrict__ scales, int K, int N,
                          __nv_bfloat16 *__restrict__ W) {
    pdl_wait();
    __shared__ __nv_bfloat16 tileS[32][64 + 2];
    const int n0 = blockIdx.x * 64, kb = blockIdx.y, e = blockIdx.z;
    const int t = threadIdx.x, n = n0 + t, m = n % 128;
    const int64_t atom = ((int64_t)e * (K / 128) + kb / 4) * (N / 128) + n / 128;
    const uint8_t *blk = data + atom * 16384 + m * 128;
    const int c0 = (kb % 4) * 2;
    const uint4 lo = *reinterpret_cast<const uint4 *>(blk + ((c0 ^ (m % 8)) * 16));
    const uint4 hi = *reinterpret_cast<const uint4 *>(blk + (((c0 + 1) ^ (m % 8)) * 16));
    const float sc = pow2f((int)scales[atom * 512 + (m % 32) * 16 + (m / 32) * 4 + (kb % 4)] - 127);
    uint4 v[4] = {dequant8(make_uint2(lo.x, lo.y), sc), dequant8(make_uint2(lo.z, lo.w), sc),
                  dequant8(make_uint2(hi.x, hi.y), sc), dequant8(make_uint2(hi.z, hi.w), sc)};
    const __nv_bfloat16 *vb = reinterpret_cast<const __nv_bfloat16 *>(v);
#pragma unroll
    for (int r = 0; r < 32; ++r) tileS[r][t] = vb[r];
    __syncthreads();
    __nv_bfloat16 *dst = W + ((int64_t)e * K + (int64_t)kb * 32) * N + n0;
    for (int r = 0; r < 32; ++r) dst[(int64_t)r * N + t] = tileS[r][t];
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_dequantize_rows_mxfp8(const uint8_t *codes, const uint8_t *tile_scales,
                                                  const int32_t *group_offsets, int G, int64_t rows, int K,
                                                  moe_bf16_t *out, void *ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_dequantize_rows_mxfp8");
    using namespace moe;
    if (rows < 0 || K < 1 || G < 1) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0 || G > 1024 || rows >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!codes || !tile_scales || !group_offsets || !out) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(codes) % 16 || reinterpret_cast<uintptr_t>(out) % 16) return MOE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < kWsHeaderBytes + (size_t)(G + 1) * sizeof(int32_t)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t *mtile = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kWsHeaderBytes);
    launch_k(mtile_prefix_kernel, dim3(1), dim3(1024), 0, s, group_offsets, G, mtile);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    const int64_t blocks = (rows + kDqWarps - 1) / kDqWarps;
    launch_k(dequantize_rows_kernel, dim3((unsigned)blocks), dim3(kDqWarps * 32), 0, s, codes, tile_scales,
             group_offsets, G, mtile, rows, K, reinterpret_cast<__nv_bfloat16 *>(out));
    return launch_status();
}

extern "C" moe_status_t moe_dequantize_weights_mxfp8(const uint8_t *data, const uint8_t *scales, int E, int K, int N,
                                                     moe_bf16_t *W, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_dequantize_weights_mxfp8");
    using namespace moe;
    if (E < 1 || K < 1 || N < 1) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0 || E > 65535 || K / 32 > 65535) return MOE_ERR_UNSUPPORTED;
    if (!data || !scales || !W) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(data) % 16) return MOE_ERR_UNSUPPORTED;
    dim3 grid(N / 64, K / 32, E);
    launch_k(dequantize_weights_kernel, grid, dim3(64), 0, (cudaStream_t)stream, data, scales, K, N,
             reinterpret_cast<__nv_bfloat16 *>(W));
    return launch_status();
}
