// quantize_mxfp8.cu -- A6: grouped MXFP8 quantisation (E4M3 + UE8M0 per 1x32 block
// along K) of activations and of expert weights.
//
// Activations: one warp per row, one 32-element block per lane per step
// (64-byte loads, 32-byte stores).  Scales go to a row-major array and/or to
// the MMA tile layout of the row's group (mx.cuh), whose tile ids follow the
// group offsets.  Weights [E, K, N] (N contiguous) are quantised along K and
// written K-contiguous as [E, N, K] with tile-layout scales, through a shared
// memory transpose.  ("Add MoE + expert-parallel Python API surface, PyTorch
// reference, and tests", BlockScaledTensor: block size 32 for mxfp8; "MoE
// training optimization": grouped quantize with device-side group sizes,
// scale swizzle fused into the quantiser.)
#include "common.cuh"
#include "mx.cuh"

namespace moe {

// mtile_start[g] = sum over groups g' < g of ceil(rows(g') / 128); [G+1] entries.
__global__ void mtile_prefix_kernel(const int32_t *__restrict__ group_offsets, int G, int32_t *__restrict__ mtile_start) {
    pdl_wait();
    __shared__ int32_t s_warp[32];
    const int g = threadIdx.x, lane = g & 31, warp = g >> 5;
    int t = 0;
    if (g < G) {
        const int rows = group_offsets[g + 1] - group_offsets[g];
        t = rows > 0 ? (rows + 127) / 128 : 0;
    }
    int incl = t;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = s_warp[lane];
        int vi = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, vi, off);
            if (lane >= off) vi += o;
        }
        s_warp[lane] = vi - v;
    }
    __syncthreads();
    const int excl = incl - t + s_warp[warp];
    if (g < G) mtile_start[g] = excl;
    if (g == G - 1) mtile_start[G] = excl + t;
}

namespace {

constexpr int kQWarps = 8;

__device__ __forceinline__ void load32_bf16(const uint4 *src, float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 p = __ldg(src + q);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&p);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            v[8 * q + 2 * i] = f.x;
            v[8 * q + 2 * i + 1] = f.y;
        }
    }
}

// Group of `row` (largest g with group_offsets[g] <= row), or -1 past the last group.
__device__ __forceinline__ int group_of(const int32_t *go, int G, int64_t row) {
    if (row >= go[G]) return -1;
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (go[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kQWarps * 32)
quantize_rows_kernel(const __nv_bfloat16 *__restrict__ in, int64_t rows, int K,
                     const int32_t *__restrict__ group_offsets, int G, const int32_t *__restrict__ mtile_start,
                     uint8_t *__restrict__ data, uint8_t *__restrict__ scale_rm, uint8_t *__restrict__ scale_tiles) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kQWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int nb = K / 32;
    int64_t tile = -1;
    int m = 0;
    if (scale_tiles) {
        const int g = group_of(group_offsets, G, row);
        if (g >= 0) {
            const int64_t i = row - group_offsets[g];
            tile = mtile_start[g] + i / 128;
            m = (int)(i % 128);
        }
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(in + row * K);
    uint4 *dst = reinterpret_cast<uint4 *>(data + row * K);
    for (int b = lane; b < nb; b += 32) {
        float v[32];
        load32_bf16(src + b * 4, v);
        const int X = mx::scale_exp(mx::amax32(v));
        uint4 lo, hi;
        mx::quantize32(v, X, lo, hi);
        dst[2 * b] = lo;
        dst[2 * b + 1] = hi;
        const uint8_t byte = (uint8_t)(X + 127);
        if (scale_rm) scale_rm[row * nb + b] = byte;
        if (tile >= 0) scale_tiles[mx::tile_sf_offset(tile, K / 128, m, b)] = byte;
    }
}

// Weights: W[e] is [K, N] (N contiguous).  Block (e, n-tile of 64, k-block of 32):
// stage [32][64] bf16 in smem, each of 64 threads quantises one column's 32 values,
// writes the 32 codes of (n, k..k+32) and one scale byte.  Codes go to the tiled
// layout: for every (expert, 128 K bytes, 128 rows n) one contiguous 16 KB block of
// 128 rows x 128 bytes, 16-byte chunk j of row r stored at chunk j ^ (r % 8) (the
// 128-byte swizzle of the MMA's K-major operand), blocks ordered [E][K/128][N/128].
__global__ void __launch_bounds__(64)
quantize_weights_kernel(const __nv_bfloat16 *__restrict__ W, int K, int N, uint8_t *__restrict__ data,
                        uint8_t *__restrict__ scales) {
    pdl_wait();
    __shared__ float tileS[32][65];
    const int n0 = blockIdx.x * 64, kb = blockIdx.y, e = blockIdx.z;
    const __nv_bfloat16 *src = W + ((int64_t)e * K + (int64_t)kb * 32) * N + n0;
    const int t = threadIdx.x;
    for (int r = 0; r < 32; ++r) tileS[r][t] = __bfloat162float(src[(int64_t)r * N + t]);
    __syncthreads();
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = tileS[i][t];
    const int X = mx::scale_exp(mx::amax32(v));
    uint4 lo, hi;
    mx::quantize32(v, X, lo, hi);
    const int n = n0 + t;
    // atoms and code blocks ordered [e][K/128][N/128], tile row = n % 128
    const int64_t atom = ((int64_t)e * (K / 128) + kb / 4) * (N / 128) + n / 128;
    const int m = n % 128;
    uint8_t *blk = data + atom * 16384 + m * 128;
    const int c0 = (kb % 4) * 2;   // the two 16-byte chunks of this 32-code run
    *reinterpret_cast<uint4 *>(blk + ((c0 ^ (m % 8)) * 16)) = lo;
    *reinterpret_cast<uint4 *>(blk + (((c0 + 1) ^ (m % 8)) * 16)) = hi;
    scales[atom * 512 + (m % 32) * 16 + (m / 32) * 4 + (kb % 4)] = (uint8_t)(X + 127);
}

}  // namespace

cudaError_t launch_quantize_rows(const __nv_bfloat16 *in, int64_t rows, int K, const int32_t *group_offsets, int G,
                                 const int32_t *mtile_start, uint8_t *data, uint8_t *scale_rm, uint8_t *scale_tiles,
                                 cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    const int64_t blocks = (rows + kQWarps - 1) / kQWarps;
    launch_k(quantize_rows_kernel, dim3((unsigned)blocks), dim3(kQWarps * 32), 0, s, in, rows, K, group_offsets, G,
             mtile_start, data, scale_rm, scale_tiles);
    return cudaGetLastError();
}

}  // namespace moe

extern "C" moe_status_t moe_grouped_quantize_mxfp8(const moe_bf16_t *in, int64_t rows, int K,
                                                   const int32_t *group_offsets, int G, uint8_t *data,
                                                   uint8_t *scale_rowmajor, uint8_t *scale_tiles, void *ws,
                                                   size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_quantize_mxfp8");
    using namespace moe;
    if (rows < 0 || K < 1) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0 || rows >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!in || !data || (!scale_rowmajor && !scale_tiles)) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({in, data})) return MOE_ERR_UNSUPPORTED;
    if (scale_tiles && (!group_offsets || G < 1 || G > 1024)) return MOE_ERR_INVALID_ARG;
    if (scale_tiles && (!ws || ws_bytes < kWsHeaderBytes + (size_t)(G + 1) * sizeof(int32_t))) return MOE_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t *mtile = nullptr;
    if (scale_tiles) {
        mtile = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kWsHeaderBytes);
        launch_k(mtile_prefix_kernel, dim3(1), dim3(1024), 0, s, group_offsets, G, mtile);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    return cuda_status(launch_quantize_rows(reinterpret_cast<const __nv_bfloat16 *>(in), rows, K, group_offsets, G,
                                            mtile, data, scale_rowmajor, scale_tiles, s));
}

extern "C" moe_status_t moe_quantize_weights_mxfp8(const moe_bf16_t *W, int E, int K, int N, uint8_t *data,
                                                   uint8_t *scales, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_quantize_weights_mxfp8");
    if (E < 1 || K < 1 || N < 1) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0 || E > 65535 || K / 32 > 65535) return MOE_ERR_UNSUPPORTED;
    if (!W || !data || !scales) return MOE_ERR_INVALID_ARG;
    if (!moe::all_aligned16({data})) return MOE_ERR_UNSUPPORTED;   // 16-byte stores of the code blocks
    dim3 grid(N / 64, K / 32, E);
    moe::launch_k(moe::quantize_weights_kernel, grid, dim3(64), 0, (cudaStream_t)stream,
                  reinterpret_cast<const __nv_bfloat16 *>(W), K, N, data, scales);
    return moe::launch_status();
}
