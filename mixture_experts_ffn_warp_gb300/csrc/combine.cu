// combine.cu -- A5: weighted unpermute / combine back to token order.
//
// One warp per token; each lane owns 8-column slices of the row (one 16-byte load
// of bf16 expert outputs per slot -- two of fp32 rows for the backward's
// unpermute-sum --, one 16-byte bf16 store) and accumulates w_j * y_perm[dst_j]
// over the k slots in slot order in fp32.  All slot loads
// of a slice are issued before the FMAs, and each lane keeps several slices
// in flight.  ("Add MoE + expert-parallel Python API surface, PyTorch
// reference, and tests", Summary: per-top-k combine.)
#include "common.cuh"
#include "mx.cuh"

namespace moe {
namespace {

constexpr int kCombineWarps = 8;

struct F8 {
    float4 a, b;
};

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const F8 &v) {
    acc[0] = fmaf(w, v.a.x, acc[0]);
    acc[1] = fmaf(w, v.a.y, acc[1]);
    acc[2] = fmaf(w, v.a.z, acc[2]);
    acc[3] = fmaf(w, v.a.w, acc[3]);
    acc[4] = fmaf(w, v.b.x, acc[4]);
    acc[5] = fmaf(w, v.b.y, acc[5]);
    acc[6] = fmaf(w, v.b.z, acc[6]);
    acc[7] = fmaf(w, v.b.w, acc[7]);
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
    uint4 r;
    __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    return r;
}

// An 8-column slice of a y_perm row as loaded (two 16-byte fp32 loads, or one 16-byte load of
// bf16 values, widened only at the FMA), and the slices each lane keeps in flight: as many
// bytes per lane for bf16 rows as for fp32 ones.
template <typename Y>
struct Slice;
template <>
struct Slice<float4> {
    using Raw = F8;
    template <int KMAX>
    static constexpr int kInFlight = KMAX <= 2 ? 4 : (KMAX <= 4 ? 2 : 1);
    __device__ static Raw load(const float4 *y, int64_t slice) {
        Raw v;
        v.a = __ldg(y + slice * 2);
        v.b = __ldg(y + slice * 2 + 1);
        return v;
    }
    __device__ static void fma(float (&acc)[8], float w, const Raw &v) { fma8(acc, w, v); }
};
template <>
struct Slice<uint4> {
    using Raw = uint4;
    template <int KMAX>
    static constexpr int kInFlight = KMAX <= 2 ? 8 : (KMAX <= 4 ? 4 : (KMAX <= 8 ? 2 : 1));
    __device__ static Raw load(const uint4 *y, int64_t slice) { return __ldg(y + slice); }
    __device__ static void fma(float (&acc)[8], float w, const Raw &raw) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p[i]);
            acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
        }
    }
};

// Y = uint4 (bf16 y_perm rows, the forward's combine) or float4 (fp32 rows: the
// backward's unpermute-sum of dx_perm).
template <int KMAX, typename Y>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const Y *__restrict__ y_perm, const int32_t *__restrict__ dst_of_route,
               const float *__restrict__ topk_w, int64_t T, int k, int slices,
               uint4 *__restrict__ out) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_dst = -1;
    float my_w = 0.0f;
    if (lane < k) {
        my_dst = dst_of_route[t * k + lane];
        my_w = topk_w ? topk_w[t * k + lane] : 1.0f;   // no weights: plain sum over the slots
    }
    int dst[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        dst[j] = __shfl_sync(0xFFFFFFFFu, my_dst, j);
        w[j] = __shfl_sync(0xFFFFFFFFu, my_w, j);
        if (j >= k) dst[j] = -1;
    }
    using S = Slice<Y>;
    constexpr int U = S::template kInFlight<KMAX>;   // slices in flight per lane
    for (int s0 = lane; s0 < slices; s0 += 32 * U) {
        typename S::Raw val[U][KMAX];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (dst[j] >= 0 && s0 + 32 * u < slices)
                    val[u][j] = S::load(y_perm, (int64_t)dst[j] * slices + s0 + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s0 + 32 * u >= slices) break;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (dst[j] >= 0) S::fma(acc, w[j], val[u][j]);
            out[t * slices + s0 + 32 * u] = pack8(acc);
        }
    }
}

template <int KMAX, typename Y>
cudaError_t launch(const Y *y, const int32_t *dst, const float *w, int64_t T, int k, int slices,
                   moe_bf16_t *out, cudaStream_t s) {
    const int64_t blocks = (T + kCombineWarps - 1) / kCombineWarps;
    launch_k(combine_kernel<KMAX, Y>, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s, y, dst, w, T, k,
             slices, reinterpret_cast<uint4 *>(out));
    return cudaGetLastError();
}

// As combine_kernel, with the output encoded as MXFP8 along H: four consecutive lanes hold
// the 32 columns of one block (8 each), take its maximum with two shuffles and quantise
// their fp32 sums; one lane in four writes the block's scale byte.  Every lane runs the
// shuffles (a block's lanes are all in range or all out, H % 32 == 0).
template <int KMAX>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_mx_kernel(const uint4 *__restrict__ y_perm, const int32_t *__restrict__ dst_of_route,
                  const float *__restrict__ topk_w, int64_t T, int k, int slices, uint2 *__restrict__ out_q,
                  uint8_t *__restrict__ out_sf) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_dst = -1;
    float my_w = 0.0f;
    if (lane < k) {
        my_dst = dst_of_route[t * k + lane];
        my_w = topk_w ? topk_w[t * k + lane] : 1.0f;
    }
    int dst[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        dst[j] = __shfl_sync(0xFFFFFFFFu, my_dst, j);
        w[j] = __shfl_sync(0xFFFFFFFFu, my_w, j);
        if (j >= k) dst[j] = -1;
    }
    for (int s0 = 0; s0 < slices; s0 += 32) {
        const int s = s0 + lane;
        const bool in = s < slices;
        uint4 val[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            if (in && dst[j] >= 0) val[j] = __ldg(y_perm + (int64_t)dst[j] * slices + s);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (in) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (dst[j] >= 0) Slice<uint4>::fma(acc, w[j], val[j]);
        }
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(acc[i]));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        const int X = mx::scale_exp(a);
        if (in) {
            out_q[t * slices + s] = mx::quantize8(acc, X);
            if ((lane & 3) == 0) out_sf[t * (slices / 4) + s / 4] = (uint8_t)(X + 127);
        }
    }
}

template <int KMAX>
cudaError_t launch_mx(const moe_bf16_t *y, const int32_t *dst, const float *w, int64_t T, int k, int slices,
                      uint8_t *out_q, uint8_t *out_sf, cudaStream_t s) {
    const int64_t blocks = (T + kCombineWarps - 1) / kCombineWarps;
    launch_k(combine_mx_kernel<KMAX>, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
             reinterpret_cast<const uint4 *>(y), dst, w, T, k, slices, reinterpret_cast<uint2 *>(out_q), out_sf);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- NVFP4 output
// E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; sign in bit 3) in blocks of 16
// along H with one E4M3 scale each: the smallest positive finite E4M3 value s with
// 6 s >= amax (448 past 6 * 448, byte 0 for an all-zero block), each element rounded to
// the nearest magnitude of |v| / s, ties to the even code.  Every decision compares fp32
// values that are exact: amax with 6 s, and |v| with s times a midpoint of the E2M1
// magnitudes (at most 7 significant bits).

// Value of a positive finite E4M3 code c in [1, 0x7E]: (8 + m) 2^(e - 10), or m 2^-9 for e = 0.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t e = c >> 3, m = c & 7u;
    return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
}

// Scale code of a block: smallest c in [1, 0x7E] with 6 * value(c) >= amax (binary search
// over the monotone codes); 0x7E if none; 0 for amax = 0.
__device__ __forceinline__ uint32_t nvfp4_scale_code(float amax) {
    if (!(amax > 0.0f)) return 0u;
    uint32_t lo = 1u, hi = 0x7Eu;
    while (lo < hi) {
        const uint32_t mid = (lo + hi) >> 1;
        if (6.0f * e4m3_value(mid) >= amax) hi = mid; else lo = mid + 1u;
    }
    return lo;
}

// 4-bit code of v at scale s > 0: the count of E2M1 midpoints that |v| / s passes, a value
// on a midpoint going to the even code (up at 0.75, 1.75, 3.5; down at 0.25, 1.25, 2.5, 5).
__device__ __forceinline__ uint32_t nvfp4_code(float v, float s) {
    const float a = fabsf(v);
    uint32_t c = (a > 0.25f * s) + (a >= 0.75f * s) + (a > 1.25f * s) + (a >= 1.75f * s) + (a > 2.5f * s) +
                 (a >= 3.5f * s) + (a > 5.0f * s);
    return c | (v < 0.0f ? 8u : 0u);
}

// As combine_kernel, with the output encoded as NVFP4 along H: two consecutive lanes hold
// the 16 columns of one block (8 each), take its maximum with one shuffle, and each packs
// its 8 codes into one 32-bit word (element order, low nibble first); the even lane writes
// the block's scale byte.  Every lane runs the shuffle (H % 16 == 0: a block's two lanes
// are both in range or both out).
template <int KMAX>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_nvfp4_kernel(const uint4 *__restrict__ y_perm, const int32_t *__restrict__ dst_of_route,
                     const float *__restrict__ topk_w, int64_t T, int k, int slices, uint32_t *__restrict__ out_q,
                     uint8_t *__restrict__ out_sf) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_dst = -1;
    float my_w = 0.0f;
    if (lane < k) {
        my_dst = dst_of_route[t * k + lane];
        my_w = topk_w ? topk_w[t * k + lane] : 1.0f;
    }
    int dst[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        dst[j] = __shfl_sync(0xFFFFFFFFu, my_dst, j);
        w[j] = __shfl_sync(0xFFFFFFFFu, my_w, j);
        if (j >= k) dst[j] = -1;
    }
    for (int s0 = 0; s0 < slices; s0 += 32) {
        const int s = s0 + lane;
        const bool in = s < slices;
        uint4 val[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            if (in && dst[j] >= 0) val[j] = __ldg(y_perm + (int64_t)dst[j] * slices + s);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (in) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (dst[j] >= 0) Slice<uint4>::fma(acc, w[j], val[j]);
        }
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(acc[i]));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        const uint32_t sc = nvfp4_scale_code(a);
        if (in) {
            uint32_t word = 0;
            if (sc) {
                const float sv = e4m3_value(sc);
#pragma unroll
                for (int i = 0; i < 8; ++i) word |= nvfp4_code(acc[i], sv) << (4 * i);
            }
            out_q[t * slices + s] = word;
            if ((lane & 1) == 0) out_sf[t * (slices / 2) + s / 2] = (uint8_t)sc;
        }
    }
}

template <int KMAX>
cudaError_t launch_nvfp4(const moe_bf16_t *y, const int32_t *dst, const float *w, int64_t T, int k, int slices,
                         uint8_t *out_q, uint8_t *out_sf, cudaStream_t s) {
    const int64_t blocks = (T + kCombineWarps - 1) / kCombineWarps;
    launch_k(combine_nvfp4_kernel<KMAX>, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
             reinterpret_cast<const uint4 *>(y), dst, w, T, k, slices, reinterpret_cast<uint32_t *>(out_q), out_sf);
    return cudaGetLastError();
}

}  // namespace

template <typename Y>
cudaError_t combine_rows_t(const Y *y, const int32_t *dst, const float *w, int64_t T, int H, int k,
                           moe_bf16_t *out, cudaStream_t s) {
    const int sl = H / 8;
    if (k <= 1) return launch<1>(y, dst, w, T, k, sl, out, s);
    if (k <= 2) return launch<2>(y, dst, w, T, k, sl, out, s);
    if (k <= 4) return launch<4>(y, dst, w, T, k, sl, out, s);
    if (k <= 8) return launch<8>(y, dst, w, T, k, sl, out, s);
    if (k <= 16) return launch<16>(y, dst, w, T, k, sl, out, s);
    return launch<32>(y, dst, w, T, k, sl, out, s);
}

cudaError_t combine_rows(const float *y, const int32_t *dst, const float *w, int64_t T, int H, int k,
                         moe_bf16_t *out, cudaStream_t s) {
    return combine_rows_t(reinterpret_cast<const float4 *>(y), dst, w, T, H, k, out, s);
}

}  // namespace moe

extern "C" moe_status_t moe_unpermute_combine(const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                              const float *topk_w, int64_t T, int H, int k,
                                              moe_bf16_t *out, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_unpermute_combine");
    if (T < 0 || H < 1) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!y_perm || !dst_of_route || !out) return MOE_ERR_INVALID_ARG;   // topk_w may be null: plain sum
    if (!moe::all_aligned16({y_perm, out})) return MOE_ERR_UNSUPPORTED;
    return moe::cuda_status(moe::combine_rows_t(reinterpret_cast<const uint4 *>(y_perm), dst_of_route, topk_w, T,
                                                H, k, out, (cudaStream_t)stream));
}

extern "C" moe_status_t moe_unpermute_combine_mxfp8(const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                                    const float *topk_w, int64_t T, int H, int k, uint8_t *out_q,
                                                    uint8_t *out_sf, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_unpermute_combine_mxfp8");
    using namespace moe;
    if (T < 0 || H < 1) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > 32 || H % 32 != 0) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!y_perm || !dst_of_route || !out_q || !out_sf) return MOE_ERR_INVALID_ARG;   // topk_w may be null
    if (reinterpret_cast<uintptr_t>(y_perm) % 16 || reinterpret_cast<uintptr_t>(out_q) % 8)
        return MOE_ERR_UNSUPPORTED;   // 16-byte row loads, 8-byte code stores
    cudaStream_t s = (cudaStream_t)stream;
    const int sl = H / 8;
    cudaError_t e;
    if (k <= 1) e = launch_mx<1>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 2) e = launch_mx<2>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 4) e = launch_mx<4>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 8) e = launch_mx<8>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 16) e = launch_mx<16>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else e = launch_mx<32>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    return cuda_status(e);
}

extern "C" moe_status_t moe_unpermute_combine_nvfp4(const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                                    const float *topk_w, int64_t T, int H, int k, uint8_t *out_q,
                                                    uint8_t *out_sf, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_unpermute_combine_nvfp4");
    using namespace moe;
    if (T < 0 || H < 1) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > 32 || H % 16 != 0) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!y_perm || !dst_of_route || !out_q || !out_sf) return MOE_ERR_INVALID_ARG;   // topk_w may be null
    if (reinterpret_cast<uintptr_t>(y_perm) % 16 || reinterpret_cast<uintptr_t>(out_q) % 4)
        return MOE_ERR_UNSUPPORTED;   // 16-byte row loads, 4-byte code stores
    cudaStream_t s = (cudaStream_t)stream;
    const int sl = H / 8;
    cudaError_t e;
    if (k <= 1) e = launch_nvfp4<1>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 2) e = launch_nvfp4<2>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 4) e = launch_nvfp4<4>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 8) e = launch_nvfp4<8>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else if (k <= 16) e = launch_nvfp4<16>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    else e = launch_nvfp4<32>(y_perm, dst_of_route, topk_w, T, k, sl, out_q, out_sf, s);
    return cuda_status(e);
}
