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
