// route_topk.cu -- A1: top-k routing over fp32 router logits.
//
// One warp per token.  Lane l holds logits l, l+32, ...; each of the k rounds
// is a 5-step butterfly max over a 64-bit key (order-preserving logit bits,
// inverted expert id), so ties go to the lowest expert id and every lane
// ends the round knowing the winner.  The weights are a softmax over the k
// selected logits ("[JAX] Expert Parallelism: JAX primitives + VJPs",
// commit log: fused_topk_with_score_function on fp32 logits).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;   // tokens per 256-thread block

// Larger key = ranks first.  +0/-0 map to the same key; NaN maps to 0,
// below -inf (whose key is 0x007FFFFF).
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) return 0u;
    uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_topk_kernel(const float *__restrict__ logits, int64_t T, int E, int k,
                  int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + t * E;

    float val[VPL];
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        int e = lane + 32 * i;
        val[i] = e < E ? __ldg(row + e) : 0.0f;
        key[i] = e < E ? order_key(val[i]) : 0u;
    }
    uint32_t avail = 0;   // bit i: element i of this lane still selectable
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) avail |= 1u << i;

    int my_idx = -1;        // lane j keeps slot j
    float my_logit = 0.0f;
    for (int j = 0; j < k; ++j) {
        // local best: highest key, then lowest expert id (lowest i)
        uint64_t best = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (avail & (1u << i)) {
                uint64_t c = ((uint64_t)key[i] << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)(lane + 32 * i));
                if (c > best) best = c;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
            if (o > best) best = o;
        }
        const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
        const int owner = e & 31, slot_i = e >> 5;
        float v = 0.0f;
        if (lane == owner) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (i == slot_i) { v = val[i]; avail &= ~(1u << i); }
        }
        v = __shfl_sync(0xFFFFFFFFu, v, owner);
        if (lane == j) { my_idx = e; my_logit = v; }
    }

    const float l0 = __shfl_sync(0xFFFFFFFFu, my_logit, 0);
    float ex = 0.0f;
    if (lane < k) ex = (l0 == -INFINITY) ? 0.0f : expf(my_logit - l0);
    float s = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    if (lane < k) {
        topk_idx[t * k + lane] = my_idx;
        topk_w[t * k + lane] = (l0 == -INFINITY) ? 0.0f : ex / s;
    }
}

template <int VPL>
cudaError_t launch(const float *logits, int64_t T, int E, int k, int32_t *idx, float *w, cudaStream_t s) {
    int64_t blocks = (T + kRouteWarps - 1) / kRouteWarps;
    route_topk_kernel<VPL><<<(unsigned)blocks, kRouteWarps * 32, 0, s>>>(logits, T, E, k, idx, w);
    return cudaGetLastError();
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_topk(const float *logits, int64_t T, int E, int k,
                                       int32_t *topk_idx, float *topk_w, moe_stream_t stream) {
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if ((T + 7) / 8 > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    int vpl = (E + 31) / 32;
    if (vpl <= 1) e = moe::launch<1>(logits, T, E, k, topk_idx, topk_w, s);
    else if (vpl <= 2) e = moe::launch<2>(logits, T, E, k, topk_idx, topk_w, s);
    else if (vpl <= 4) e = moe::launch<4>(logits, T, E, k, topk_idx, topk_w, s);
    else if (vpl <= 8) e = moe::launch<8>(logits, T, E, k, topk_idx, topk_w, s);
    else if (vpl <= 16) e = moe::launch<16>(logits, T, E, k, topk_idx, topk_w, s);
    else e = moe::launch<32>(logits, T, E, k, topk_idx, topk_w, s);
    return moe::cuda_status(e);
}
