// route_topk.cu -- A1: top-k routing over fp32 router logits, its sigmoid
// variant and the router backward.
//
// One warp per token.  Lane l holds experts l, l+32, ...; each of the k rounds
// is a 5-step butterfly max over a 64-bit key (order-preserving bits of the
// score, inverted expert id), so ties go to the lowest expert id and every lane
// ends the round knowing the winner.  Softmax router: the score is the logit and
// the weights are a softmax over the k selected logits.  Sigmoid router: the
// score is sigmoid(logit) (+ the expert routing bias, for the selection only) and
// the weights are the selected sigmoid scores, divided by (their sum + 1e-20)
// when normalising ("[JAX] Expert Parallelism: JAX primitives + VJPs", commit
// log: fused_topk_with_score_function on fp32 logits, sigmoid scores with an
// expert routing bias, the kernel's sum + 1e-20 normalisation, and its backward
// giving the fp32 logits cotangent).
#include "carveout.cuh"
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

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

template <int VPL, bool SIGMOID>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_topk_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int64_t T, int E, int k,
                  int normalize, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + t * E;

    float val[VPL];   // softmax: the logit; sigmoid: the unbiased score
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        int e = lane + 32 * i;
        val[i] = e < E ? __ldg(row + e) : 0.0f;
        if constexpr (SIGMOID) {
            val[i] = sigmoid_f(val[i]);
            key[i] = e < E ? order_key(bias ? val[i] + __ldg(bias + e) : val[i]) : 0u;
        } else {
            key[i] = e < E ? order_key(val[i]) : 0u;
        }
    }
    uint32_t avail = 0;   // bit i: element i of this lane still selectable
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) avail |= 1u << i;

    int my_idx = -1;        // lane j keeps slot j
    float my_val = 0.0f;
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
        if (lane == j) { my_idx = e; my_val = v; }
    }

    if constexpr (SIGMOID) {
        const float sc = (lane < k && my_val == my_val) ? my_val : 0.0f;   // a NaN logit scores 0
        float S = sc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);
        if (lane < k) {
            topk_idx[t * k + lane] = my_idx;
            topk_w[t * k + lane] = normalize ? sc / (S + 1e-20f) : sc;
        }
    } else {
        const float l0 = __shfl_sync(0xFFFFFFFFu, my_val, 0);
        float ex = 0.0f;
        if (lane < k) ex = (l0 == -INFINITY) ? 0.0f : expf(my_val - l0);
        float S = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);
        if (lane < k) {
            topk_idx[t * k + lane] = my_idx;
            topk_w[t * k + lane] = (l0 == -INFINITY) ? 0.0f : ex / S;
        }
    }
}

template <int VPL, bool SIGMOID>
cudaError_t launch(const float *logits, const float *bias, int64_t T, int E, int k, int normalize, int32_t *idx,
                   float *w, cudaStream_t s) {
    int64_t blocks = (T + kRouteWarps - 1) / kRouteWarps;
    prefer_max_smem_carveout<route_topk_kernel<VPL, SIGMOID>>();   // the counting pass runs next
    return launch_k(route_topk_kernel<VPL, SIGMOID>, dim3((unsigned)blocks), dim3(kRouteWarps * 32), 0, s, logits,
                    bias, T, E, k, normalize, idx, w);
}

template <bool SIGMOID>
cudaError_t dispatch(const float *logits, const float *bias, int64_t T, int E, int k, int normalize, int32_t *idx,
                     float *w, cudaStream_t s) {
    const int vpl = (E + 31) / 32;
    if (vpl <= 1) return launch<1, SIGMOID>(logits, bias, T, E, k, normalize, idx, w, s);
    if (vpl <= 2) return launch<2, SIGMOID>(logits, bias, T, E, k, normalize, idx, w, s);
    if (vpl <= 4) return launch<4, SIGMOID>(logits, bias, T, E, k, normalize, idx, w, s);
    if (vpl <= 8) return launch<8, SIGMOID>(logits, bias, T, E, k, normalize, idx, w, s);
    if (vpl <= 16) return launch<16, SIGMOID>(logits, bias, T, E, k, normalize, idx, w, s);
    return launch<32, SIGMOID>(logits, bias, T, E, k, normalize, idx, w, s);
}

// Router backward, one warp per token.  Lanes j < k hold route j (expert e_j,
// its d_topk_w g_j) and recompute its weight from the logits; every lane then
// writes the dense row of d_logits for its experts (0 where not selected).
//   softmax over the valid selected:  dl_j = w_j (g_j - sum_i w_i g_i)
//   sigmoid s_j:  ds_j = normalize ? (g_j - sum_i w_i g_i) / (S + 1e-20) : g_j,
//                 dl_j = ds_j s_j (1 - s_j)
template <int VPL, bool SIGMOID>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_bwd_kernel(const float *__restrict__ logits, const int32_t *__restrict__ topk_idx,
                 const float *__restrict__ d_topk_w, int64_t T, int E, int k, int normalize,
                 float *__restrict__ d_logits) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + t * E;
    int e = -1;
    float g = 0.0f, l = 0.0f;
    if (lane < k) {
        e = topk_idx[t * k + lane];
        if (e < 0 || e >= E) e = -1;
        g = d_topk_w[t * k + lane];
        if (e >= 0) l = __ldg(row + e);
    }
    float dl = 0.0f;
    if constexpr (SIGMOID) {
        const float sc = e >= 0 ? sigmoid_f(l) : 0.0f;
        float S = sc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);
        const float den = S + 1e-20f;
        float gw = (e >= 0 && normalize) ? g * (sc / den) : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) gw += __shfl_xor_sync(0xFFFFFFFFu, gw, off);
        const float ds = normalize ? (g - gw) / den : g;
        dl = e >= 0 ? ds * sc * (1.0f - sc) : 0.0f;
    } else {
        float lmax = e >= 0 ? l : -INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, off));
        const float ex = (e >= 0 && lmax != -INFINITY) ? expf(l - lmax) : 0.0f;
        float S = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);
        const float w = S > 0.0f ? ex / S : 0.0f;
        float gw = w * g;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) gw += __shfl_xor_sync(0xFFFFFFFFu, gw, off);
        dl = e >= 0 ? w * (g - gw) : 0.0f;
    }
    float acc[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
        const float dj = __shfl_sync(0xFFFFFFFFu, dl, j);
        if (ej >= 0 && (ej & 31) == lane) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (i == (ej >> 5)) acc[i] += dj;
        }
    }
    float *drow = d_logits + t * E;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) drow[lane + 32 * i] = acc[i];
}

template <bool SIGMOID>
cudaError_t dispatch_bwd(const float *logits, const int32_t *idx, const float *dw, int64_t T, int E, int k,
                         int normalize, float *dl, cudaStream_t s) {
    const int vpl = (E + 31) / 32;
    const unsigned blocks = (unsigned)((T + kRouteWarps - 1) / kRouteWarps);
#define MOE_ROUTE_BWD(V) \
    launch_k(route_bwd_kernel<V, SIGMOID>, dim3(blocks), dim3(kRouteWarps * 32), 0, s, logits, idx, dw, T, E, k, \
             normalize, dl)
    if (vpl <= 1) MOE_ROUTE_BWD(1);
    else if (vpl <= 2) MOE_ROUTE_BWD(2);
    else if (vpl <= 4) MOE_ROUTE_BWD(4);
    else if (vpl <= 8) MOE_ROUTE_BWD(8);
    else if (vpl <= 16) MOE_ROUTE_BWD(16);
    else MOE_ROUTE_BWD(32);
#undef MOE_ROUTE_BWD
    return cudaGetLastError();
}

}  // namespace
}  // namespace moe

namespace {

moe_status_t check_route(int64_t T, int E, int k) {
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED;
    if ((T + 7) / 8 > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_route_topk(const float *logits, int64_t T, int E, int k,
                                       int32_t *topk_idx, float *topk_w, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_route_topk");
    moe_status_t st = check_route(T, E, k);
    if (st != MOE_OK || T == 0) return st;
    if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    return moe::cuda_status(moe::dispatch<false>(logits, nullptr, T, E, k, 0, topk_idx, topk_w, (cudaStream_t)stream));
}

extern "C" moe_status_t moe_route_topk_sigmoid(const float *logits, const float *expert_bias, int64_t T, int E,
                                               int k, int normalize, int32_t *topk_idx, float *topk_w,
                                               moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_route_topk_sigmoid");
    moe_status_t st = check_route(T, E, k);
    if (st != MOE_OK || T == 0) return st;
    if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    return moe::cuda_status(moe::dispatch<true>(logits, expert_bias, T, E, k, normalize ? 1 : 0, topk_idx, topk_w,
                                                (cudaStream_t)stream));
}

extern "C" moe_status_t moe_route_topk_bwd(const float *logits, const int32_t *topk_idx, const float *d_topk_w,
                                           int64_t T, int E, int k, int score_fn, int normalize, float *d_logits,
                                           moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_route_topk_bwd");
    moe_status_t st = check_route(T, E, k);
    if (st != MOE_OK || T == 0) return st;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (!logits || !topk_idx || !d_topk_w || !d_logits) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const int nz = normalize ? 1 : 0;
    cudaError_t e = score_fn == MOE_SCORE_SIGMOID
                        ? moe::dispatch_bwd<true>(logits, topk_idx, d_topk_w, T, E, k, nz, d_logits, s)
                        : moe::dispatch_bwd<false>(logits, topk_idx, d_topk_w, T, E, k, nz, d_logits, s);
    return moe::cuda_status(e);
}
