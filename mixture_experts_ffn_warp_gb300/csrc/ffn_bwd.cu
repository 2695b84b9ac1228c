// ffn_bwd.cu -- A8: backward of the expert FFN and of the combine.
//
//   B1 combine_bwd      dy_perm[row(t,j)] = bf16(w[t,j] * dY[t]); d_topk_w[t,j] = <dY[t], y(t,j)>
//   B2+B3 dgrad FC2     dh = dy_perm W_down^T (fp32 in TMEM), then dSwiGLU from the fc1_c
//                       stash in the epilogue: dg = dh*u*s*(1+g*(1-s)), du = dh*g*s -> bf16
//                       (CTA pairs with tokens on M when F % 256 == 0)
//   B4 dgrad FC1        dx_perm = [dg|du] [W_gate; W_up]^T (K = 2F), fp32
//   B5 wgrad            dW_down[e] = h_e^T dy_e;  dW_gate|dW_up[e] = x_e^T [dg|du]_e  (fp32;
//                       K = the rows of group e, read on the device; 0-token experts -> 0)
//   B6 unpermute-sum    dx[t] = bf16(sum_j dx_perm[row(t,j)])
// ("Add MoE + expert-parallel Python API surface, PyTorch reference, and tests",
// Summary: backward re-dispatches gradient rows along the forward routes, recomputes
// SwiGLU from the fc1_c stash, returns FP32 weight gradients and route gradients;
// "[Draft][JAX] MoE block optimization": grouped_gemm_dswiglu; "[JAX] Expert
// Parallelism", commit log: zero-filled wgrad of experts with no tokens.)
#include "gemm_launch.cuh"
#include "grouped_gemm_pair.cuh"

using namespace moe;
using gg::Op;

namespace {

constexpr int kBwdWarps = 8;

template <int KMAX>
__global__ void __launch_bounds__(kBwdWarps * 32)
combine_bwd_kernel(const uint4 *__restrict__ dY, const uint4 *__restrict__ y_perm,
                   const int32_t *__restrict__ dst_of_route, const float *__restrict__ topk_w, int64_t T,
                   int k, int slices, uint4 *__restrict__ dy_perm, float *__restrict__ d_topk_w,
                   const int32_t *__restrict__ group_sizes, const int32_t *__restrict__ group_offsets,
                   int64_t rows_cap, int64_t token_blocks) {
    pdl_wait();
    if ((int64_t)blockIdx.x >= token_blocks) {
        // one block per expert: its padding rows (aligned groups) get a zero gradient row,
        // never uninitialised memory
        const int e = (int)(blockIdx.x - token_blocks);
        const int64_t first = (int64_t)group_offsets[e] + group_sizes[e];
        const int64_t last = group_offsets[e + 1] < rows_cap ? group_offsets[e + 1] : rows_cap;
        for (int64_t row = first; row < last; ++row)
            for (int v = threadIdx.x; v < slices; v += blockDim.x) dy_perm[row * slices + v] = make_uint4(0, 0, 0, 0);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_dst = -1;
    float my_w = 0.0f;
    if (lane < k) {
        my_dst = dst_of_route[t * k + lane];
        my_w = topk_w[t * k + lane];
    }
    int dst[KMAX];
    float w[KMAX], dot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        dst[j] = __shfl_sync(0xFFFFFFFFu, my_dst, j);
        w[j] = __shfl_sync(0xFFFFFFFFu, my_w, j);
        if (j >= k) dst[j] = -1;
        dot[j] = 0.0f;
    }
    const bool want_dot = d_topk_w != nullptr;
    // U 16-byte slices a lane per pass: the U dY loads, then per route the U y loads, are
    // in flight together (one slice at a time left the loop bound by load latency)
    constexpr int U = 4;
    for (int s0 = lane; s0 < slices; s0 += 32 * U) {
        uint4 g[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (s0 + 32 * u < slices) g[u] = __ldg(dY + t * slices + s0 + 32 * u);
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (dst[j] < 0) continue;
            const uint4 *yrow = y_perm + (int64_t)dst[j] * slices;
            uint4 *orow = dy_perm + (int64_t)dst[j] * slices;
            uint4 yv[U];
            if (want_dot) {   // bf16 expert output of the route, widened exactly
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (s0 + 32 * u < slices) yv[u] = __ldg(yrow + s0 + 32 * u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (s0 + 32 * u >= slices) continue;
                const __nv_bfloat162 *gp = reinterpret_cast<const __nv_bfloat162 *>(&g[u]);
                uint4 o;
                __nv_bfloat162 *op = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 d = __bfloat1622float2(gp[i]);
                    op[i] = __floats2bfloat162_rn(w[j] * d.x, w[j] * d.y);
                    if (want_dot) {
                        const float2 f = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(&yv[u])[i]);
                        dot[j] = fmaf(d.x, f.x, dot[j]);
                        dot[j] = fmaf(d.y, f.y, dot[j]);
                    }
                }
                orow[s0 + 32 * u] = o;
            }
        }
    }
    if (!want_dot) return;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        float v = dot[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0 && j < k) d_topk_w[t * k + j] = dst[j] >= 0 ? v : 0.0f;
    }
}

template <int KMAX>
// T tokens' blocks plus one block per expert for the padding rows.
cudaError_t launch_combine_bwd(const moe_bf16_t *dY, const moe_bf16_t *y_perm, const int32_t *dst, const float *w,
                               int64_t T, int H, int E, int k, moe_bf16_t *dy_perm, float *d_topk_w,
                               const int32_t *group_sizes, const int32_t *group_offsets, int64_t rows_cap,
                               cudaStream_t s) {
    const int64_t blocks = (T + kBwdWarps - 1) / kBwdWarps;
    launch_k(combine_bwd_kernel<KMAX>, dim3((unsigned)(blocks + E)), dim3(kBwdWarps * 32), 0, s,
             reinterpret_cast<const uint4 *>(dY), reinterpret_cast<const uint4 *>(y_perm), dst, w, T, k, H / 8,
             reinterpret_cast<uint4 *>(dy_perm), d_topk_w, group_sizes, group_offsets, rows_cap, blocks);
    return cudaGetLastError();
}

moe_status_t check_sizes(int E, int H, int F, int64_t rows_cap, void *ws, size_t ws_bytes) {
    if (E < 1 || H < 1 || F < 1 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (E > gg::kMaxE || H % 128 != 0 || F % 128 != 0 || rows_cap >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int64_t mblock_bound(int64_t rows_cap, int E) { return (rows_cap + gg::BM - 1) / gg::BM + E; }
// upper bound of the token blocks of the pair GEMMs over all experts
int64_t token_block_bound(int64_t rows_cap, int E) { return (rows_cap + gp::BT - 1) / gp::BT + E; }

}  // namespace

extern "C" moe_status_t moe_combine_bwd(const moe_bf16_t *dY, const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                        const float *topk_w, const int32_t *group_sizes,
                                        const int32_t *group_offsets, int64_t T, int H, int E, int k,
                                        int64_t rows_cap, moe_bf16_t *dy_perm, float *d_topk_w,
                                        moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_combine_bwd");
    if (T < 0 || H < 1 || E < 1 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > 32 || H % 8 != 0 || E > gg::kMaxE) return MOE_ERR_UNSUPPORTED;
    if (!group_sizes || !group_offsets || !dy_perm) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!dY || !dst_of_route || !topk_w || (d_topk_w && !y_perm))) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({dY, y_perm, dy_perm})) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    if (T > 0) {   // (with no tokens every group is empty: no padding rows either)
        cudaError_t e;
#define MOE_COMBINE_BWD(KM) \
    launch_combine_bwd<KM>(dY, y_perm, dst_of_route, topk_w, T, H, E, k, dy_perm, d_topk_w, group_sizes, \
                           group_offsets, rows_cap, s)
        if (k <= 1) e = MOE_COMBINE_BWD(1);
        else if (k <= 2) e = MOE_COMBINE_BWD(2);
        else if (k <= 4) e = MOE_COMBINE_BWD(4);
        else if (k <= 8) e = MOE_COMBINE_BWD(8);
        else if (k <= 16) e = MOE_COMBINE_BWD(16);
        else e = MOE_COMBINE_BWD(32);
#undef MOE_COMBINE_BWD
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

namespace {

// clamp (nullable): gate_lo, gate_hi, up_lo, up_hi of the forward's SwiGLU input clamp
moe_status_t dgrad_fc2_impl(const moe_bf16_t *dy_perm, const moe_bf16_t *W_down, const moe_bf16_t *fc1_c,
                            const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap, moe_bf16_t *dgu,
                            void *ws, size_t ws_bytes, moe_stream_t stream, const float *clamp) {
    moe_status_t st = check_sizes(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK || rows_cap == 0) return st;
    if (!dy_perm || !W_down || !fc1_c || !group_offsets || !dgu) return MOE_ERR_INVALID_ARG;
    if (F % 256 == 0) {
        // CTA pairs: 256 token rows (M, 128 per CTA) x 256 features (N) per pair tile, both
        // operands K-major (dy_perm rows, W_down rows); the epilogue reads the stash rows
        CUtensorMap tW, tX, tOut;
        if (!tmap_bf16_3d(&tW, W_down, H, F, E, 64, 128) || !tmap_bf16_2d(&tX, dy_perm, H, rows_cap, H, 64, 128) ||
            !tmap_store_2d(&tOut, dgu, 2, 2 * (uint64_t)F, rows_cap, 2 * (uint64_t)F))
            return MOE_ERR_UNSUPPORTED;
        gp::Args a{};
        a.group_offsets = group_offsets;
        a.E = E;
        a.K = H;
        a.N_out = F;
        a.n_fb = F / 256;
        a.rows_cap = rows_cap;
        a.y16 = reinterpret_cast<__nv_bfloat16 *>(dgu);
        a.aux = reinterpret_cast<const __nv_bfloat16 *>(fc1_c);
        if (clamp) {
            a.clamp = 1;
            a.gate_lo = clamp[0];
            a.gate_hi = clamp[1];
            a.up_lo = clamp[2];
            a.up_hi = clamp[3];
        }
        a.err = ws_error_word(ws);
        return gp::launch<gp::Op::DSWIGLU>(tW, tW, tX, tOut, tOut, a, token_block_bound(rows_cap, E) * a.n_fb,
                                           (cudaStream_t)stream);
    }
    const int bn = 128;
    // A = dy_perm [rows, H] (K-major), B = W_down[e] as [F rows][H] (K-major)
    CUtensorMap tA, tB, tC;
    if (!tmap_bf16_2d(&tA, dy_perm, H, rows_cap, H, 64, 128) || !tmap_bf16_3d(&tB, W_down, H, F, E, 64, bn) ||
        !tmap_store_2d(&tC, dgu, 2, 2 * (uint64_t)F, rows_cap, 2 * (uint64_t)F))
        return MOE_ERR_UNSUPPORTED;
    gg::Args a{};
    a.group_offsets = group_offsets;
    a.E = E;
    a.N = F;
    a.K = H;
    a.n_tiles = F / bn;
    a.rows_cap = rows_cap;
    a.out0 = reinterpret_cast<__nv_bfloat16 *>(dgu);
    a.ld0 = 2 * (int64_t)F;
    a.aux = reinterpret_cast<const __nv_bfloat16 *>(fc1_c);
    a.ld_aux = 2 * (int64_t)F;
    if (clamp) {
        a.clamp = 1;
        a.gate_lo = clamp[0];
        a.gate_hi = clamp[1];
        a.up_lo = clamp[2];
        a.up_hi = clamp[3];
    }
    a.err = ws_error_word(ws);
    const int64_t bound = mblock_bound(rows_cap, E) * a.n_tiles;
    return gg::launch<Op::DGRAD_DSWIGLU, 128>(tA, tB, tB, tC, tC, a, bound, (cudaStream_t)stream);
}

}  // namespace

extern "C" moe_status_t moe_grouped_dgrad_fc2_dswiglu(const moe_bf16_t *dy_perm, const moe_bf16_t *W_down,
                                                      const moe_bf16_t *fc1_c, const int32_t *group_offsets,
                                                      int E, int H, int F, int64_t rows_cap, moe_bf16_t *dgu,
                                                      void *ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_dgrad_fc2_dswiglu");
    return dgrad_fc2_impl(dy_perm, W_down, fc1_c, group_offsets, E, H, F, rows_cap, dgu, ws, ws_bytes, stream,
                          nullptr);
}

extern "C" moe_status_t moe_grouped_dgrad_fc2_dswiglu_clamped(const moe_bf16_t *dy_perm, const moe_bf16_t *W_down,
                                                              const moe_bf16_t *fc1_c, const int32_t *group_offsets,
                                                              int E, int H, int F, int64_t rows_cap, float gate_lo,
                                                              float gate_hi, float up_lo, float up_hi,
                                                              moe_bf16_t *dgu, void *ws, size_t ws_bytes,
                                                              moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_dgrad_fc2_dswiglu_clamped");
    if (!(gate_lo <= gate_hi && up_lo <= up_hi)) return MOE_ERR_INVALID_ARG;   // also rejects NaN
    const float c[4] = {gate_lo, gate_hi, up_lo, up_hi};
    return dgrad_fc2_impl(dy_perm, W_down, fc1_c, group_offsets, E, H, F, rows_cap, dgu, ws, ws_bytes, stream, c);
}

extern "C" moe_status_t moe_grouped_dgrad_fc1(const moe_bf16_t *dgu, const moe_bf16_t *W_gate,
                                              const moe_bf16_t *W_up, const int32_t *group_offsets, int E, int H,
                                              int F, int64_t rows_cap, float *dx_perm, void *ws, size_t ws_bytes,
                                              moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_dgrad_fc1");
    moe_status_t st = check_sizes(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK || rows_cap == 0) return st;
    if (!dgu || !W_gate || !W_up || !group_offsets || !dx_perm) return MOE_ERR_INVALID_ARG;
    if (H % 256 == 0) {
        // CTA pairs: 256 rows of W_gate / W_up (hidden units) x up to 256 tokens per pair tile
        CUtensorMap tW0, tW1, tX, tOut;
        if (!tmap_bf16_3d(&tW0, W_gate, F, H, E, 64, 128) || !tmap_bf16_3d(&tW1, W_up, F, H, E, 64, 128) ||
            !tmap_bf16_2d(&tX, dgu, 2 * (uint64_t)F, rows_cap, 2 * (uint64_t)F, 64, 128) ||
            !tmap_store_plain(&tOut, dx_perm, 4, H, rows_cap, H, 32, 16))
            return MOE_ERR_UNSUPPORTED;
        gp::Args a{};
        a.group_offsets = group_offsets;
        a.E = E;
        a.K = 2 * F;
        a.k_split = F;
        a.N_out = H;
        a.n_fb = H / 256;
        a.rows_cap = rows_cap;
        a.y = dx_perm;
        a.err = ws_error_word(ws);
        return gp::launch<gp::Op::DGRAD_FC1>(tW0, tW1, tX, tOut, tOut, a, token_block_bound(rows_cap, E) * a.n_fb,
                                             (cudaStream_t)stream);
    }
    const int bn = 128;
    // A = [dg | du] [rows, 2F] (K-major), B = W_gate[e] / W_up[e] as [H rows][F] (K-major)
    CUtensorMap tA, tB0, tB1, tC;
    if (!tmap_bf16_2d(&tA, dgu, 2 * (uint64_t)F, rows_cap, 2 * (uint64_t)F, 64, 128) ||
        !tmap_bf16_3d(&tB0, W_gate, F, H, E, 64, bn) || !tmap_bf16_3d(&tB1, W_up, F, H, E, 64, bn) ||
        !tmap_store_2d(&tC, dx_perm, 4, H, rows_cap, H))
        return MOE_ERR_UNSUPPORTED;
    gg::Args a{};
    a.group_offsets = group_offsets;
    a.E = E;
    a.N = H;
    a.K = 2 * F;
    a.k_split = F;
    a.n_tiles = H / bn;
    a.rows_cap = rows_cap;
    a.out_f32 = dx_perm;
    a.ld0 = H;
    a.err = ws_error_word(ws);
    const int64_t bound = mblock_bound(rows_cap, E) * a.n_tiles;
    return gg::launch<Op::DGRAD_FC1, 128>(tA, tB0, tB1, tC, tC, a, bound, (cudaStream_t)stream);
}

namespace {

// The weight gradients, stored as fp32 (elem = 4) or bf16 (elem = 2); fp32 accumulation either way.
moe_status_t wgrad_impl(const moe_bf16_t *x_perm, const moe_bf16_t *h, const moe_bf16_t *dy_perm,
                        const moe_bf16_t *dgu, const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap,
                        void *dW_gate, void *dW_up, void *dW_down, int elem, void *ws, size_t ws_bytes,
                        moe_stream_t stream) {
    moe_status_t st = check_sizes(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (!group_offsets || !dW_gate || !dW_up || !dW_down) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (rows_cap == 0) {   // no rows at all: every expert's gradient is zero
        const size_t n = (size_t)E * H * F * (size_t)elem;
        if (cudaMemsetAsync(dW_gate, 0, n, s) != cudaSuccess || cudaMemsetAsync(dW_up, 0, n, s) != cudaSuccess ||
            cudaMemsetAsync(dW_down, 0, n, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (!x_perm || !h || !dy_perm || !dgu) return MOE_ERR_INVALID_ARG;
    const uint64_t rows = (uint64_t)rows_cap;
    if (H % 256 == 0 && F % 256 == 0 && rows_cap >= 1024 * (int64_t)E) {
        // CTA pairs (256 x 256 gradient tiles) when the experts hold enough rows that each tile's
        // K loop outweighs its epilogue (the 32 fp32 columns x 256 rows it stores per CTA)
        for (int which = 0; which < 2; ++which) {
            const bool down = which == 0;
            // dW_down[e] [F, H] = h_e^T dy_e;  [dW_gate | dW_up][e] [H, 2F] = x_e^T [dg | du]_e
            const moe_bf16_t *A = down ? h : x_perm, *B = down ? dy_perm : dgu;
            const int M = down ? F : H, N = down ? H : 2 * F;
            CUtensorMap tA, tB, tC0, tC1;
            // each operand's 128 columns of a 64-row K step in one load (two 64-column chunks)
            if (!tmap_bf16_col_chunks(&tA, A, M, rows, M, 64) || !tmap_bf16_col_chunks(&tB, B, N, rows, N, 64))
                return MOE_ERR_UNSUPPORTED;
            if (down ? !tmap_store_2d(&tC0, dW_down, elem, H, (uint64_t)E * F, H)
                     : (!tmap_store_2d(&tC0, dW_gate, elem, F, (uint64_t)E * H, F) ||
                        !tmap_store_2d(&tC1, dW_up, elem, F, (uint64_t)E * H, F)))
                return MOE_ERR_UNSUPPORTED;
            if (down) tC1 = tC0;
            gp::Args a{};
            a.group_offsets = group_offsets;
            a.E = E;
            a.M = M;
            a.nt_m = M / 256;
            a.nt_n = N / 256;
            a.m_fastest = a.nt_m <= a.nt_n ? 1 : 0;   // the smaller dimension fastest: a small L2 working set
            a.n_split = down ? 0 : F;
            a.a_rows = reinterpret_cast<const __nv_bfloat16 *>(A);
            a.lda = M;
            a.b_rows = reinterpret_cast<const __nv_bfloat16 *>(B);
            a.ldb = N;
            a.rows_cap = rows_cap;
            a.w_bf16 = elem == 2;
            a.err = ws_error_word(ws);
            st = gp::launch<gp::Op::WGRAD>(tA, tA, tB, tC0, tC1, a, (int64_t)E * a.nt_m * a.nt_n, s);
            if (st != MOE_OK) return st;
        }
        return MOE_OK;
    }
    {   // dW_down[e] [F, H] = h_e^T dy_e: A = h (MN-major), B = dy_perm (MN-major)
        const int bn = (H % 256 == 0) ? 256 : 128;
        CUtensorMap tA, tB, tC;
        if (!tmap_bf16_2d(&tA, h, F, rows, F, 64, 64) || !tmap_bf16_2d(&tB, dy_perm, H, rows, H, 64, 64) ||
            !tmap_store_2d(&tC, dW_down, elem, H, (uint64_t)E * F, H))
            return MOE_ERR_UNSUPPORTED;
        gg::Args a{};
        a.group_offsets = group_offsets;
        a.E = E;
        a.M = F;
        a.N = H;
        a.m_tiles = F / gg::BM;
        a.n_tiles = H / bn;
        a.rows_cap = rows_cap;
        a.out_f32 = static_cast<float *>(dW_down);
        a.out0 = static_cast<__nv_bfloat16 *>(dW_down);
        a.w_bf16 = elem == 2;
        a.ld0 = H;
        a.expert_stride = (int64_t)F * H;
        a.err = ws_error_word(ws);
        const int64_t tiles = (int64_t)E * a.m_tiles * a.n_tiles;
        st = (bn == 256) ? gg::launch<Op::WGRAD_DOWN, 256>(tA, tB, tB, tC, tC, a, tiles, s)
                         : gg::launch<Op::WGRAD_DOWN, 128>(tA, tB, tB, tC, tC, a, tiles, s);
        if (st != MOE_OK) return st;
    }
    {   // [dW_gate | dW_up][e] [H, 2F] = x_e^T [dg | du]_e: A = x_perm (MN-major), B = dgu (MN-major)
        CUtensorMap tA, tB, tC0, tC1;
        if (!tmap_bf16_2d(&tA, x_perm, H, rows, H, 64, 64) ||
            !tmap_bf16_2d(&tB, dgu, 2 * (uint64_t)F, rows, 2 * (uint64_t)F, 64, 64) ||
            !tmap_store_2d(&tC0, dW_gate, elem, F, (uint64_t)E * H, F) ||
            !tmap_store_2d(&tC1, dW_up, elem, F, (uint64_t)E * H, F))
            return MOE_ERR_UNSUPPORTED;
        gg::Args a{};
        a.group_offsets = group_offsets;
        a.E = E;
        a.M = H;
        a.N = 2 * F;
        a.n_split = F;
        a.m_tiles = H / gg::BM;
        a.n_tiles = 2 * F / 256;
        a.rows_cap = rows_cap;
        a.out_f32 = static_cast<float *>(dW_gate);
        a.out0 = static_cast<__nv_bfloat16 *>(dW_gate);
        a.ld0 = F;
        a.out1_f32 = static_cast<float *>(dW_up);
        a.out1 = static_cast<__nv_bfloat16 *>(dW_up);
        a.ld1 = F;
        a.w_bf16 = elem == 2;
        a.expert_stride = (int64_t)H * F;
        a.err = ws_error_word(ws);
        const int64_t tiles = (int64_t)E * a.m_tiles * a.n_tiles;
        return gg::launch<Op::WGRAD_GATEUP, 256>(tA, tB, tB, tC0, tC1, a, tiles, s);
    }
}

}  // namespace

extern "C" moe_status_t moe_grouped_wgrad(const moe_bf16_t *x_perm, const moe_bf16_t *h, const moe_bf16_t *dy_perm,
                                          const moe_bf16_t *dgu, const int32_t *group_offsets, int E, int H, int F,
                                          int64_t rows_cap, float *dW_gate, float *dW_up, float *dW_down, void *ws,
                                          size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_wgrad");
    return wgrad_impl(x_perm, h, dy_perm, dgu, group_offsets, E, H, F, rows_cap, dW_gate, dW_up, dW_down, 4, ws,
                      ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_wgrad_bf16(const moe_bf16_t *x_perm, const moe_bf16_t *h,
                                               const moe_bf16_t *dy_perm, const moe_bf16_t *dgu,
                                               const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap,
                                               moe_bf16_t *dW_gate, moe_bf16_t *dW_up, moe_bf16_t *dW_down, void *ws,
                                               size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_wgrad_bf16");
    return wgrad_impl(x_perm, h, dy_perm, dgu, group_offsets, E, H, F, rows_cap, dW_gate, dW_up, dW_down, 2, ws,
                      ws_bytes, stream);
}

extern "C" moe_status_t moe_unpermute_sum(const float *dx_perm, const int32_t *dst_of_route, int64_t T, int H, int k,
                                          moe_bf16_t *dx, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_unpermute_sum");
    if (T < 0 || H < 1) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!dx_perm || !dst_of_route || !dx) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({dx_perm, dx})) return MOE_ERR_UNSUPPORTED;
    return cuda_status(combine_rows(dx_perm, dst_of_route, nullptr, T, H, k, dx, (cudaStream_t)stream));
}

namespace {

moe_status_t ffn_bwd_impl(const moe_bf16_t *dY, const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                          const moe_bf16_t *W_up, const moe_bf16_t *W_down, const moe_bf16_t *fc1_c,
                          const moe_bf16_t *h, const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                          const int32_t *group_sizes, const int32_t *group_offsets, const float *topk_w, int64_t T,
                          int H, int F, int E, int k, int64_t rows_cap, moe_bf16_t *dy_perm, moe_bf16_t *dgu,
                          float *dx_perm, moe_bf16_t *dx, void *dW_gate, void *dW_up, void *dW_down, int elem,
                          float *d_topk_w, void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status_t st = check_sizes(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK) return st;
    st = moe_combine_bwd(dY, y_perm, dst_of_route, topk_w, group_sizes, group_offsets, T, H, E, k, rows_cap,
                         dy_perm, d_topk_w, stream);
    if (st != MOE_OK) return st;
    if (rows_cap > 0) {
        st = moe_grouped_dgrad_fc2_dswiglu(dy_perm, W_down, fc1_c, group_offsets, E, H, F, rows_cap, dgu, ws,
                                           ws_bytes, stream);
        if (st != MOE_OK) return st;
        st = moe_grouped_dgrad_fc1(dgu, W_gate, W_up, group_offsets, E, H, F, rows_cap, dx_perm, ws, ws_bytes,
                                   stream);
        if (st != MOE_OK) return st;
    }
    st = wgrad_impl(x_perm, h, dy_perm, dgu, group_offsets, E, H, F, rows_cap, dW_gate, dW_up, dW_down, elem, ws,
                    ws_bytes, stream);
    if (st != MOE_OK) return st;
    return moe_unpermute_sum(dx_perm, dst_of_route, T, H, k, dx, stream);
}

}  // namespace

extern "C" moe_status_t moe_grouped_ffn_bwd(
    const moe_bf16_t *dY, const moe_bf16_t *x_perm, const moe_bf16_t *W_gate, const moe_bf16_t *W_up,
    const moe_bf16_t *W_down, const moe_bf16_t *fc1_c, const moe_bf16_t *h, const moe_bf16_t *y_perm,
    const int32_t *dst_of_route, const int32_t *group_sizes, const int32_t *group_offsets, const float *topk_w,
    int64_t T, int H, int F, int E, int k, int64_t rows_cap, moe_bf16_t *dy_perm, moe_bf16_t *dgu,
    float *dx_perm, moe_bf16_t *dx, float *dW_gate, float *dW_up, float *dW_down, float *d_topk_w, void *ws,
    size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_ffn_bwd");
    return ffn_bwd_impl(dY, x_perm, W_gate, W_up, W_down, fc1_c, h, y_perm, dst_of_route, group_sizes, group_offsets,
                        topk_w, T, H, F, E, k, rows_cap, dy_perm, dgu, dx_perm, dx, dW_gate, dW_up, dW_down, 4,
                        d_topk_w, ws, ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_ffn_bwd_bf16(
    const moe_bf16_t *dY, const moe_bf16_t *x_perm, const moe_bf16_t *W_gate, const moe_bf16_t *W_up,
    const moe_bf16_t *W_down, const moe_bf16_t *fc1_c, const moe_bf16_t *h, const moe_bf16_t *y_perm,
    const int32_t *dst_of_route, const int32_t *group_sizes, const int32_t *group_offsets, const float *topk_w,
    int64_t T, int H, int F, int E, int k, int64_t rows_cap, moe_bf16_t *dy_perm, moe_bf16_t *dgu,
    float *dx_perm, moe_bf16_t *dx, moe_bf16_t *dW_gate, moe_bf16_t *dW_up, moe_bf16_t *dW_down, float *d_topk_w,
    void *ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_ffn_bwd_bf16");
    return ffn_bwd_impl(dY, x_perm, W_gate, W_up, W_down, fc1_c, h, y_perm, dst_of_route, group_sizes, group_offsets,
                        topk_w, T, H, F, E, k, rows_cap, dy_perm, dgu, dx_perm, dx, dW_gate, dW_up, dW_down, 2,
                        d_topk_w, ws, ws_bytes, stream);
}
