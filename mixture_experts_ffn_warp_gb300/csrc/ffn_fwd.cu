// ffn_fwd.cu -- A3 + A4: grouped gate/up GEMM with SwiGLU epilogue, then the
// grouped down projection, both on tcgen05 with group sizes read on the device.
#include "gemm_launch.cuh"
#include "grouped_gemm_pair.cuh"

using namespace moe;
using gg::Op;

namespace {

moe_status_t check_common(int E, int H, int F, int64_t rows_cap, void *ws, size_t ws_bytes) {
    if (E < 1 || H < 1 || F < 1 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (E > gg::kMaxE || H % 128 != 0 || F % 128 != 0 || rows_cap >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int64_t mblock_bound(int64_t rows_cap, int E) { return (rows_cap + gg::BM - 1) / gg::BM + E; }
// upper bound of the token blocks of the pair GEMMs over all experts
int64_t token_block_bound(int64_t rows_cap, int E) { return (rows_cap + gp::BT - 1) / gp::BT + E; }

// FC1 + SwiGLU and FC2; topk_w / src_of_row non-null: the router weight of each row's
// route is applied in the epilogue (to h, or to y).
// clamp (nullable): gate_lo, gate_hi, up_lo, up_hi of the SwiGLU input clamp
moe_status_t fc1_impl(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate, const moe_bf16_t *W_up,
                      const int32_t *group_offsets, const int32_t *src_of_row, const float *topk_w, int E, int H,
                      int F, int64_t rows_cap, moe_bf16_t *h, moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                      moe_stream_t stream, const float *clamp = nullptr) {
    moe_status_t st = check_common(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK || rows_cap == 0) return st;
    if (!x_perm || !W_gate || !W_up || !group_offsets || !h) return MOE_ERR_INVALID_ARG;
    // h [rows, F] = SwiGLU(x_perm [rows, H] x (W_gate | W_up) [H, F]) on CTA pairs: per pair
    // tile 128 gate + 128 up weight columns (M = 256) x up to 256 tokens (N)
    CUtensorMap tW0, tW1, tX, tOut, tStash;
    if (!tmap_bf16_3d(&tW0, W_gate, F, H, E, 64, 64) || !tmap_bf16_3d(&tW1, W_up, F, H, E, 64, 64) ||
        !tmap_bf16_2d(&tX, x_perm, H, rows_cap, H, 64, 128) || !tmap_store_plain(&tOut, h, 2, F, rows_cap, F, 32, 16))
        return MOE_ERR_UNSUPPORTED;
    tStash = tOut;
    if (fc1_c && !tmap_store_plain(&tStash, fc1_c, 2, 2 * (uint64_t)F, rows_cap, 2 * (uint64_t)F, 32, 16))
        return MOE_ERR_UNSUPPORTED;
    gp::Args a{};
    a.group_offsets = group_offsets;
    a.E = E;
    a.K = H;
    a.N_out = F;
    a.n_fb = F / 128;
    a.rows_cap = rows_cap;
    a.h = reinterpret_cast<__nv_bfloat16 *>(h);
    a.stash = reinterpret_cast<__nv_bfloat16 *>(fc1_c);
    a.route_w = topk_w;
    a.src_of_row = src_of_row;
    if (clamp) {
        a.clamp = 1;
        a.gate_lo = clamp[0];
        a.gate_hi = clamp[1];
        a.up_lo = clamp[2];
        a.up_hi = clamp[3];
    }
    a.err = ws_error_word(ws);
    return gp::launch<gp::Op::FC1>(tW0, tW1, tX, tOut, tStash, a, token_block_bound(rows_cap, E) * a.n_fb,
                                   (cudaStream_t)stream);
}

moe_status_t fc2_impl(const moe_bf16_t *h, const moe_bf16_t *W_down, const int32_t *group_offsets,
                      const int32_t *src_of_row, const float *topk_w, int E, int H, int F, int64_t rows_cap,
                      moe_bf16_t *y_perm, void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status_t st = check_common(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK || rows_cap == 0) return st;
    if (!h || !W_down || !group_offsets || !y_perm) return MOE_ERR_INVALID_ARG;
    // h [rows, F] x W_down [F, H] -> y_perm [rows, H], fp32 accumulation stored as bf16
    if (H % 256 == 0) {
        // CTA pairs: 256 output columns (M) x up to 256 tokens (N) per pair tile
        CUtensorMap tW, tX, tOut;
        if (!tmap_bf16_3d(&tW, W_down, H, F, E, 64, 64) || !tmap_bf16_2d(&tX, h, F, rows_cap, F, 64, 128) ||
            !tmap_store_plain(&tOut, y_perm, 2, H, rows_cap, H, 32, 16))
            return MOE_ERR_UNSUPPORTED;
        gp::Args a{};
        a.group_offsets = group_offsets;
        a.E = E;
        a.K = F;
        a.N_out = H;
        a.n_fb = H / 256;
        a.rows_cap = rows_cap;
        a.y16 = reinterpret_cast<__nv_bfloat16 *>(y_perm);
        a.route_w = topk_w;
        a.src_of_row = src_of_row;
        a.err = ws_error_word(ws);
        return gp::launch<gp::Op::FC2>(tW, tW, tX, tOut, tOut, a, token_block_bound(rows_cap, E) * a.n_fb,
                                       (cudaStream_t)stream);
    }
    const int bn = 128;
    CUtensorMap tA, tB, tC;
    if (!tmap_bf16_2d(&tA, h, F, rows_cap, F, 64, 128) || !tmap_bf16_3d(&tB, W_down, H, F, E, 64, 64) ||
        !tmap_store_2d(&tC, y_perm, 2, H, rows_cap, H))
        return MOE_ERR_UNSUPPORTED;
    gg::Args b{};
    b.group_offsets = group_offsets;
    b.E = E;
    b.N = H;
    b.K = F;
    b.n_tiles = H / bn;
    b.rows_cap = rows_cap;
    b.out0 = reinterpret_cast<__nv_bfloat16 *>(y_perm);
    b.ld0 = H;
    b.route_w = topk_w;
    b.src_of_row = src_of_row;
    b.err = ws_error_word(ws);
    const int64_t bound = mblock_bound(rows_cap, E) * b.n_tiles;
    return gg::launch<Op::FC2, 128>(tA, tB, tB, tC, tC, b, bound, (cudaStream_t)stream);
}

// Bounds of the SwiGLU clamp: each interval non-empty, no NaN (infinite ends allowed).
bool clamp_bounds_ok(float gate_lo, float gate_hi, float up_lo, float up_hi) {
    return gate_lo <= gate_hi && up_lo <= up_hi;   // false for any NaN
}

}  // namespace

extern "C" moe_status_t moe_grouped_fc1_swiglu(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                               const moe_bf16_t *W_up, const int32_t *group_offsets,
                                               int E, int H, int F, int64_t rows_cap, moe_bf16_t *h,
                                               moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                               moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc1_swiglu");
    return fc1_impl(x_perm, W_gate, W_up, group_offsets, nullptr, nullptr, E, H, F, rows_cap, h, fc1_c, ws,
                    ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_fc2(const moe_bf16_t *h, const moe_bf16_t *W_down,
                                        const int32_t *group_offsets, int E, int H, int F,
                                        int64_t rows_cap, moe_bf16_t *y_perm, void *ws, size_t ws_bytes,
                                        moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc2");
    return fc2_impl(h, W_down, group_offsets, nullptr, nullptr, E, H, F, rows_cap, y_perm, ws, ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_fc1_swiglu_weighted(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                                        const moe_bf16_t *W_up, const int32_t *group_offsets,
                                                        const int32_t *src_of_row, const float *topk_w, int E,
                                                        int H, int F, int64_t rows_cap, moe_bf16_t *h,
                                                        moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                                        moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc1_swiglu_weighted");
    if (rows_cap > 0 && (!src_of_row || !topk_w)) return MOE_ERR_INVALID_ARG;
    return fc1_impl(x_perm, W_gate, W_up, group_offsets, src_of_row, topk_w, E, H, F, rows_cap, h, fc1_c, ws,
                    ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_fc2_weighted(const moe_bf16_t *h, const moe_bf16_t *W_down,
                                                 const int32_t *group_offsets, const int32_t *src_of_row,
                                                 const float *topk_w, int E, int H, int F, int64_t rows_cap,
                                                 moe_bf16_t *y_perm, void *ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc2_weighted");
    if (rows_cap > 0 && (!src_of_row || !topk_w)) return MOE_ERR_INVALID_ARG;
    return fc2_impl(h, W_down, group_offsets, src_of_row, topk_w, E, H, F, rows_cap, y_perm, ws, ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_ffn_fwd(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                            const moe_bf16_t *W_up, const moe_bf16_t *W_down,
                                            const int32_t *group_offsets, int E, int H, int F,
                                            int64_t rows_cap, moe_bf16_t *h, moe_bf16_t *y_perm,
                                            moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                            moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_ffn_fwd");
    moe_status_t st = check_common(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK || rows_cap == 0) return st;
    if (!x_perm || !W_gate || !W_up || !W_down || !group_offsets || !h || !y_perm) return MOE_ERR_INVALID_ARG;
    st = moe_grouped_fc1_swiglu(x_perm, W_gate, W_up, group_offsets, E, H, F, rows_cap, h, fc1_c, ws,
                                ws_bytes, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_fc2(h, W_down, group_offsets, E, H, F, rows_cap, y_perm, ws, ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_fc1_swiglu_clamped(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                                       const moe_bf16_t *W_up, const int32_t *group_offsets,
                                                       const int32_t *src_of_row, const float *topk_w, int E, int H,
                                                       int F, int64_t rows_cap, float gate_lo, float gate_hi,
                                                       float up_lo, float up_hi, moe_bf16_t *h, moe_bf16_t *fc1_c,
                                                       void *ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc1_swiglu_clamped");
    if (!clamp_bounds_ok(gate_lo, gate_hi, up_lo, up_hi)) return MOE_ERR_INVALID_ARG;
    if (rows_cap > 0 && (src_of_row == nullptr) != (topk_w == nullptr)) return MOE_ERR_INVALID_ARG;
    const float c[4] = {gate_lo, gate_hi, up_lo, up_hi};
    return fc1_impl(x_perm, W_gate, W_up, group_offsets, src_of_row, topk_w, E, H, F, rows_cap, h, fc1_c, ws,
                    ws_bytes, stream, c);
}
