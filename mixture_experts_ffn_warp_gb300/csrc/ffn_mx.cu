// ffn_mx.cu -- A7: the grouped expert FFN on MXFP8 operands (E4M3 data, UE8M0 scales
// per 32 K elements) with block-scaled tcgen05 MMAs.  FC1 quantises h to MXFP8
// along F in its epilogue; FC2 writes fp32 expert outputs.  Activation tiles come
// in by TMA; weight tiles (pre-swizzled 16 KB blocks from moe_quantize_weights_mxfp8)
// and all scale atoms by plain bulk copies.
#include "gemm_launch.cuh"

using namespace moe;
using gg::Op;

namespace {

moe_status_t check_mx(int E, int H, int F, int64_t rows_cap, void *ws, size_t ws_bytes) {
    if (E < 1 || H < 1 || F < 1 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (E > gg::kMaxE || H % 128 != 0 || F % 128 != 0 || rows_cap >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int64_t mblock_bound(int64_t rows_cap, int E) { return (rows_cap + gg::BM - 1) / gg::BM + E; }

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

namespace {

// clamp (nullable): gate_lo, gate_hi, up_lo, up_hi of the SwiGLU input clamp
moe_status_t fc1_mx_impl(const uint8_t *x_q, const uint8_t *x_sf, const uint8_t *Wg_q, const uint8_t *Wg_sf,
                         const uint8_t *Wu_q, const uint8_t *Wu_sf, const int32_t *group_offsets, int E, int H,
                         int F, int64_t rows_cap, uint8_t *h_q, uint8_t *h_sf, moe_bf16_t *fc1_c, void *ws,
                         size_t ws_bytes, moe_stream_t stream, const float *clamp) {
    moe_status_t st = check_mx(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK || rows_cap == 0) return st;
    if (!x_q || !x_sf || !Wg_q || !Wg_sf || !Wu_q || !Wu_sf || !group_offsets || !h_q || !h_sf)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_sf) || !aligned16(Wg_sf) || !aligned16(Wu_sf) || !aligned16(Wg_q) || !aligned16(Wu_q))
        return MOE_ERR_UNSUPPORTED;
    CUtensorMap tA, tC;
    if (!tmap_u8_2d(&tA, x_q, H, rows_cap, H, 128, 128) || !tmap_store_2d(&tC, h_q, 1, F, rows_cap, F))
        return MOE_ERR_UNSUPPORTED;
    gg::Args a{};
    a.group_offsets = group_offsets;
    a.E = E;
    a.N = F;
    a.K = H;
    a.n_tiles = F / 128;
    a.rows_cap = rows_cap;
    a.sfa = x_sf;
    a.sfb0 = Wg_sf;
    a.sfb1 = Wu_sf;
    a.b0_tiles = Wg_q;
    a.b1_tiles = Wu_q;
    a.nb_rows = F;
    a.out_q = h_q;
    a.ld0 = F;
    a.out_sf = h_sf;
    a.out1 = reinterpret_cast<__nv_bfloat16 *>(fc1_c);   // nullable: the g | u stash
    a.ld1 = 2 * (int64_t)F;
    if (clamp) {
        a.clamp = 1;
        a.gate_lo = clamp[0];
        a.gate_hi = clamp[1];
        a.up_lo = clamp[2];
        a.up_hi = clamp[3];
    }
    a.err = ws_error_word(ws);
    return gg::launch<Op::FC1_MX, 256>(tA, tA, tA, tC, tC, a, mblock_bound(rows_cap, E) * a.n_tiles,
                                       (cudaStream_t)stream);
}

}  // namespace

extern "C" moe_status_t moe_grouped_fc1_swiglu_mxfp8(const uint8_t *x_q, const uint8_t *x_sf, const uint8_t *Wg_q,
                                                     const uint8_t *Wg_sf, const uint8_t *Wu_q, const uint8_t *Wu_sf,
                                                     const int32_t *group_offsets, int E, int H, int F,
                                                     int64_t rows_cap, uint8_t *h_q, uint8_t *h_sf,
                                                     moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                                     moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc1_swiglu_mxfp8");
    return fc1_mx_impl(x_q, x_sf, Wg_q, Wg_sf, Wu_q, Wu_sf, group_offsets, E, H, F, rows_cap, h_q, h_sf, fc1_c, ws,
                       ws_bytes, stream, nullptr);
}

extern "C" moe_status_t moe_grouped_fc1_swiglu_mxfp8_clamped(
    const uint8_t *x_q, const uint8_t *x_sf, const uint8_t *Wg_q, const uint8_t *Wg_sf, const uint8_t *Wu_q,
    const uint8_t *Wu_sf, const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap, float gate_lo,
    float gate_hi, float up_lo, float up_hi, uint8_t *h_q, uint8_t *h_sf, moe_bf16_t *fc1_c, void *ws,
    size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc1_swiglu_mxfp8_clamped");
    if (!(gate_lo <= gate_hi && up_lo <= up_hi)) return MOE_ERR_INVALID_ARG;   // also rejects NaN
    const float c[4] = {gate_lo, gate_hi, up_lo, up_hi};
    return fc1_mx_impl(x_q, x_sf, Wg_q, Wg_sf, Wu_q, Wu_sf, group_offsets, E, H, F, rows_cap, h_q, h_sf, fc1_c, ws,
                       ws_bytes, stream, c);
}

namespace {

// FC2_MX: y_perm rows in bf16 (fp32 accumulation, one rounding per element).
moe_status_t fc2_mx_impl(const uint8_t *h_q, const uint8_t *h_sf, const uint8_t *Wd_q, const uint8_t *Wd_sf,
                         const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap, moe_bf16_t *y_perm,
                         void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status_t st = check_mx(E, H, F, rows_cap, ws, ws_bytes);
    if (st != MOE_OK || rows_cap == 0) return st;
    if (!h_q || !h_sf || !Wd_q || !Wd_sf || !group_offsets || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(h_sf) || !aligned16(Wd_sf) || !aligned16(Wd_q)) return MOE_ERR_UNSUPPORTED;
    const int bn = (H % 256 == 0) ? 256 : 128;
    CUtensorMap tA, tC;
    if (!tmap_u8_2d(&tA, h_q, F, rows_cap, F, 128, 128) || !tmap_store_2d(&tC, y_perm, 2, H, rows_cap, H))
        return MOE_ERR_UNSUPPORTED;
    gg::Args a{};
    a.group_offsets = group_offsets;
    a.E = E;
    a.N = H;
    a.K = F;
    a.n_tiles = H / bn;
    a.rows_cap = rows_cap;
    a.sfa = h_sf;
    a.sfb0 = Wd_sf;
    a.b0_tiles = Wd_q;
    a.nb_rows = H;
    a.out0 = reinterpret_cast<__nv_bfloat16 *>(y_perm);
    a.ld0 = H;
    a.err = ws_error_word(ws);
    const int64_t bound = mblock_bound(rows_cap, E) * a.n_tiles;
    if (bn == 256) return gg::launch<Op::FC2_MX, 256>(tA, tA, tA, tC, tC, a, bound, (cudaStream_t)stream);
    return gg::launch<Op::FC2_MX, 128>(tA, tA, tA, tC, tC, a, bound, (cudaStream_t)stream);
}

}  // namespace

extern "C" moe_status_t moe_grouped_fc2_mxfp8(const uint8_t *h_q, const uint8_t *h_sf, const uint8_t *Wd_q,
                                              const uint8_t *Wd_sf, const int32_t *group_offsets, int E, int H, int F,
                                              int64_t rows_cap, moe_bf16_t *y_perm, void *ws, size_t ws_bytes,
                                              moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_fc2_mxfp8");
    return fc2_mx_impl(h_q, h_sf, Wd_q, Wd_sf, group_offsets, E, H, F, rows_cap, y_perm, ws, ws_bytes, stream);
}

extern "C" moe_status_t moe_grouped_ffn_fwd_mxfp8(const uint8_t *x_q, const uint8_t *x_sf, const uint8_t *Wg_q,
                                                  const uint8_t *Wg_sf, const uint8_t *Wu_q, const uint8_t *Wu_sf,
                                                  const uint8_t *Wd_q, const uint8_t *Wd_sf,
                                                  const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap,
                                                  uint8_t *h_q, uint8_t *h_sf, moe_bf16_t *y_perm, void *ws,
                                                  size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_grouped_ffn_fwd_mxfp8");
    moe_status_t st = moe_grouped_fc1_swiglu_mxfp8(x_q, x_sf, Wg_q, Wg_sf, Wu_q, Wu_sf, group_offsets, E, H, F,
                                                   rows_cap, h_q, h_sf, nullptr, ws, ws_bytes, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_fc2_mxfp8(h_q, h_sf, Wd_q, Wd_sf, group_offsets, E, H, F, rows_cap, y_perm, ws, ws_bytes,
                                 stream);
}
