// ffn_mx.cu -- A7: the grouped expert FFN on MXFP8 operands (E4M3 data, UE8M0 scales
// per 32 K elements) with block-scaled tcgen05 MMAs.  FC1 quantises h to MXFP8
// along F in its epilogue; FC2 writes bf16 expert outputs.  FC1 runs on CTA pairs with the
// tokens on N (grouped_gemm_pair_mx.cuh) unless the bf16 g | u stash is asked for; FC2, and
// FC1 with the stash, on the one-CTA kernel (grouped_gemm.cuh), whose weight tiles and scale
// atoms come in by plain bulk copies.
#include "gemm_launch.cuh"
#include "grouped_gemm_pair_mx.cuh"

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
// upper bound of the pair GEMMs' token blocks over all experts
int64_t token_block_bound(int64_t rows_cap, int E) { return (rows_cap + gpm::BT - 1) / gpm::BT + E; }
// 128-row scale tiles of the tile layout (moe_mx_tile_scale_bytes)
uint64_t scale_tiles(int64_t rows_cap, int E) { return (uint64_t)((rows_cap + 127) / 128 + E); }

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
    if (fc1_c) {
        // with the g | u stash: one CTA per tile, tokens on M, so that each epilogue thread
        // holds one token's row and writes the stash rows with 16-byte stores (the pair kernel
        // holds one feature per thread and measured slower with the stash: 2.07 against 1.94 ms
        // on the DeepSeek-V3 shape)
        CUtensorMap tA, tC;
        if (!tmap_u8_2d(&tA, x_q, H, rows_cap, H, 128, 128) || !tmap_store_2d(&tC, h_q, 1, F, rows_cap, F))
            return MOE_ERR_UNSUPPORTED;
        gg::Args b{};
        b.group_offsets = group_offsets;
        b.E = E;
        b.N = F;
        b.K = H;
        b.n_tiles = F / 128;
        b.rows_cap = rows_cap;
        b.sfa = x_sf;
        b.sfb0 = Wg_sf;
        b.sfb1 = Wu_sf;
        b.b0_tiles = Wg_q;
        b.b1_tiles = Wu_q;
        b.nb_rows = F;
        b.out_q = h_q;
        b.ld0 = F;
        b.out_sf = h_sf;
        b.out1 = reinterpret_cast<__nv_bfloat16 *>(fc1_c);
        b.ld1 = 2 * (int64_t)F;
        if (clamp) {
            b.clamp = 1;
            b.gate_lo = clamp[0];
            b.gate_hi = clamp[1];
            b.up_lo = clamp[2];
            b.up_hi = clamp[3];
        }
        b.err = ws_error_word(ws);
        return gg::launch<Op::FC1_MX, 256>(tA, tA, tA, tC, tC, b, mblock_bound(rows_cap, E) * b.n_tiles,
                                           (cudaStream_t)stream);
    }
    // without it: CTA pairs, per pair tile the gate (first CTA) and up (second CTA) weight
    // blocks of 128 features (M = 256) x up to 256 tokens (N)
    const uint64_t wblocks = (uint64_t)E * (H / 128) * (F / 128);
    CUtensorMap tA0, tA1, tSA0, tSA1, tX, tX32, tSB;
    if (!tmap_u8_rows(&tA0, Wg_q, 128, wblocks * 128, 128) || !tmap_u8_rows(&tA1, Wu_q, 128, wblocks * 128, 128) ||
        !tmap_u8_rows(&tSA0, Wg_sf, 16, wblocks * 32, 32) || !tmap_u8_rows(&tSA1, Wu_sf, 16, wblocks * 32, 32) ||
        !tmap_u8_2d(&tX, x_q, H, rows_cap, H, 128, 128) || !tmap_u8_2d(&tX32, x_q, H, rows_cap, H, 128, 32) ||
        !tmap_sf_tile_pairs(&tSB, x_sf, H / 128, scale_tiles(rows_cap, E)))
        return MOE_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(h_q) % 16 != 0) return MOE_ERR_UNSUPPORTED;   // 16-byte code stores
    gpm::Args a{};
    a.group_offsets = group_offsets;
    a.E = E;
    a.K = H;
    a.N_out = F;
    a.n_fb = F / 128;
    a.rows_cap = rows_cap;
    a.h_q = h_q;
    a.h_sf = h_sf;
    if (clamp) {
        a.clamp = 1;
        a.gate_lo = clamp[0];
        a.gate_hi = clamp[1];
        a.up_lo = clamp[2];
        a.up_hi = clamp[3];
    }
    a.err = ws_error_word(ws);
    return gpm::launch(tA0, tA1, tSA0, tSA1, tX, tX32, tSB, a,
                                     token_block_bound(rows_cap, E) * a.n_fb, (cudaStream_t)stream);
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
    // one CTA per tile: 128 tokens (M) x 256 (or 128) output columns (N)
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
