// grouped_gemm_pair_mx.cuh -- the MXFP8 FC1 (gate/up GEMM + SwiGLU, h quantised to MXFP8
// along F) on CTA pairs with the routed tokens on the MMA's N axis: the block-scaled
// counterpart of the bf16 pair FC1 in grouped_gemm_pair.cuh.
//
// A pair tile is 256 weight rows (M, 128 per CTA) x up to 256 tokens (N) of one expert,
// 128 E4M3 elements of K per ring stage, tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale
// (M = 256, K = 32 per instruction, one UE8M0 scale per 32 K elements).  Per stage each CTA
// loads one pre-swizzled 16 KB weight block (its 128 rows, as moe_quantize_weights_mxfp8
// lays them out), its half of the tile's token rows (K-major E4M3 rows; boxes of 128 rows,
// or 32 when the CTA's half is at most 32 tokens), the 512-byte scale atom of its weight block
// and the two atoms that hold the scales of all the tile's tokens (each CTA's MMA half reads
// the scales of every N column).  The leader's tcgen05.cp.cta_group::2 moves each CTA's atoms
// from its own shared memory into its own TMEM.  Per CTA and K step that is 34 KB for 512
// tensor-pipe cycles, against 49.5 KB for the one-CTA MXFP8 tile (128 tokens x 256 weight rows)
// of the same MMA work.
//
// Token blocks start at multiples of 256 rows inside an expert (the last one takes the rest),
// so a block's tokens are whole 128-row tiles of the tile-layout scales: block b of expert e
// has its token scales in tiles mt(e) + 2b and mt(e) + 2b + 1, mt(e) = the 128-row tiles of
// the experts before e (the layout moe_permute_mxfp8 and the FC1 epilogue write).
//
// TMEM holds one accumulator of 256 columns; the scale slots (12 columns per ring stage: A 4,
// B 8) leave no room for a second, so a tile's epilogue finishes before the next tile's MMAs.
// The epilogue hands it back early: eight epilogue warps (two per TMEM lane quarter, alternate
// 32-token chunks) each load their 128 columns into registers and release the accumulator
// before they compute and store (straight to global memory), while the next tile's MMAs run.
//
// CTA 0 of the pair holds the gate rows of the tile's 128 features, CTA 1 the up rows of the
// same features (one weight block each).  The epilogue warps of the two CTAs pair up through
// distributed shared memory: per 32-token chunk each hands its partner the 16 tokens the
// partner finishes (CTA 0 finishes tokens 0..15 of the chunk, CTA 1 tokens 16..31).
// h = silu(g) * u is then transposed through the same buffer so that two lanes hold one
// token's 32 features (one MX block along F: its maximum, scale and 32 codes in registers, 16
// code bytes per lane stored at once), the scale bytes written in the tile layout.  (The bf16
// g | u stash of the straight-through backward is left to the one-CTA kernel, whose threads
// hold token rows.)
//
// (The same pair scheme for FC2 -- CTA c on output columns 256 fb + 128 c.. -- measured no
// faster than the one-CTA kernel on the DeepSeek-V3 shape: its tiles are four times shorter
// along K, so the hand-over of the single accumulator at every tile costs a larger share.)
// ("MoE training optimization" issue: MXFP8 grouped GEMM; "Add MoE + expert-parallel Python
// API surface, PyTorch reference, and tests", Summary: mxfp8 operands, SwiGLU experts,
// DeepSeek-style clamp.)
#pragma once

#include "grouped_gemm_pair.cuh"
#include "mx.cuh"

namespace moe {
namespace gpm {

constexpr int kThreads = 320;               // warps: producer, MMA, 8 epilogue
constexpr int BT = 256;                      // tokens per pair tile (N)
constexpr int kMaxE = 1024;
constexpr int A_BYTES = 16384;               // one weight block: 128 rows x 128 K bytes
constexpr int B_BYTES = 16384;               // up to 128 token rows x 128 K bytes (128-byte swizzle)
constexpr int B_SMALL_BYTES = 32 * 128;      // the 32-row token box
constexpr int SFA_OFF = A_BYTES + B_BYTES;   // the weight block's scale atom (512 B)
constexpr int SFB_OFF = SFA_OFF + 512;       // the token scale atoms of two 128-row tiles (1 KB)
constexpr int STAGE_BYTES = 34816;           // A + B + 1.5 KB of scales, rounded up to 1 KB
constexpr int ACC_COLS = 256;
constexpr int SF_COLS = 12;                  // TMEM columns of one stage's scales: A 4, B 8
constexpr int TMEM_COLS = 512;

struct MCfg {
    static constexpr int STAGES = 5;
    // the exchange: per epilogue warp, 2 chunk parities x 16 tokens x 32 features fp32
    static constexpr int XBUF_BYTES = 8 * 2 * 16 * 32 * 4;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + XBUF_BYTES + 1024;   // + alignment slack
    // with the static tables (3 x 4 KB) and barriers within the 227 KB a CTA may use
    static_assert(SMEM_BYTES + 13 * 1024 <= 232448, "shared memory budget");
    static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
};

struct Args {
    const int32_t *group_offsets;   // [E+1]
    int E;
    int K;          // contraction length H (a multiple of 128)
    int N_out;      // output columns F
    int n_fb;       // feature blocks per expert: F / 128
    int64_t rows_cap;
    uint8_t *h_q;             // h codes [rows, F]
    uint8_t *h_sf;            // h scales, tile layout over F
    int clamp;                // clamp of the SwiGLU inputs (inclusive bounds) when != 0
    float gate_lo, gate_hi, up_lo, up_hi;
    uint32_t *err;
};

struct MTile {
    int e, fb;
    int t0;       // first permuted row of the token block
    int l0;       // its index inside the expert (a multiple of 256)
    int nvalid;   // rows of the block that belong to the expert (1..256)
    int n;        // MMA N: nvalid rounded up to 16
};

// pair tile p -> (expert, feature block, token block); s_start[e] = tiles before expert e.
// Within an expert: bands of up to 16 token blocks, in each band the feature block outer and
// the token block fastest (the clusters working at once share weight blocks in the L2).
__device__ __forceinline__ MTile decode(int p, const Args &a, const int *s_off, const int *s_start) {
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= p) lo = mid; else hi = mid - 1;
    }
    MTile t;
    t.e = lo;
    const int rows = s_off[lo + 1] - s_off[lo];
    const int ntb = (rows + BT - 1) / BT;
    const int local = p - s_start[lo];
    const int band_tiles = gp::kBandBlocks * a.n_fb;
    const int band = local / band_tiles;
    const int bsz = ntb - band * gp::kBandBlocks < gp::kBandBlocks ? ntb - band * gp::kBandBlocks : gp::kBandBlocks;
    const int in_band = local - band * band_tiles;
    t.fb = in_band / bsz;
    const int tb = band * gp::kBandBlocks + (in_band - t.fb * bsz);
    t.l0 = tb * BT;
    t.t0 = s_off[lo] + t.l0;
    const int left = rows - t.l0;
    t.nvalid = left < BT ? left : BT;
    t.n = (t.nvalid + 15) & ~15;
    return t;
}

// Maps: tmA0 / tmA1 the gate / up weight blocks, tmSA0 / tmSA1 their scale atoms, tmX / tmX32
// the token codes (boxes of 128 / 32 rows), tmSB the token scales (tile pairs).
// 168 registers a thread at most (three of the ten warps share one of the SM's four 16K-register
// files); the epilogue warps, which hold 128 accumulator values each, spill a little
__global__ void __launch_bounds__(kThreads, 1)
pair_fc1_mx_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
               const __grid_constant__ CUtensorMap tmSA0, const __grid_constant__ CUtensorMap tmSA1,
               const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmX32,
               const __grid_constant__ CUtensorMap tmSB, const Args args) {
    using C = MCfg;
    constexpr int S = C::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[S], empty_bar[S], tfull_bar, tempty_bar, drain_bar;
    __shared__ uint64_t xbar[8][2];   // FC1 exchange: [epilogue warp][chunk parity], the peer's 32 lanes
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_off[kMaxE + 1];
    __shared__ int s_start[kMaxE + 1];
    __shared__ int s_mt[kMaxE + 1];   // 128-row scale tiles of the experts before e
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = sm100::cluster_ctarank();
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = sm100::smem_u32(smem);

    // ---------------------------------------------------------------- set-up (on chip)
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            sm100::mbar_init(&full_bar[s], 1);
            sm100::mbar_init(&empty_bar[s], 1);
        }
        sm100::mbar_init(&tfull_bar, 1);
        sm100::mbar_init(&tempty_bar, 2 * 8);   // one lane of each epilogue warp of both CTAs
        sm100::mbar_init(&drain_bar, 1);
        for (int i = 0; i < 16; ++i) sm100::mbar_init(&xbar[i >> 1][i & 1], 32);
        s_abort = 0;
        sm100::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        sm100::prefetch_tmap(&tmA0);
        sm100::prefetch_tmap(&tmSA0);
        sm100::prefetch_tmap(&tmA1);
        sm100::prefetch_tmap(&tmSA1);
        sm100::prefetch_tmap(&tmX);
        sm100::prefetch_tmap(&tmSB);
    }
    if (warp == 1) {
        sm100::tmem_alloc_pair(&s_tmem_base, TMEM_COLS);
        sm100::tmem_relinquish_pair();
    }
    sm100::tc_fence_before();
    sm100::cluster_sync();   // both CTAs' barriers initialised before either touches the other's
    sm100::tc_fence_after();

    pdl_wait();   // from here on the kernel reads what earlier kernels on the stream wrote
    const uint64_t wait_ns = device_wait_limit(args.err);
    const int E = args.E;
    for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = args.group_offsets[i];
    __syncthreads();
    if (warp == 2) {
        // s_start[e] = pair tiles before expert e (token blocks x feature blocks), s_mt[e] =
        // 128-row scale tiles before it
        const int seg = (E + 31) / 32;
        const int e0 = lane * seg;
        auto rows_of = [&](int e) {
            const int r = s_off[e + 1] - s_off[e];
            return r > 0 ? r : 0;
        };
        int sum = 0, msum = 0;
        for (int i = 0; i < seg; ++i)
            if (e0 + i < E) {
                sum += ((rows_of(e0 + i) + BT - 1) / BT) * args.n_fb;
                msum += (rows_of(e0 + i) + 127) / 128;
            }
        int incl = sum, mincl = msum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            const int mo = __shfl_up_sync(0xFFFFFFFFu, mincl, off);
            if (lane >= off) {
                incl += o;
                mincl += mo;
            }
        }
        int run = incl - sum, mrun = mincl - msum;
        for (int i = 0; i < seg; ++i) {
            if (e0 + i < E) {
                s_start[e0 + i] = run;
                s_mt[e0 + i] = mrun;
                run += ((rows_of(e0 + i) + BT - 1) / BT) * args.n_fb;
                mrun += (rows_of(e0 + i) + 127) / 128;
            }
        }
        const bool offs_ok = group_offsets_in_bounds(s_off, E, args.rows_cap, lane, args.err);
        if (lane == 31) {
            s_start[E] = offs_ok ? incl : 0;   // no tiles for offsets out of bounds
            s_mt[E] = mincl;
        }
    }
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;
    const int total = s_start[E];
    const int G = (int)(gridDim.x >> 1), cid = (int)(blockIdx.x >> 1);
    const int rounds = (total + G - 1) / G;
    const int kblocks = args.K / 128;
    volatile int *abort = &s_abort;

    if (warp == 0) {
        // ============================================================ producer (both CTAs)
        if (lane == 0) {
            const uint32_t full0 = sm100::cluster_addr(&full_bar[0], 0);   // the first CTA's barriers
            // the first CTA loads gate blocks, the second up blocks (F / 128 per K block)
            const int nblk = args.n_fb;
            const CUtensorMap *tA = rank == 1 ? &tmA1 : &tmA0;
            const CUtensorMap *tSA = rank == 1 ? &tmSA1 : &tmSA0;
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int r = 0; r < rounds && ok; ++r) {
                const int p = gp::round_tile(r, cid, G, total);
                if (p < 0) continue;
                const MTile tl = decode(p, args, s_off, s_start);
                const int half = tl.n >> 1;                     // tokens per CTA
                const int trow = tl.t0 + (int)rank * half;      // this CTA's first token row
                const bool small = half <= 32;
                const uint32_t tx = 2u * (uint32_t)(A_BYTES + (small ? B_SMALL_BYTES : B_BYTES) + 512 + 1024);
                const int mt0 = s_mt[tl.e] + (tl.l0 >> 7);      // the block's first scale tile
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!sm100::mbar_wait(&empty_bar[stage], phase ^ 1u, abort, args.err, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_base + stage * STAGE_BYTES;
                    const uint32_t fb_c = full0 + (uint32_t)(stage * sizeof(uint64_t));
                    if (rank == 0) sm100::mbar_arrive_expect_tx(&full_bar[stage], tx);
                    const int64_t blk = ((int64_t)tl.e * kblocks + kb) * nblk + tl.fb;
                    sm100::tma_load_2d_pair(sa, tA, fb_c, 0, (int)(blk * 128));
                    sm100::tma_load_2d_pair(sa + SFA_OFF, tSA, fb_c, 0, (int)(blk * 32));
                    sm100::tma_load_2d_pair(sa + A_BYTES, small ? &tmX32 : &tmX, fb_c, kb * 128, trow);
                    sm100::tma_load_4d_pair(sa + SFB_OFF, &tmSB, fb_c, 0, 0, kb, mt0);
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // the copies in flight land before the CTA can exit: its stages are free again
                // once the first CTA's MMAs (or its drain) release them
                int st = stage;
                uint32_t ph = phase;
                for (int i = 0; i < S && i < issued; ++i) {
                    if (--st < 0) { st = S - 1; ph ^= 1u; }
                    int dummy = 0;
                    sm100::mbar_wait(&empty_bar[st], ph, &dummy, nullptr, 10000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer (first CTA)
        if (rank == 0) {
            const uint64_t a_desc0 = sm100::sdesc_sw128(smem_base, 16, 1024);            // K-major weight rows
            const uint64_t b_desc0 = sm100::sdesc_sw128(smem_base + A_BYTES, 16, 1024);  // K-major token rows
            constexpr uint64_t KSTEP = 32 >> 4;   // 32 E4M3 elements of K
            constexpr uint64_t STAGE_STEP = STAGE_BYTES >> 4;
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, issued_any = false;
            for (int r = 0; r < rounds && ok; ++r) {
                const int p = gp::round_tile(r, cid, G, total);
                if (p < 0) continue;
                const int n = decode(p, args, s_off, s_start).n;
                const uint32_t idesc = sm100::idesc_mxf8(256, n);
                const bool got_acc = sm100::mbar_wait_cluster(&tempty_bar, acc_phase ^ 1u, abort, args.err, wait_ns);
                if (__any_sync(0xFFFFFFFFu, !got_acc)) { ok = false; break; }
                sm100::tc_fence_after();
                for (int kb = 0; kb < kblocks; ++kb) {
                    const bool got = sm100::mbar_wait(&full_bar[stage], phase, abort, args.err, wait_ns);
                    if (__any_sync(0xFFFFFFFFu, !got)) { ok = false; break; }
                    sm100::tc_fence_after();
                    const uint64_t ad = a_desc0 + (uint64_t)stage * STAGE_STEP;
                    const uint64_t bd = b_desc0 + (uint64_t)stage * STAGE_STEP;
                    const uint32_t ssf = smem_base + stage * STAGE_BYTES + SFA_OFF;
                    const uint32_t tsf = tmem_base + ACC_COLS + stage * SF_COLS;
                    if (sm100::elect_one()) {
                        // this stage's scales into its TMEM slot (A: 4 columns; B: the two token
                        // tiles' atoms, 8 columns), then four MMAs of K = 32 picking scale byte kk
                        sm100::tmem_cp_32x128b_x4_pair(tsf, sm100::sdesc_plain(ssf));
                        sm100::tmem_cp_32x128b_x4_pair(tsf + 4, sm100::sdesc_plain(ssf + 512));
                        sm100::tmem_cp_32x128b_x4_pair(tsf + 8, sm100::sdesc_plain(ssf + 1024));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            sm100::mma_mxf8_pair(tmem_base, ad + kk * KSTEP, bd + kk * KSTEP,
                                                 idesc | sm100::idesc_sf_ids(kk, kk), tsf, tsf + 4,
                                                 (kb | kk) != 0 ? 1u : 0u);
                        sm100::mma_commit_pair(&empty_bar[stage], 0x3);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (sm100::elect_one()) sm100::mma_commit_pair(&tfull_bar, 0x3);
                __syncwarp();
                acc_phase ^= 1u;
            }
            if (!ok && issued_any && sm100::elect_one()) {
                // drain: the MMAs already issued finish before TMEM is released
                sm100::mma_commit_pair(&drain_bar, 0x1);
                int dummy = 0;
                sm100::mbar_wait(&drain_bar, 0, &dummy, nullptr, 10000000ull);
            }
            __syncwarp();
        }
    } else {
        // ============================================================ epilogue (both CTAs)
        // Eight warps, two per TMEM lane quarter q: warp `sub` of a quarter takes the 32-token
        // chunks 2 i + sub.  Every store goes straight to global memory (no staging, nothing
        // to wait for before the accumulator is released).
        const int ew = warp - 2;             // epilogue warp 0..7
        const int q = warp & 3;              // TMEM lane quarter of this warp
        const int sub = ew >> 2;             // which of the quarter's two warps
        const uint32_t tempty0 = sm100::cluster_addr(&tempty_bar, 0);
        uint32_t acc_phase = 0;
        int chunk_parity = 0;
        uint32_t xphase = 0;   // bit b: parity of the next wait on xbar[ew][b]
        bool alive = true;
        for (int r = 0; r < rounds && alive; ++r) {
            const int p = gp::round_tile(r, cid, G, total);
            if (p < 0) continue;
            const MTile tl = decode(p, args, s_off, s_start);
            const bool got = sm100::mbar_wait(&tfull_bar, acc_phase, abort, args.err, wait_ns);
            if (__any_sync(0xFFFFFFFFu, !got)) break;
            sm100::tc_fence_after();
            // this warp's four chunks (128 accumulator columns of its lane quarter) into
            // registers, then the accumulator goes back to the MMA warp at once: the next
            // tile's MMAs run while these values are finished and stored
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16);
            uint32_t raw[4][32];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (32 * sub + 64 * i < tl.n) sm100::tmem_ld32(tacc + 32 * sub + 64 * i, raw[i]);
            sm100::tmem_ld_wait();
            sm100::tc_fence_before();
            __syncwarp();
            if (lane == 0) sm100::mbar_arrive_cluster(tempty0);
            acc_phase ^= 1u;

            {
                const bool gate = rank == 0;              // TMEM lanes: gate (CTA 0) or up (CTA 1) rows
                const int F = args.N_out;
                const int fcol = tl.fb * 128 + q * 32;    // this warp's first feature; lane = feature
                float *xown = reinterpret_cast<float *>(smem + S * STAGE_BYTES) + ew * 1024;   // [parity][16][32]
                const uint32_t xpeer = sm100::cluster_addr(xown, rank ^ 1u);
                const int kblk32 = fcol / 32;             // this warp's MX block along F
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c0 = 32 * sub + 64 * i;
                    if (c0 >= tl.n || !alive) continue;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[i][j]);
                    if (args.clamp) {
                        const float lo = gate ? args.gate_lo : args.up_lo, hi = gate ? args.gate_hi : args.up_hi;
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = fminf(fmaxf(v[j], lo), hi);
                    }
                    // exchange with the other CTA's warp of the same place: CTA 0 keeps tokens
                    // 0..15 of the chunk and hands over 16..31, CTA 1 the other way round
                    const uint32_t xdst = xpeer + (uint32_t)(chunk_parity * 2048);
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        sm100::st_cluster_f32(xdst + (uint32_t)((t * 32 + lane) * 4), gate ? v[16 + t] : v[t]);
                    sm100::mbar_arrive_cluster(sm100::cluster_addr(&xbar[ew][chunk_parity], rank ^ 1u));
                    const bool xok = sm100::mbar_wait_cluster(&xbar[ew][chunk_parity], (xphase >> chunk_parity) & 1u,
                                                              abort, args.err, wait_ns);
                    xphase ^= 1u << chunk_parity;
                    if (__any_sync(0xFFFFFFFFu, !xok)) { alive = false; continue; }
                    float *xr = xown + chunk_parity * 512;   // the peer's 16 tokens, [t][lane]
                    float hv[16];
                    if (gate) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) hv[t] = gp::silu(v[t]) * xr[t * 32 + lane];
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) hv[t] = gp::silu(xr[t * 32 + lane]) * v[16 + t];
                    }
                    chunk_parity ^= 1;
                    const int tok0 = c0 + (gate ? 0 : 16);   // first token of this CTA's 16
                    const int nv = tl.nvalid - tok0;
                    // MX quantisation along F, one block = a token's 32 features of this warp:
                    // h goes through the exchange buffer (read out above) transposed, 16-byte
                    // pieces of row t at piece ^ (t % 8) (conflict-free both ways); lane l then
                    // holds features 16 (l & 1) .. of token l / 2
                    __syncwarp();
#pragma unroll
                    for (int t = 0; t < 16; ++t) xr[t * 32 + ((((lane >> 2) ^ (t & 7))) << 2) + (lane & 3)] = hv[t];
                    __syncwarp();
                    const int tt = lane >> 1, hh = lane & 1;
                    float qv[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 f4 = *reinterpret_cast<const float4 *>(xr + tt * 32 + (((4 * hh + j) ^ (tt & 7)) << 2));
                        qv[4 * j] = f4.x;
                        qv[4 * j + 1] = f4.y;
                        qv[4 * j + 2] = f4.z;
                        qv[4 * j + 3] = f4.w;
                    }
                    float amax = 0.0f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(qv[j]));
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
                    const int X = mx::scale_exp(amax);
                    const float sc = mx::inv_pow2(X);
                    uint32_t w4[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const __nv_fp8x2_storage_t p0 = __nv_cvt_float2_to_fp8x2(
                            make_float2(qv[4 * j] * sc, qv[4 * j + 1] * sc), __NV_SATFINITE, __NV_E4M3);
                        const __nv_fp8x2_storage_t p1 = __nv_cvt_float2_to_fp8x2(
                            make_float2(qv[4 * j + 2] * sc, qv[4 * j + 3] * sc), __NV_SATFINITE, __NV_E4M3);
                        w4[j] = (uint32_t)p0 | ((uint32_t)p1 << 16);
                    }
                    if (tt < nv) {
                        *reinterpret_cast<uint4 *>(args.h_q + (int64_t)(tl.t0 + tok0 + tt) * F + fcol + 16 * hh) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        if (hh == 0) {
                            const int l = tl.l0 + tok0 + tt;   // row inside the expert
                            args.h_sf[mx::tile_sf_offset(s_mt[tl.e] + (l >> 7), F / 128, l & 127, kblk32)] =
                                (uint8_t)(X + 127);
                        }
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    sm100::tc_fence_before();
    __syncthreads();
    sm100::cluster_sync();   // no arrive, store or copy of one CTA still targets the other
    if (warp == 1) {
        sm100::tc_fence_after();
        sm100::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// Host launch: clusters of two CTAs, as many as can be resident at once (persistent
// schedule), at most one per pair tile; programmatic stream serialization.
inline moe_status_t launch(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &sa0, const CUtensorMap &sa1,
                    const CUtensorMap &x, const CUtensorMap &x32, const CUtensorMap &sb, const Args &args,
                    int64_t tiles_bound, cudaStream_t s) {
    if (tiles_bound <= 0) return MOE_OK;
    auto kern = pair_fc1_mx_kernel;
    constexpr int smem = MCfg::SMEM_BYTES;
    static PerDeviceOnce once;   // per device: the smem attribute set, resident clusters counted
    int max_clusters = 0;
    const moe_status_t st = once.get(
        [&](int *n) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                return MOE_ERR_CUDA;
            cudaLaunchConfig_t q{};
            q.gridDim = dim3(2);
            q.blockDim = dim3(kThreads);
            q.dynamicSmemBytes = smem;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 2;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(n, kern, &q) != cudaSuccess || *n < 1) return MOE_ERR_CUDA;
            return MOE_OK;
        },
        &max_clusters);
    if (st != MOE_OK) return st;
    const int64_t G = tiles_bound < max_clusters ? tiles_bound : max_clusters;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(2 * G));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, a0, a1, sa0, sa1, x, x32, sb, args) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_status();
}

}  // namespace gpm
}  // namespace moe
