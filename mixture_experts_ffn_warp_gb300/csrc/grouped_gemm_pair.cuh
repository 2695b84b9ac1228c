// grouped_gemm_pair.cuh -- the expert FFN's forward GEMMs (FC1 + SwiGLU, FC2) on CTA
// pairs, with the routed tokens on the MMA's N axis; the backward's FC1 dgrad and weight
// gradients on the same kernel (below).
//
// Each thread-block cluster of two CTAs (one per SM of an SM pair) computes one pair tile
// at a time: 256 expert-weight rows (M, 128 per CTA) x up to 256 tokens (N) of one
// expert, K = the contraction length, with tcgen05.mma.cta_group::2 (M = 256, K = 16).
// Per 64-wide K step a CTA loads 16 KB of weights (its 128 M rows, MN-major: the weight
// matrices' own layout) and 16 KB of tokens (its half of N, K-major rows of the permuted
// activations), 32 KB in all against 48 KB for a one-CTA 128 x 256 tile of the same MMA
// work, so six stages fit in shared memory.  Putting tokens on N makes an expert's last,
// partial token block cost its own width rounded up to 16 tokens rather than a whole
// 128-row tile.
//
// Roles (192 threads per CTA):
//   warp 0      TMA producer in each CTA (one lane): its weight rows and its half of the
//               token rows; completion is counted on the first CTA's `full` barrier
//   warp 1      MMA issuer (one lane of the first CTA only); TMEM (512 columns, two
//               accumulators of up to 256 columns) allocated by warp 1 of both CTAs
//   warps 2..5  epilogue in each CTA: tcgen05.ld of its 128 lanes -> SwiGLU / scaling ->
//               bf16 (h, y_perm) or fp32 (dx_perm) -> shared-memory staging -> TMA stores
//               (row by row only at an expert's last token block)
//
// FC1: CTA c of the pair holds, for the 128 features [128 fb, 128 fb + 128) of the tile,
// gate rows of features 128 fb + 64 c + [0, 64) in TMEM lanes 0..63 and the up rows of the
// same features in lanes 64..127.  The warps of lanes 0..31 (gate) and 64..95 (up) pair up
// through shared memory: each hands the other half of a 32-token chunk, and both finish
// h = silu(g) * u for 16 tokens.
// FC2: CTA c holds output columns 256 fb + 128 c + [0, 128) in its 128 lanes.
//
// Tile order: expert, band of up to 16 token blocks, feature block, token block (fastest), so
// the clusters working at the same time share weight blocks and token rows in the L2.  Cluster i takes in round r
// the tile r * G + (i + r) mod G (G clusters): the rotation spreads the cheaper last token
// blocks of the experts evenly over the clusters.
// ("Add MoE + expert-parallel Python API surface, PyTorch reference, and tests", Summary:
// SwiGLU experts, fc1_c stash, router weight in an FFN epilogue, DeepSeek-style clamp;
// "[Draft][JAX] MoE block optimization": grouped GEMM with the SwiGLU fused.)
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace moe {
namespace gp {

enum class Op : int { FC1, FC2, DGRAD_FC1, WGRAD, DSWIGLU };

// DGRAD_FC1 (the backward's dx_perm = [dg|du] [W_gate; W_up]^T, M = H, K = 2F, fp32 out)
// reads the weights K-major: their rows are the MMA's M rows.
//
// DSWIGLU (the backward's dh = dy_perm W_down^T followed by the dSwiGLU, M = tokens, N = F,
// K = H) puts the routed tokens on M instead: a pair tile is 256 token rows of one expert
// (128 per CTA, both operands K-major: dy_perm rows and W_down rows) x 256 features, so each
// CTA's TMEM lanes are its 128 token rows and the epilogue reads the token-major fc1_c stash
// and writes the token-major [dg | du] rows directly.  The rows of an expert's last token
// block past its end are multiplied and never stored.  (With tokens on N the epilogue had to
// transpose the stash and the outputs through shared memory and measured slower.)
template <Op OP>
constexpr bool a_kmajor() { return OP == Op::DGRAD_FC1 || OP == Op::DSWIGLU; }

// WGRAD (the backward's weight gradients, K-grouped: K = the rows of each expert):
//   dW_down[e] = h_e^T dy_e          M = F, N = H
//   [dW_gate|dW_up][e] = x_e^T [dg|du]_e   M = H, N = 2F (columns >= F go to dW_up)
// Both operands come MN-major from the permuted row tensors; the pair MMAs cover the
// expert's rows in whole 16-row slices loaded by TMA, then one more slice holding the last
// (rows mod 16) rows zero-padded, written by the producer warps of both CTAs into an 8 KB
// tail buffer outside the ring, so no row of the next expert is ever multiplied.

constexpr int kThreads = 192;
constexpr int BT = 256;                  // tokens per pair tile (N), 128 rows loaded per CTA
constexpr int kMaxE = 1024;
constexpr int A_BYTES = 128 * 128;       // 128 weight rows x 64 K (two 64-wide MN chunks)
constexpr int B_BYTES = 128 * 128;       // 128 token rows x 64 K
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 6;
constexpr int TMEM_COLS = 512;           // two accumulators of BT fp32 columns

// Epilogue shared memory: FC1 exchange buffers (2 warp pairs x 2 chunk parities x 2
// directions x 16 tokens x 32 features fp32 = 16 KB) and output staging, two slots per
// epilogue warp of 16 token rows (FC1 and FC2 bf16 rows of 64 B, DGRAD_FC1 fp32 rows of
// 128 B).
template <Op OP>
struct PCfg {
    static constexpr int XBUF_BYTES = OP == Op::FC1 ? 2 * 2 * 2 * 16 * 32 * 4 : 0;
    // WGRAD, DSWIGLU: 32 rows x 64 B (16 fp32 or 32 bf16 columns in the 64-byte swizzle)
    static constexpr int SLOT_BYTES = (OP == Op::FC1 || OP == Op::FC2) ? 16 * 64 : 16 * 128;
    static constexpr int STG_BYTES = 4 * 2 * SLOT_BYTES;
    // WGRAD: the K-tail buffer, outside the ring: 2 operands x 2 MN chunks x 16 K rows x 128 B
    static constexpr int TAIL_BYTES = OP == Op::WGRAD ? 2 * 2 * 16 * 128 : 0;
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + XBUF_BYTES + STG_BYTES + TAIL_BYTES + 1024;   // + alignment slack
    // with the static tables and barriers (9 KB) within the 227 KB a CTA may use
    static_assert(SMEM_BYTES + 9 * 1024 + 512 <= 232448, "shared memory budget");
};

struct Args {
    const int32_t *group_offsets;   // [E+1]
    int E;
    int K;             // contraction length: FC1 H, FC2 F, DGRAD_FC1 2F
    int N_out;         // output columns: FC1 F, FC2 H, DGRAD_FC1 H
    int n_fb;          // feature blocks per expert: FC1 F / 128, others (output columns) / 256
    int k_split;       // DGRAD_FC1: K index where the weights switch from W_gate to W_up (= F)
    // WGRAD: rows M of each expert's gradient, 256-blocks along M and N, the tile order
    // within an expert (M blocks fastest or N blocks fastest), the column where the output
    // switches to the second matrix (0: none), and the operands' row tensors for the K tail
    int M, nt_m, nt_n, m_fastest, n_split;
    int w_bf16;        // WGRAD: the gradients are stored as bf16 (else fp32)
    const __nv_bfloat16 *a_rows;   // [rows, M]
    int64_t lda;
    const __nv_bfloat16 *b_rows;   // [rows, N]
    int64_t ldb;
    int64_t rows_cap;  // rows of the permuted tensors
    __nv_bfloat16 *h;        // FC1: h [rows, F]
    __nv_bfloat16 *stash;    // FC1: [g | u] bf16 [rows, 2F] (nullable)
    __nv_bfloat16 *y16;      // FC2: y_perm bf16 [rows, H]; DSWIGLU: [dg | du] bf16 [rows, 2F]
    float *y;                // DGRAD_FC1: dx_perm fp32 [rows, H]
    const __nv_bfloat16 *aux;   // DSWIGLU: the fc1_c stash [g | u] bf16 [rows, 2F]
    // router weight of each row's route applied in the epilogue (padding rows get 0); null = unweighted
    const float *route_w;
    const int32_t *src_of_row;
    // FC1: optional clamp of the SwiGLU inputs, inclusive bounds (clamp != 0)
    int clamp;
    float gate_lo, gate_hi, up_lo, up_hi;
    uint32_t *err;
};

struct PTile {
    int e, fb;
    int t0;       // first permuted row of the token block
    int nvalid;   // rows of the block that belong to the expert (1..BT)
    int n;        // MMA N: nvalid rounded up to 16
};

// Token blocks per band of the tile order: the ~76 clusters working at once then cover about
// 5 feature blocks x 16 token blocks of an expert (tens of MB of weights and token rows, held
// in the L2), instead of one feature block x all token blocks of an expert with many tokens,
// whose token rows would stream from DRAM again for every feature block.
constexpr int kBandBlocks = 16;

// pair tile p -> (expert, feature block, token block); s_start[e] = tiles before expert e.
// An expert's rows are cut into ceil(rows / BT) blocks of equal width (rounded up to 16):
// an expert of 400 tokens gets blocks of 208 + 192 rather than 256 + 144, so no block is
// so narrow that its MMAs finish faster than one thread issues them, and the blocks cost
// alike under the static schedule.
__device__ __forceinline__ PTile decode(int p, const Args &a, const int *s_off, const int *s_start) {
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= p) lo = mid; else hi = mid - 1;
    }
    PTile t;
    t.e = lo;
    const int rows = s_off[lo + 1] - s_off[lo];
    const int ntb = (rows + BT - 1) / BT;
    const int bs = ((rows + ntb - 1) / ntb + 15) & ~15;   // <= BT
    // within the expert: bands of up to kBandBlocks token blocks, in each band the feature
    // block outer and the token block fastest
    const int local = p - s_start[lo];
    const int band_tiles = kBandBlocks * a.n_fb;
    const int band = local / band_tiles;
    const int bsz = ntb - band * kBandBlocks < kBandBlocks ? ntb - band * kBandBlocks : kBandBlocks;
    const int in_band = local - band * band_tiles;
    t.fb = in_band / bsz;
    const int tb = band * kBandBlocks + (in_band - t.fb * bsz);
    t.t0 = s_off[lo] + tb * bs;
    const int left = rows - tb * bs;
    t.nvalid = left < bs ? left : bs;
    t.n = (t.nvalid + 15) & ~15;
    return t;
}

// DSWIGLU pair tile p -> (expert, 256-token block, 256-feature block): within an expert the
// token blocks vary fastest, so the clusters working at once share the feature block's W_down
// rows and cover all of the expert's dy rows (tens of MB, held in the L2).
struct MTile {
    int e, fb;
    int m0;      // first permuted row of the token block (CTA r holds rows m0 + 128 r + [0, 128))
    int m_end;   // end of the expert's rows
};

__device__ __forceinline__ MTile decode_m(int p, const Args &a, const int *s_off, const int *s_start) {
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= p) lo = mid; else hi = mid - 1;
    }
    MTile t;
    t.e = lo;
    const int rows = s_off[lo + 1] - s_off[lo];
    const int nmb = (rows + BT - 1) / BT;
    const int local = p - s_start[lo];
    const int mb = local % nmb;
    t.fb = local / nmb;
    t.m0 = s_off[lo] + mb * BT;
    t.m_end = s_off[lo + 1];
    return t;
}

struct WTile {
    int e, m0, n0;
    int row0;     // the expert's first permuted row
    int rows;     // its rows
    int full16;   // rows in whole 16-row slices (multiplied by the MMAs)
    int kblocks;  // 64-row K blocks holding them
};

__device__ __forceinline__ WTile decode_w(int p, const Args &a, const int *s_off) {
    WTile t;
    const int per = a.nt_m * a.nt_n;
    t.e = p / per;
    const int l = p - t.e * per;
    int mb, nb;
    if (a.m_fastest) { mb = l % a.nt_m; nb = l / a.nt_m; }
    else { nb = l % a.nt_n; mb = l / a.nt_n; }
    t.m0 = mb * 256;
    t.n0 = nb * 256;
    t.row0 = s_off[t.e];
    const int r = s_off[t.e + 1] - t.row0;
    t.rows = r > 0 ? r : 0;
    t.full16 = t.rows & ~15;
    t.kblocks = (t.full16 + 63) / 64;
    return t;
}

__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Tile of round r for cluster `cid` of G (-1 past the end).
__device__ __forceinline__ int round_tile(int r, int cid, int G, int total) {
    const int p = r * G + (cid + r) % G;
    return p < total ? p : -1;
}

template <Op OP>
__global__ void __launch_bounds__(kThreads, 1)
pair_gemm_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                 const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmOut,
                 const __grid_constant__ CUtensorMap tmStash, const Args args) {
    using PC = PCfg<OP>;
    constexpr int XBUF_BYTES = PC::XBUF_BYTES, SLOT_BYTES = PC::SLOT_BYTES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint64_t xbar[2][2];   // FC1 exchange: [warp pair][chunk parity], 64 arrivals
    // WGRAD: both CTAs' K tails written (the first CTA's, 2 arrivals); the tail buffer free
    // again (each CTA's, the pair MMA's commit)
    __shared__ uint64_t tail_full, tail_empty;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_off[kMaxE + 1];
    __shared__ int s_start[kMaxE + 1];
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = sm100::cluster_ctarank();
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = sm100::smem_u32(smem);

    // ---------------------------------------------------------------- set-up (on chip)
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            sm100::mbar_init(&full_bar[s], 1);
            sm100::mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            sm100::mbar_init(&tfull_bar[b], 1);
            sm100::mbar_init(&tempty_bar[b], 2 * 4);   // one lane of each epilogue warp of both CTAs
        }
        sm100::mbar_init(&drain_bar, 1);
        for (int i = 0; i < 4; ++i) sm100::mbar_init(&xbar[i >> 1][i & 1], 64);
        sm100::mbar_init(&tail_full, 2);
        sm100::mbar_init(&tail_empty, 1);
        s_abort = 0;
        sm100::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        sm100::prefetch_tmap(&tmW0);
        if constexpr (OP == Op::FC1 || OP == Op::DGRAD_FC1) sm100::prefetch_tmap(&tmW1);
        sm100::prefetch_tmap(&tmX);
    }
    if (warp == 1) {
        sm100::tmem_alloc_pair(&s_tmem_base, TMEM_COLS);
        sm100::tmem_relinquish_pair();
    }
    // both CTAs' barriers are initialised before either CTA touches the other's
    sm100::tc_fence_before();
    sm100::cluster_sync();
    sm100::tc_fence_after();

    // from here on the kernel reads what earlier kernels on the stream wrote
    pdl_wait();
    const uint64_t wait_ns = device_wait_limit(args.err);   // pipeline waits' limit
    const int E = args.E;
    for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = args.group_offsets[i];
    __syncthreads();
    if (warp == 2) {
        // s_start[e] = pair tiles before expert e (feature blocks x token blocks)
        const int seg = (E + 31) / 32;
        const int e0 = lane * seg;
        auto tiles_of = [&](int e) {
            if constexpr (OP == Op::WGRAD) return args.nt_m * args.nt_n;
            int rows = s_off[e + 1] - s_off[e];
            if (rows < 0) rows = 0;
            return ((rows + BT - 1) / BT) * args.n_fb;
        };
        int sum = 0;
        for (int i = 0; i < seg; ++i)
            if (e0 + i < E) sum += tiles_of(e0 + i);
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - sum;
        for (int i = 0; i < seg; ++i) {
            if (e0 + i < E) {
                s_start[e0 + i] = run;
                run += tiles_of(e0 + i);
            }
        }
        const bool offs_ok = group_offsets_in_bounds(s_off, E, args.rows_cap, lane, args.err);
        if (lane == 31) s_start[E] = offs_ok ? incl : 0;   // no tiles for offsets out of bounds
    }
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;
    const int total = s_start[E];
    const int G = (int)(gridDim.x >> 1), cid = (int)(blockIdx.x >> 1);
    const int rounds = (total + G - 1) / G;
    const int kblocks = args.K / 64;
    volatile int *abort = &s_abort;

    if (warp == 0 && OP == Op::WGRAD) {
        // ============================================================ producer, WGRAD (both CTAs)
        // Lane 0 issues the TMA loads of the whole 16-row slices: this CTA's 128 gradient rows
        // (two 64-wide MN chunks of the A rows) and 128 gradient columns (of the B rows), 64
        // K rows (tokens) per stage, one 3-D box per operand.  An expert's last (rows mod 16) rows go into the tail
        // buffer, written by the whole warp: rows zero-padded to a 16-row slice in the MMA's
        // swizzled layout, so the pair MMAs never multiply a row of the next expert.  The tail
        // buffer sits outside the ring, so it takes no stage from the loads' lead over the MMAs.
        const uint32_t full0 = sm100::cluster_addr(&full_bar[0], 0);
        const uint32_t tail_full0 = sm100::cluster_addr(&tail_full, 0);
        uint8_t *tbuf = smem + STAGES * STAGE_BYTES + XBUF_BYTES + PC::STG_BYTES;
        int stage = 0;
        uint32_t phase = 0, tphase = 0;
        int issued = 0;
        bool ok = true;
        for (int r = 0; r < rounds && ok; ++r) {
            const int p = round_tile(r, cid, G, total);
            if (p < 0) continue;
            const WTile tl = decode_w(p, args, s_off);
            const int ntail = tl.rows - tl.full16;
            const int m0 = tl.m0 + (int)rank * 128, n0 = tl.n0 + (int)rank * 128;
            // the tail's 2 operands x 2 chunks x 16 K rows x 8 16-byte pieces, 16 per lane: loaded
            // into registers before the whole slices, so that their latency overlaps those stages
            uint4 tv[16];
            {
                const int64_t trow0 = (int64_t)tl.row0 + tl.full16;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int opnd = i >> 3, j = (i >> 2) & 1, k = 4 * (i & 3) + (lane >> 3), c16 = lane & 7;
                    tv[i] = make_uint4(0, 0, 0, 0);
                    if (k < ntail)
                        tv[i] = __ldg(reinterpret_cast<const uint4 *>(
                            opnd == 0 ? args.a_rows + (trow0 + k) * args.lda + m0 + j * 64 + c16 * 8
                                      : args.b_rows + (trow0 + k) * args.ldb + n0 + j * 64 + c16 * 8));
                }
            }
            for (int kb = 0; kb < tl.kblocks; ++kb) {
                bool got = true;
                if (lane == 0) got = sm100::mbar_wait(&empty_bar[stage], phase ^ 1u, abort, args.err, wait_ns);
                if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) { ok = false; break; }
                if (lane == 0) {
                    const uint32_t sa = smem_base + stage * STAGE_BYTES, sb = sa + A_BYTES;
                    const uint32_t fb_c = full0 + (uint32_t)(stage * sizeof(uint64_t));
                    if (rank == 0) sm100::mbar_arrive_expect_tx(&full_bar[stage], 2 * STAGE_BYTES);
                    // one 3-D box per operand: its two 64-column chunks of 64 K rows (measured
                    // on mixtral: 677 cycles per K step against 782 with four 2-D boxes)
                    const int krow = tl.row0 + kb * 64;
                    sm100::tma_load_3d_pair(sa, &tmW0, fb_c, 0, krow, m0 / 64);
                    sm100::tma_load_3d_pair(sb, &tmX, fb_c, 0, krow, n0 / 64);
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (ntail > 0) {
                // the previous tail has been multiplied; then the layout the TMA loads give
                // (128-byte swizzle), with the MN chunks 16 K rows apart
                bool got = true;
                if (lane == 0) got = sm100::mbar_wait(&tail_empty, tphase ^ 1u, abort, args.err, wait_ns);
                if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) { ok = false; break; }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int opnd = i >> 3, j = (i >> 2) & 1, k = 4 * (i & 3) + (lane >> 3), c16 = lane & 7;
                    *reinterpret_cast<uint4 *>(tbuf + opnd * 4096 + j * 2048 + k * 128 + ((c16 ^ (k & 7)) << 4)) = tv[i];
                }
                sm100::fence_proxy_async_smem();   // the generic writes -> the MMA's async proxy
                __syncwarp();
                if (lane == 0) sm100::mbar_arrive_cluster(tail_full0);
                tphase ^= 1u;
            }
        }
        if (!ok && lane == 0) {
            int st = stage;
            uint32_t ph = phase;
            for (int i = 0; i < STAGES && i < issued; ++i) {
                if (--st < 0) { st = STAGES - 1; ph ^= 1u; }
                int dummy = 0;
                sm100::mbar_wait(&empty_bar[st], ph, &dummy, nullptr, 10000000ull);
            }
        }
    } else if (warp == 0) {
        // ============================================================ producer (both CTAs)
        if (lane == 0) {
            const uint32_t full0 = sm100::cluster_addr(&full_bar[0], 0);   // the first CTA's barriers
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int r = 0; r < rounds && ok && OP == Op::DSWIGLU; ++r) {
                const int p = round_tile(r, cid, G, total);
                if (p < 0) continue;
                const MTile tl = decode_m(p, args, s_off, s_start);
                const int arow = tl.m0 + (int)rank * 128;          // this CTA's 128 token rows
                const int brow = tl.fb * BT + (int)rank * 128;     // and its 128 rows (features) of W_down
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!sm100::mbar_wait(&empty_bar[stage], phase ^ 1u, abort, args.err, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_base + stage * STAGE_BYTES, sb = sa + A_BYTES;
                    const uint32_t fb_c = full0 + (uint32_t)(stage * sizeof(uint64_t));
                    if (rank == 0) sm100::mbar_arrive_expect_tx(&full_bar[stage], 2 * STAGE_BYTES);
                    const int k0 = kb * 64;
                    sm100::tma_load_2d_pair(sa, &tmX, fb_c, k0, arow);          // dy_perm, K-major
                    sm100::tma_load_3d_pair(sb, &tmW0, fb_c, k0, brow, tl.e);   // W_down [E][F][H], K-major
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            for (int r = 0; r < rounds && ok && OP != Op::WGRAD && OP != Op::DSWIGLU; ++r) {
                const int p = round_tile(r, cid, G, total);
                if (p < 0) continue;
                const PTile tl = decode(p, args, s_off, s_start);
                const int trow = tl.t0 + (int)rank * (tl.n >> 1);   // this CTA's half of the tokens
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!sm100::mbar_wait(&empty_bar[stage], phase ^ 1u, abort, args.err, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_base + stage * STAGE_BYTES, sb = sa + A_BYTES;
                    const uint32_t fb_c = full0 + (uint32_t)(stage * sizeof(uint64_t));
                    if (rank == 0) sm100::mbar_arrive_expect_tx(&full_bar[stage], 2 * STAGE_BYTES);
                    const int k0 = kb * 64;
                    if constexpr (OP == Op::FC1) {
                        // 64 gate then 64 up feature columns of W [E][K][F] (MN-major chunks)
                        const int f0 = tl.fb * 128 + (int)rank * 64;
                        sm100::tma_load_3d_pair(sa, &tmW0, fb_c, f0, k0, tl.e);
                        sm100::tma_load_3d_pair(sa + 8192, &tmW1, fb_c, f0, k0, tl.e);
                    } else if constexpr (OP == Op::DGRAD_FC1) {
                        // 128 rows (hidden units) of W_gate [E][H][F] for K < F, then of W_up
                        const int r0 = tl.fb * 256 + (int)rank * 128;
                        if (k0 < args.k_split) sm100::tma_load_3d_pair(sa, &tmW0, fb_c, k0, r0, tl.e);
                        else sm100::tma_load_3d_pair(sa, &tmW1, fb_c, k0 - args.k_split, r0, tl.e);
                    } else {
                        // 128 output columns of W_down [E][K][H]
                        const int c0 = tl.fb * 256 + (int)rank * 128;
                        sm100::tma_load_3d_pair(sa, &tmW0, fb_c, c0, k0, tl.e);
                        sm100::tma_load_3d_pair(sa + 8192, &tmW0, fb_c, c0 + 64, k0, tl.e);
                    }
                    sm100::tma_load_2d_pair(sb, &tmX, fb_c, k0, trow);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // the CTA's copies in flight land before it can exit: its own stages are
                // free again once the first CTA's MMAs (or its drain) release them
                int st = stage;
                uint32_t ph = phase;
                for (int i = 0; i < STAGES && i < issued; ++i) {
                    if (--st < 0) { st = STAGES - 1; ph ^= 1u; }
                    int dummy = 0;
                    sm100::mbar_wait(&empty_bar[st], ph, &dummy, nullptr, 10000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer (first CTA)
        // The whole warp runs the loop and computes the operand descriptors (warp-uniform
        // values); one elected lane issues the MMAs and their commits.  Measured: the same
        // loop with the descriptor arithmetic inside a one-lane branch issued an MMA every
        // ~170 cycles, below the tensor pipe's rate.
        if (rank == 0) {
            // weights MN-major (forward) or K-major (dgrad); tokens K-major
            const uint64_t a_desc0 = a_kmajor<OP>() ? sm100::sdesc_sw128(smem_base, 16, 1024)
                                                    : sm100::sdesc_sw128(smem_base, 8192, 1024);
            const uint64_t b_desc0 = sm100::sdesc_sw128(smem_base + A_BYTES, 16, 1024);
            constexpr uint64_t A_KSTEP = a_kmajor<OP>() ? (32 >> 4) : (2048 >> 4), B_KSTEP = 32 >> 4,
                               STAGE_STEP = STAGE_BYTES >> 4;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued_any = false;
            if constexpr (OP == Op::WGRAD) {
                // both operands MN-major; only the whole 16-row slices of the expert's rows
                const uint64_t wa0 = sm100::sdesc_sw128(smem_base, 8192, 1024);
                const uint64_t wb0 = sm100::sdesc_sw128(smem_base + A_BYTES, 8192, 1024);
                constexpr uint64_t KSTEP = 2048 >> 4;
                constexpr uint32_t idesc = sm100::idesc_bf16(256, 256, true, true);
                // the tail buffer: MN chunks 16 K rows (2048 B) apart
                const uint32_t tbuf_s = smem_base + STAGES * STAGE_BYTES + PC::XBUF_BYTES + PC::STG_BYTES;
                const uint64_t ta = sm100::sdesc_sw128(tbuf_s, 2048, 1024);
                const uint64_t tb = sm100::sdesc_sw128(tbuf_s + 4096, 2048, 1024);
                uint32_t tphase = 0;
                for (int r = 0; r < rounds && ok; ++r) {
                    const int p = round_tile(r, cid, G, total);
                    if (p < 0) continue;
                    const WTile tl = decode_w(p, args, s_off);
                    const int ntail = tl.rows - tl.full16;
                    if (tl.rows == 0) continue;   // the epilogue writes this tile's zeros alone
                    const bool got_acc =
                        sm100::mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1u, abort, args.err, wait_ns);
                    if (__any_sync(0xFFFFFFFFu, !got_acc)) { ok = false; break; }
                    sm100::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BT);
                    for (int kb = 0; kb < tl.kblocks; ++kb) {
                        const bool got = sm100::mbar_wait(&full_bar[stage], phase, abort, args.err, wait_ns);
                        if (__any_sync(0xFFFFFFFFu, !got)) { ok = false; break; }
                        sm100::tc_fence_after();
                        const uint64_t ad = wa0 + (uint64_t)stage * STAGE_STEP;
                        const uint64_t bd = wb0 + (uint64_t)stage * STAGE_STEP;
                        const int left = (tl.full16 - kb * 64) >> 4;   // 16-row slices left
                        const int kk_end = left < 4 ? left : 4;
                        // a whole stage as four straight-line MMAs, as the other ops issue them
                        const uint32_t acc0 = kb != 0 ? 1u : 0u;
                        if (sm100::elect_one()) {
                            if (kk_end == 4) {
                                sm100::mma_bf16_pair(d_tmem, ad, bd, idesc, acc0);
                                sm100::mma_bf16_pair(d_tmem, ad + KSTEP, bd + KSTEP, idesc, 1u);
                                sm100::mma_bf16_pair(d_tmem, ad + 2 * KSTEP, bd + 2 * KSTEP, idesc, 1u);
                                sm100::mma_bf16_pair(d_tmem, ad + 3 * KSTEP, bd + 3 * KSTEP, idesc, 1u);
                            } else {
                                for (int kk = 0; kk < kk_end; ++kk)
                                    sm100::mma_bf16_pair(d_tmem, ad + kk * KSTEP, bd + kk * KSTEP, idesc,
                                                         (kb | kk) != 0 ? 1u : 0u);
                            }
                            sm100::mma_commit_pair(&empty_bar[stage], 0x3);
                        }
                        __syncwarp();
                        issued_any = true;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    if (ntail > 0) {   // the zero-padded tail written by both producers
                        const bool got =
                            sm100::mbar_wait_cluster(&tail_full, tphase, abort, args.err, wait_ns);
                        if (__any_sync(0xFFFFFFFFu, !got)) { ok = false; break; }
                        tphase ^= 1u;
                        sm100::tc_fence_after();
                        if (sm100::elect_one()) {
                            sm100::mma_bf16_pair(d_tmem, ta, tb, idesc, tl.kblocks > 0 ? 1u : 0u);
                            sm100::mma_commit_pair(&tail_empty, 0x3);
                        }
                        __syncwarp();
                        issued_any = true;
                    }
                    if (sm100::elect_one()) sm100::mma_commit_pair(&tfull_bar[acc], 0x3);
                    __syncwarp();
                    if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                }
            }
            for (int r = 0; r < rounds && ok && OP != Op::WGRAD; ++r) {
                const int p = round_tile(r, cid, G, total);
                if (p < 0) continue;
                // tokens on N: the token block's width rounded up to 16; DSWIGLU: 256 features
                const int n_mma = OP == Op::DSWIGLU ? BT : decode(p, args, s_off, s_start).n;
                const uint32_t idesc = sm100::idesc_bf16(256, n_mma, !a_kmajor<OP>(), false);
                const bool got_acc =
                    sm100::mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1u, abort, args.err, wait_ns);
                if (__any_sync(0xFFFFFFFFu, !got_acc)) { ok = false; break; }
                sm100::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BT);
                for (int kb = 0; kb < kblocks; ++kb) {
                    const bool got = sm100::mbar_wait(&full_bar[stage], phase, abort, args.err, wait_ns);
                    if (__any_sync(0xFFFFFFFFu, !got)) { ok = false; break; }
                    sm100::tc_fence_after();
                    const uint64_t ad = a_desc0 + (uint64_t)stage * STAGE_STEP;
                    const uint64_t bd = b_desc0 + (uint64_t)stage * STAGE_STEP;
                    if (sm100::elect_one()) {
                        sm100::mma_bf16_pair(d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u);
                        sm100::mma_bf16_pair(d_tmem, ad + A_KSTEP, bd + B_KSTEP, idesc, 1u);
                        sm100::mma_bf16_pair(d_tmem, ad + 2 * A_KSTEP, bd + 2 * B_KSTEP, idesc, 1u);
                        sm100::mma_bf16_pair(d_tmem, ad + 3 * A_KSTEP, bd + 3 * B_KSTEP, idesc, 1u);
                        sm100::mma_commit_pair(&empty_bar[stage], 0x3);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (sm100::elect_one()) sm100::mma_commit_pair(&tfull_bar[acc], 0x3);
                __syncwarp();
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
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
        const int q = warp & 3;              // TMEM lane quarter of this warp
        const uint32_t tempty0 = sm100::cluster_addr(&tempty_bar[0], 0);
        uint8_t *stg = smem + STAGES * STAGE_BYTES + XBUF_BYTES + q * 2 * SLOT_BYTES;
        const uint32_t stg_s = smem_base + STAGES * STAGE_BYTES + XBUF_BYTES + q * 2 * SLOT_BYTES;
        int slot = 0;
        auto slot_open = [&]() {
            if (lane == 0) sm100::bulk_wait_read<1>();   // the store that last read this slot is done
            __syncwarp();
        };
        auto slot_store = [&](const CUtensorMap *tm, int col, int row) {
            sm100::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                sm100::tma_store_2d(tm, stg_s + slot * SLOT_BYTES, col, row);
                sm100::bulk_commit();
            }
            slot ^= 1;
        };
        // 16 tokens x 32 bf16 features (this thread's feature = lane): staged as 64-byte
        // token rows (pairs of lanes swap values so that every store is a 32-bit word)
        auto put_bf16x16 = [&](const float (&v)[16]) {
            uint32_t *w = reinterpret_cast<uint32_t *>(stg + slot * SLOT_BYTES);
#pragma unroll
            for (int t = 0; t < 16; t += 2) {
                const float send = (lane & 1) ? v[t] : v[t + 1];
                const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 1);
                __nv_bfloat162 pk;
                int row;
                if (lane & 1) { pk = __floats2bfloat162_rn(recv, v[t + 1]); row = t + 1; }
                else { pk = __floats2bfloat162_rn(v[t], recv); row = t; }
                w[row * 16 + (lane >> 1)] = *reinterpret_cast<uint32_t *>(&pk);
            }
        };
        // store 16 tokens (rows row0 ..) of one feature column block; nv of them valid
        auto store_bf16x16 = [&](const float (&v)[16], const CUtensorMap *tm, __nv_bfloat16 *base, int64_t ld,
                                 int col, int row0, int nv) {
            if (nv >= 16) {
                slot_open();
                put_bf16x16(v);
                slot_store(tm, col, row0);
            } else if (nv > 0) {
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    if (t < nv) base[(int64_t)(row0 + t) * ld + col + lane] = __float2bfloat16_rn(v[t]);
            }
        };
        auto route_weight = [&](int row, bool valid) {
            const int src = valid ? args.src_of_row[row] : -1;
            return src >= 0 ? args.route_w[src] : 0.0f;
        };

        int acc = 0;
        uint32_t acc_phase = 0;
        int chunk_parity = 0;
        uint32_t xphase = 0;   // bit b: parity of the next wait on xbar[pair][b]
        bool alive = true;
        if constexpr (OP == Op::WGRAD) {
            // this thread's gradient row; 32 columns at a time staged as 32 rows x 64 B (64-byte
            // swizzle) and stored by TMA in boxes of 16 fp32 or 32 bf16 columns x 32 rows
            auto put_w = [&](int j, uint4 v) {
                *reinterpret_cast<uint4 *>(stg + slot * SLOT_BYTES + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
            };
            for (int r = 0; r < rounds && alive; ++r) {
                const int p = round_tile(r, cid, G, total);
                if (p < 0) continue;
                const WTile tl = decode_w(p, args, s_off);
                const bool mma = tl.rows > 0;   // else an expert without rows: exact zeros
                if (mma) {
                    const bool got = sm100::mbar_wait(&tfull_bar[acc], acc_phase, abort, args.err, wait_ns);
                    if (__any_sync(0xFFFFFFFFu, !got)) break;
                    sm100::tc_fence_after();
                }
                const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BT);
                const int64_t grow0 = (int64_t)tl.e * args.M + tl.m0 + (int)rank * 128 + q * 32;
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    float v[32];
                    if (mma) {
                        uint32_t raw[32];
                        sm100::tmem_ld32(tacc + c0, raw);
                        sm100::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                    }
                    const int ncol = tl.n0 + c0;
                    const bool second = args.n_split > 0 && ncol >= args.n_split;
                    const int col = second ? ncol - args.n_split : ncol;
                    if (args.w_bf16) {   // 32 bf16 columns: one 32-row x 64-byte slot, one TMA store
                        slot_open();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 pk;
                            __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                            for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
                            put_w(j, pk);
                        }
                        slot_store(second ? &tmStash : &tmOut, col, (int)grow0);
                        continue;
                    }
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        slot_open();
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            put_w(j, make_uint4(__float_as_uint(v[16 * hf + 4 * j]), __float_as_uint(v[16 * hf + 4 * j + 1]),
                                                __float_as_uint(v[16 * hf + 4 * j + 2]),
                                                __float_as_uint(v[16 * hf + 4 * j + 3])));
                        slot_store(second ? &tmStash : &tmOut, col + 16 * hf, (int)grow0);
                    }
                }
                if (mma) {
                    sm100::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) sm100::mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
                    if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                }
            }
            alive = false;   // the loop below is the other ops'
        }
        if constexpr (OP == Op::DSWIGLU) {
            // this thread's token row: per 32-feature chunk, dh from TMEM, g and u from the stash,
            // dg and du (bf16) staged as 32 rows x 64 B in the 64-byte swizzle and stored by TMA
            // in boxes of 32 columns x 32 rows -- row by row for a warp whose rows leave the expert
            auto put_h = [&](int j, uint4 v) {
                *reinterpret_cast<uint4 *>(stg + slot * SLOT_BYTES + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
            };
            auto pack8 = [](const float *v) {
                uint4 pk;
                __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                return pk;
            };
            auto unpack8 = [](const uint4 &pk, float *v) {
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&pk);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(h2[i]);
                    v[2 * i] = f.x;
                    v[2 * i + 1] = f.y;
                }
            };
            const int F = args.N_out;
            const int64_t ld = 2 * (int64_t)F;   // stash and output row pitch
            for (int r = 0; r < rounds && alive; ++r) {
                const int p = round_tile(r, cid, G, total);
                if (p < 0) continue;
                const MTile tl = decode_m(p, args, s_off, s_start);
                const bool got = sm100::mbar_wait(&tfull_bar[acc], acc_phase, abort, args.err, wait_ns);
                if (__any_sync(0xFFFFFFFFu, !got)) break;
                sm100::tc_fence_after();
                const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BT);
                const int64_t wrow0 = (int64_t)tl.m0 + (int)rank * 128 + q * 32;   // this warp's first row
                const int64_t row = wrow0 + lane;
                const bool whole = wrow0 + 32 <= tl.m_end && wrow0 + 32 <= args.rows_cap;   // warp-uniform
                const bool valid = row < tl.m_end && row < args.rows_cap;
                // the stash values of a chunk are loaded one chunk ahead of their use
                uint4 gq[4] = {}, uq[4] = {}, gn[4] = {}, un[4] = {};
                auto load_stash = [&](int c0, uint4 (&g)[4], uint4 (&u)[4]) {
                    if (whole || valid) {
                        const uint4 *gs = reinterpret_cast<const uint4 *>(args.aux + row * ld + tl.fb * BT + c0);
                        const uint4 *us = reinterpret_cast<const uint4 *>(args.aux + row * ld + F + tl.fb * BT + c0);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            g[j] = __ldg(gs + j);
                            u[j] = __ldg(us + j);
                        }
                    }
                };
                load_stash(0, gq, uq);
#pragma unroll 1
                for (int c0 = 0; c0 < BT; c0 += 32) {
                    if (c0 + 32 < BT) load_stash(c0 + 32, gn, un);
                    uint32_t d[32];
                    sm100::tmem_ld32(tacc + c0, d);
                    sm100::tmem_ld_wait();
                    const int f = tl.fb * BT + c0;   // feature of this chunk's first column
                    float dg[32], du[32];
                    if (whole || valid) {
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            float gv[8], uv[8];
                            unpack8(gq[c / 8], gv);
                            unpack8(uq[c / 8], uv);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float dh = __uint_as_float(d[c + i]);
                                const float G = gv[i], U = uv[i];
                                if (args.clamp) {   // clamped inputs; zero derivative outside the bounds
                                    const float gc = fminf(fmaxf(G, args.gate_lo), args.gate_hi);
                                    const float uc = fminf(fmaxf(U, args.up_lo), args.up_hi);
                                    const float sg = __fdividef(1.0f, 1.0f + __expf(-gc));
                                    const bool gin = G >= args.gate_lo && G <= args.gate_hi;
                                    const bool uin = U >= args.up_lo && U <= args.up_hi;
                                    dg[c + i] = gin ? dh * uc * sg * (1.0f + gc * (1.0f - sg)) : 0.0f;
                                    du[c + i] = uin ? dh * gc * sg : 0.0f;
                                } else {
                                    const float sg = __fdividef(1.0f, 1.0f + __expf(-G));
                                    dg[c + i] = dh * U * sg * (1.0f + G * (1.0f - sg));
                                    du[c + i] = dh * G * sg;
                                }
                            }
                        }
                    }
                    if (whole) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {   // dg to columns f.., du to F + f..
                            const float *v = half ? du : dg;
                            slot_open();
#pragma unroll
                            for (int j = 0; j < 4; ++j) put_h(j, pack8(v + 8 * j));
                            slot_store(&tmOut, half ? F + f : f, (int)wrow0);
                        }
                    } else if (valid) {
                        uint4 *dgr = reinterpret_cast<uint4 *>(args.y16 + row * ld + f);
                        uint4 *dur = reinterpret_cast<uint4 *>(args.y16 + row * ld + F + f);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            dgr[j] = pack8(dg + 8 * j);
                            dur[j] = pack8(du + 8 * j);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        gq[j] = gn[j];
                        uq[j] = un[j];
                    }
                }
                sm100::tc_fence_before();
                __syncwarp();
                if (lane == 0) sm100::mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            alive = false;   // the loop below is the other ops'
        }
        for (int r = 0; r < rounds && alive; ++r) {
            const int p = round_tile(r, cid, G, total);
            if (p < 0) continue;
            const PTile tl = decode(p, args, s_off, s_start);
            const bool got = sm100::mbar_wait(&tfull_bar[acc], acc_phase, abort, args.err, wait_ns);
            if (__any_sync(0xFFFFFFFFu, !got)) break;
            sm100::tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BT);

            if constexpr (OP == Op::FC1) {
                const int pr = q & 1;                  // feature half of this warp
                const bool gate = q < 2;               // lanes 0..63 gate, 64..127 up
                const int F = args.N_out;
                const int fcol = tl.fb * 128 + (int)rank * 64 + pr * 32;   // first of this warp's 32 features
                float *xg = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES) + pr * 2048;   // 8 KB per pair
#pragma unroll 1
                for (int c0 = 0; c0 < tl.n; c0 += 32) {
                    uint32_t raw[32];
                    sm100::tmem_ld32(tacc + c0, raw);
                    sm100::tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
                    if (args.stash) {   // unclamped g (gate warps) or u (up warps), bf16
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            float sv[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) sv[i] = v[16 * hf + i];
                            store_bf16x16(sv, &tmStash, args.stash, 2 * (int64_t)F, gate ? fcol : F + fcol,
                                          tl.t0 + c0 + 16 * hf, tl.nvalid - c0 - 16 * hf);
                        }
                    }
                    if (args.clamp) {
                        const float lo = gate ? args.gate_lo : args.up_lo, hi = gate ? args.gate_hi : args.up_hi;
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = fminf(fmaxf(v[i], lo), hi);
                    }
                    // exchange: the gate warp keeps tokens 0..15 of the chunk and hands over
                    // 16..31; the up warp the other way round
                    float *xb = xg + chunk_parity * 1024;   // [direction][16 tokens][32 lanes]
                    if (gate) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) xb[t * 32 + lane] = v[16 + t];
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) xb[512 + t * 32 + lane] = v[t];
                    }
                    uint64_t *xbr = &xbar[pr][chunk_parity];
                    sm100::mbar_arrive(xbr);
                    const bool xok = sm100::mbar_wait(xbr, (xphase >> chunk_parity) & 1u, abort, args.err, wait_ns);
                    xphase ^= 1u << chunk_parity;
                    if (__any_sync(0xFFFFFFFFu, !xok)) { alive = false; break; }
                    float hv[16];
                    if (gate) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) hv[t] = silu(v[t]) * xb[512 + t * 32 + lane];
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) hv[t] = silu(xb[t * 32 + lane]) * v[16 + t];
                    }
                    chunk_parity ^= 1;
                    const int tok0 = c0 + (gate ? 0 : 16);          // first token of this warp's 16
                    const int nv = tl.nvalid - tok0;
                    if (args.route_w) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) hv[t] *= route_weight(tl.t0 + tok0 + t, t < nv);
                    }
                    store_bf16x16(hv, &tmOut, args.h, F, fcol, tl.t0 + tok0, nv);
                }
                if (!alive) break;
            } else {   // FC2 (y_perm, bf16 rows) and DGRAD_FC1 (dx_perm, fp32 rows)
                const int H = args.N_out;
                const int hcol = tl.fb * 256 + (int)rank * 128 + q * 32;   // this warp's 32 output columns
#pragma unroll 1
                for (int c0 = 0; c0 < tl.n; c0 += 32) {
                    uint32_t raw[32];
                    sm100::tmem_ld32(tacc + c0, raw);
                    sm100::tmem_ld_wait();
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int tok0 = c0 + 16 * hf;
                        const int nv = tl.nvalid - tok0;
                        float v[16];
#pragma unroll
                        for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(raw[16 * hf + t]);
                        if (args.route_w) {
#pragma unroll
                            for (int t = 0; t < 16; ++t) v[t] *= route_weight(tl.t0 + tok0 + t, t < nv);
                        }
                        if constexpr (OP == Op::FC2) {
                            store_bf16x16(v, &tmOut, args.y16, H, hcol, tl.t0 + tok0, nv);
                        } else if (nv >= 16) {
                            slot_open();
                            float *w = reinterpret_cast<float *>(stg + slot * SLOT_BYTES);
#pragma unroll
                            for (int t = 0; t < 16; ++t) w[t * 32 + lane] = v[t];   // 128-byte token rows
                            slot_store(&tmOut, hcol, tl.t0 + tok0);
                        } else if (nv > 0) {
#pragma unroll
                            for (int t = 0; t < 16; ++t)
                                if (t < nv) args.y[(int64_t)(tl.t0 + tok0 + t) * H + hcol + lane] = v[t];
                        }
                    }
                }
            }
            sm100::tc_fence_before();
            __syncwarp();
            if (lane == 0) sm100::mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        // every TMA store of this warp has finished before the CTA can exit
        if (lane == 0) sm100::bulk_wait_all();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    sm100::tc_fence_before();
    __syncthreads();
    sm100::cluster_sync();   // no arrive or copy of one CTA still targets the other
    if (warp == 1) {
        sm100::tc_fence_after();
        sm100::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace gp
}  // namespace moe

namespace moe {
namespace gp {

// Host launch: clusters of two CTAs, as many as can be resident at once (the schedule is
// persistent), at most one per pair tile; programmatic stream serialization as every
// kernel of the library.
template <Op OP>
moe_status_t launch(const CUtensorMap &w0, const CUtensorMap &w1, const CUtensorMap &x, const CUtensorMap &out,
                    const CUtensorMap &stash, const Args &args, int64_t tiles_bound, cudaStream_t s) {
    if (tiles_bound <= 0) return MOE_OK;
    auto kern = pair_gemm_kernel<OP>;
    constexpr int smem = PCfg<OP>::SMEM_BYTES;
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
    if (cudaLaunchKernelEx(&cfg, kern, w0, w1, x, out, stash, args) != cudaSuccess) return MOE_ERR_CUDA;
    return launch_status();
}

}  // namespace gp
}  // namespace moe
