// grouped_gemm.cuh -- persistent, warp-specialised grouped GEMM on tcgen05 for the
// expert FFN (forward, backward and the MXFP8 forward).
//
// One CTA per SM, 6 or 10 warps:
//   warp 0      TMA producer (one lane): A and B tiles (and, for MXFP8, their
//               block scales) -> a ring of smem stages
//   warp 1      MMA issuer (one elected lane issues tcgen05.mma, M=128 x N=BN; K=16 per
//               instruction for bf16, K=32 for E4M3); fp32 accumulators live in
//               TMEM (double-buffered for bf16, single for MXFP8, whose scales
//               take the other half of TMEM)
//   warps 2..5  epilogue: tcgen05.ld -> fused activation -> swizzled smem slots ->
//   (or 2..9)   TMA stores (row by row only for a warp whose rows cross a group end)
// Tiles are scheduled on the device from group_offsets (no host round trip).
//
// Ops (A row = one permuted route unless stated):
//   FC1_SWIGLU     h = silu(x W_gate) * (x W_up)        M-grouped, K = H
//   FC2            y = h W_down (bf16 out)              M-grouped, K = F
//   DGRAD_DSWIGLU  dh = dy W_down^T, then dSwiGLU       M-grouped, K = H
//   DGRAD_FC1      dx = dg W_gate^T + du W_up^T (fp32)   M-grouped, K = 2F
//   WGRAD_DOWN     dW_down[e] = h_e^T dy_e (fp32 / bf16) K-grouped (K = rows of e)
//   WGRAD_GATEUP   [dW_gate|dW_up][e] = x_e^T [dg|du]_e K-grouped
//   FC1_MX         FC1_SWIGLU on MXFP8 operands; h is quantised to MXFP8 (along F)
//                  in the epilogue, scales written in the MMA tile layout
//   FC2_MX         FC2 on MXFP8 operands (bf16 out)
// ("Add MoE + expert-parallel Python API surface, PyTorch reference, and
// tests", Summary: SwiGLU experts, fc1_c stash, backward, MXFP8 operands;
// "[Draft][JAX] MoE block optimization": fused grouped GEMM + SwiGLU and
// grouped_gemm_dswiglu; "[JAX] Expert Parallelism": zero wgrad for experts
// with no tokens; "MoE training optimization": MXFP8 grouped GEMM.)
#pragma once

#include "common.cuh"
#include "mx.cuh"
#include "sm100.cuh"

namespace moe {
namespace gg {

enum class Op : int { FC1_SWIGLU, FC2, DGRAD_DSWIGLU, DGRAD_FC1, WGRAD_DOWN, WGRAD_GATEUP, FC1_MX, FC2_MX };

constexpr int BM = 128;
constexpr int UMMA_K = 16;
constexpr int kMaxE = 1024;

template <Op OP>
struct Traits {
    static constexpr bool mx = (OP == Op::FC1_MX || OP == Op::FC2_MX);
    static constexpr bool k_grouped = (OP == Op::WGRAD_DOWN || OP == Op::WGRAD_GATEUP);
    static constexpr bool a_mn = k_grouped;                       // A is MN-major only for wgrad
    static constexpr bool b_mn = (OP == Op::FC1_SWIGLU || OP == Op::FC2 || k_grouped);
    static constexpr bool b_two = (OP == Op::FC1_SWIGLU || OP == Op::DGRAD_FC1 || OP == Op::FC1_MX);
    static constexpr bool swiglu = (OP == Op::FC1_SWIGLU || OP == Op::FC1_MX);
    static constexpr int BK = mx ? 128 : 64;   // K elements per stage: one 128-byte swizzle row
};

struct Args {
    const int32_t *group_offsets;   // [E+1]
    int E;
    int M;            // K-grouped: rows of each expert's output matrix
    int N;            // output columns (FC1: F; FC2: H; DSWIGLU: F; DGRAD_FC1: H; WGRAD: N)
    int K;            // M-grouped contraction length
    int n_tiles;      // tiles along N
    int m_tiles;      // K-grouped: tiles along M
    int k_split;      // DGRAD_FC1: K index where B switches from W_gate to W_up (= F)
    int n_split;      // WGRAD_GATEUP: column where output switches from out0 to out1 (= F)
    int64_t rows_cap; // rows of the permuted tensors
    __nv_bfloat16 *out0;   // FC1: h; DSWIGLU: [dg | du]; FC2, FC2_MX: y_perm
    float *out_f32;        // DGRAD_FC1: dx_perm; WGRAD: dW_down / dW_gate (row pitch ld0)
    int64_t ld0;
    __nv_bfloat16 *out1;   // FC1, FC1_MX: fc1_c stash (nullable)
    float *out1_f32;       // WGRAD_GATEUP: dW_up (row pitch ld1)
    int64_t ld1;
    const __nv_bfloat16 *aux;   // DSWIGLU: fc1_c
    int64_t ld_aux;
    int64_t expert_stride;      // K-grouped: elements between experts' outputs
    // MXFP8: A scales in tile layout [mtile][K/128][512]; B scales [E][K/128][N_B/128][512]
    const uint8_t *sfa;
    const uint8_t *sfb0;
    const uint8_t *sfb1;
    const uint8_t *b0_tiles;   // MXFP8: weight codes in 16 KB pre-swizzled blocks [E][K/128][N_B/128]
    const uint8_t *b1_tiles;   // FC1_MX: the W_up codes
    int nb_rows;          // MXFP8: rows (N) of each expert's B matrix
    uint8_t *out_q;       // FC1_MX: quantised h [rows, N] (E4M3)
    uint8_t *out_sf;      // FC1_MX: h scales in tile layout [mtile][N/128][512]
    // FC1_SWIGLU / FC2: the router weight of each row's route applied in the epilogue
    // (h or y scaled by route_w[src_of_row[row]]; padding rows get 0); null = unweighted
    const float *route_w;
    const int32_t *src_of_row;
    // FC1_SWIGLU / DGRAD_DSWIGLU: optional clamp of the SwiGLU inputs (clamp != 0): g to
    // [gate_lo, gate_hi] and u to [up_lo, up_hi] before SwiGLU, inclusive bounds
    int clamp;
    float gate_lo, gate_hi, up_lo, up_hi;
    // WGRAD_*: the gradients are stored as bf16 in out0 / out1 (row pitch ld0 / ld1) instead of
    // fp32 in out_f32 / out1_f32
    int w_bf16;
    uint32_t *err;
};

template <Op OP, int BN>
struct Cfg {
    static constexpr bool MX = Traits<OP>::mx;
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = BN * 128;
    static constexpr int SF_BYTES = MX ? 512 + (BN / 128) * 512 : 0;
    static constexpr int STAGE_BYTES = (A_BYTES + B_BYTES + SF_BYTES + 1023) / 1024 * 1024;
    // Epilogue warps: eight (two per TMEM lane quarter, alternate 32-column chunks) for the ops
    // whose chunks are independent stores -- FC2, FC2_MX, DGRAD_FC1 and the weight gradients,
    // where the epilogue is exposed (the MXFP8 single accumulator) or outweighs a short K loop
    // (experts with few rows) -- with one 2 KB staging slot each; four with two slots otherwise.
    static constexpr int EPI = (Traits<OP>::k_grouped || OP == Op::FC2 || OP == Op::FC2_MX || OP == Op::DGRAD_FC1) ? 8 : 4;
    static constexpr int THREADS = 64 + 32 * EPI;
    static constexpr int SLOTS = EPI == 8 ? 1 : 2;
    static constexpr int STG_BYTES = EPI * SLOTS * 2048;
    // dynamic shared memory: 227 KB per CTA less ~9 KB of static tables and barriers
    static constexpr int DYN_BUDGET = 232448 - 9216;
    static constexpr int FIT = (DYN_BUDGET - STG_BYTES - 1024) / STAGE_BYTES;
    static constexpr int STAGES = FIT < ((BN == 256) ? 4 : 6) ? FIT : ((BN == 256) ? 4 : 6);
    static constexpr int ACC_BUFS = MX ? 1 : 2;
    static constexpr int TMEM_COLS = MX ? 512 : ((2 * BN <= 256) ? 256 : 512);
    static constexpr int SF_COL0 = BN;                          // MXFP8 scale slots after the accumulator
    static constexpr int SF_COLS = 4 + 4 * (BN / 128);          // per stage: A (4) + B (4 per 128 rows)
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STG_BYTES + 1024;   // + alignment slack
    static_assert(STAGES >= 2, "shared memory ring too shallow");
    // two GEMM CTAs never share an SM, so the TMEM allocation made before the programmatic
    // launch wait never contends with a preceding GEMM still running there
    static_assert(2 * SMEM_BYTES > 232448, "GEMM CTAs must not be co-resident");
    // output columns produced per tile
    static constexpr int OUT_COLS = Traits<OP>::swiglu ? BN / 2 : BN;
    static_assert(!MX || SF_COL0 + STAGES * SF_COLS <= TMEM_COLS, "TMEM overflow");
};

// silu(g) = g * sigmoid(g) and sigmoid(g), with CUDA's fast exponential and fast
// division (__fdividef, within 2 ulp): far below the bf16 / E4M3 rounding of the
// stored results, and several times cheaper than IEEE division in the epilogue.
// For g -> -inf the denominator overflows to inf and both give 0.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_fast(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const float (&v)[32]) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 pk;
        __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
        d[q] = pk;
    }
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16 *src, float (&v)[32]) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 pk = __ldg(s + q);
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(p[i]);
            v[8 * q + 2 * i] = f.x;
            v[8 * q + 2 * i + 1] = f.y;
        }
    }
}

__device__ __forceinline__ void store_f32x32(float *dst, const uint32_t (&d)[32]) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d4[q] = make_uint4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
}

struct Tile {
    int e;
    int m0;      // M-grouped: first row in the permuted tensor; K-grouped: row in the expert's output
    int m_end;   // M-grouped: end of the group's rows
    int n0;      // first output column
    int kb;      // number of K blocks
    int k_row0;  // K-grouped: first permuted row of the group
    int k_rows;  // K-grouped: rows of the group
    int mtile;   // M-grouped: global 128-row tile id (expert-major), the MXFP8 scale tile
};

template <Op OP, int BN>
__device__ __forceinline__ Tile decode_tile(int t, const Args &a, const int *s_off, const int *s_start) {
    using TR = Traits<OP>;
    Tile tl;
    if constexpr (TR::k_grouped) {
        const int per = a.m_tiles * a.n_tiles;
        tl.e = t / per;
        const int local = t - tl.e * per;
        const int mb = local % a.m_tiles, nb = local / a.m_tiles;
        tl.m0 = mb * BM;
        tl.m_end = a.M;
        tl.n0 = nb * BN;
        const int r0 = s_off[tl.e], r1 = s_off[tl.e + 1];
        tl.k_row0 = r0;
        tl.k_rows = r1 > r0 ? r1 - r0 : 0;
        tl.kb = (tl.k_rows + TR::BK - 1) / TR::BK;
        tl.mtile = 0;
    } else {
        // largest e with s_start[e] <= t
        int lo = 0, hi = a.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_start[mid] <= t) lo = mid; else hi = mid - 1;
        }
        tl.e = lo;
        const int rows = s_off[lo + 1] - s_off[lo];
        const int nmb = (rows + BM - 1) / BM;
        const int local = t - s_start[lo];
        const int mb = local % nmb, nb = local / nmb;
        tl.m0 = s_off[lo] + mb * BM;
        tl.m_end = s_off[lo + 1];
        tl.n0 = nb * Cfg<OP, BN>::OUT_COLS;
        tl.kb = (a.K + TR::BK - 1) / TR::BK;
        tl.k_row0 = 0;
        tl.k_rows = 0;
        tl.mtile = s_start[lo] / a.n_tiles + mb;
    }
    return tl;
}

template <Op OP, int BN>
__global__ void __launch_bounds__(Cfg<OP, BN>::THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmC0,
                    const __grid_constant__ CUtensorMap tmC1, const Args args) {
    using TR = Traits<OP>;
    using C = Cfg<OP, BN>;
    constexpr int S = C::STAGES;
    constexpr int NACC = C::ACC_BUFS;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[S], empty_bar[S], tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_off[kMaxE + 1];
    __shared__ int s_start[kMaxE + 1];
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = sm100::smem_u32(smem);

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            sm100::mbar_init(&full_bar[s], 1);
            sm100::mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            sm100::mbar_init(&tfull_bar[b], 1);
            sm100::mbar_init(&tempty_bar[b], C::EPI * 32);
        }
        sm100::mbar_init(&drain_bar, 1);
        s_abort = 0;
        sm100::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        sm100::prefetch_tmap(&tmA);
        sm100::prefetch_tmap(&tmB0);
        if constexpr (TR::b_two) sm100::prefetch_tmap(&tmB1);
    }
    if (warp == 1) {
        sm100::tmem_alloc(&s_tmem_base, C::TMEM_COLS);
        sm100::tmem_relinquish();
    }
    // everything above is on-chip set-up; from here on the kernel reads what earlier
    // kernels on the stream wrote
    pdl_wait();
    const uint64_t wait_ns = device_wait_limit(args.err);   // pipeline waits' limit
    const int E = args.E;
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = args.group_offsets[i];
    __syncthreads();
    if (warp == 2) {
        // s_start[e] = tiles before expert e (M-grouped: m-blocks x n_tiles)
        const int seg = (E + 31) / 32;
        const int e0 = lane * seg;
        auto tiles_of = [&](int e) {
            if constexpr (TR::k_grouped) {
                return args.m_tiles * args.n_tiles;
            } else {
                int rows = s_off[e + 1] - s_off[e];
                if (rows < 0) rows = 0;
                return ((rows + BM - 1) / BM) * args.n_tiles;
            }
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
    const int total_tiles = s_start[E];
    volatile int *abort = &s_abort;

    if (warp == 0) {
        // ============================================================ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile<OP, BN>(t, args, s_off, s_start);
                for (int kb = 0; kb < tl.kb; ++kb) {
                    if (!sm100::mbar_wait(&empty_bar[stage], phase ^ 1u, abort, args.err, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_BYTES;
                    uint64_t *fb = &full_bar[stage];
                    sm100::mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES + C::SF_BYTES);
                    const int k0 = kb * TR::BK;
                    if constexpr (TR::mx) {
                        // E4M3 rows are K-contiguous: A [rows, K], B [E][N_B rows][K]
                        const uint32_t ssf = sb + C::B_BYTES;
                        const int kblocks = args.K / 128;
                        sm100::tma_load_2d(sa, &tmA, fb, k0, tl.m0);
                        sm100::bulk_load(ssf, args.sfa + ((int64_t)tl.mtile * kblocks + kb) * 512, 512, fb);
                        // weights: contiguous pre-swizzled 16 KB code blocks and 512-byte scale
                        // atoms, both ordered [E][K/128][N/128] -> plain bulk copies
                        const int nblk = args.nb_rows / 128;
                        const int64_t blk = ((int64_t)tl.e * kblocks + kb) * nblk + tl.n0 / 128;
                        if constexpr (OP == Op::FC1_MX) {
                            // 128 gate rows then 128 up rows, with their scale atoms
                            sm100::bulk_load(sb, args.b0_tiles + blk * 16384, 16384, fb);
                            sm100::bulk_load(sb + 16384, args.b1_tiles + blk * 16384, 16384, fb);
                            sm100::bulk_load(ssf + 512, args.sfb0 + blk * 512, 512, fb);
                            sm100::bulk_load(ssf + 1024, args.sfb1 + blk * 512, 512, fb);
                        } else {
                            sm100::bulk_load(sb, args.b0_tiles + blk * 16384, (BN / 128) * 16384, fb);
                            sm100::bulk_load(ssf + 512, args.sfb0 + blk * 512, (BN / 128) * 512, fb);
                        }
                    } else if constexpr (TR::k_grouped) {
                        const int krow = tl.k_row0 + k0;
                        sm100::tma_load_2d(sa, &tmA, fb, tl.m0, krow);
                        sm100::tma_load_2d(sa + 8192, &tmA, fb, tl.m0 + 64, krow);
#pragma unroll
                        for (int i = 0; i < BN / 64; ++i) sm100::tma_load_2d(sb + i * 8192, &tmB0, fb, tl.n0 + 64 * i, krow);
                    } else {
                        sm100::tma_load_2d(sa, &tmA, fb, k0, tl.m0);
                        if constexpr (OP == Op::FC1_SWIGLU) {
                            // gate columns [n0, n0+BN/2) then up columns, each as 64-wide MN chunks
#pragma unroll
                            for (int i = 0; i < BN / 128; ++i) {
                                sm100::tma_load_3d(sb + i * 8192, &tmB0, fb, tl.n0 + 64 * i, k0, tl.e);
                                sm100::tma_load_3d(sb + (BN / 128 + i) * 8192, &tmB1, fb, tl.n0 + 64 * i, k0, tl.e);
                            }
                        } else if constexpr (OP == Op::FC2) {
#pragma unroll
                            for (int i = 0; i < BN / 64; ++i) sm100::tma_load_3d(sb + i * 8192, &tmB0, fb, tl.n0 + 64 * i, k0, tl.e);
                        } else if constexpr (OP == Op::DGRAD_DSWIGLU) {
                            sm100::tma_load_3d(sb, &tmB0, fb, k0, tl.n0, tl.e);
                        } else {   // DGRAD_FC1: K in [0, F) from W_gate, [F, 2F) from W_up
                            if (k0 < args.k_split) sm100::tma_load_3d(sb, &tmB0, fb, k0, tl.n0, tl.e);
                            else sm100::tma_load_3d(sb, &tmB1, fb, k0 - args.k_split, tl.n0, tl.e);
                        }
                    }
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                int st = stage;
                uint32_t ph = phase;
                for (int i = 0; i < S && i < issued; ++i) {
                    if (--st < 0) { st = S - 1; ph ^= 1u; }
                    int dummy = 0;
                    sm100::mbar_wait(&full_bar[st], ph, &dummy, nullptr, 10000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        constexpr uint32_t IDESC = TR::mx ? sm100::idesc_mxf8(BM, BN) : sm100::idesc_bf16(BM, BN, TR::a_mn, TR::b_mn);
        // stage-0 operand descriptors; a K step of 16 (bf16) or 32 (E4M3) elements moves the
        // start address by 32 bytes (K-major) or one 2 KB group of 16 rows (MN-major)
        const uint64_t a_desc0 = TR::a_mn ? sm100::sdesc_sw128(smem_base, 8192, 1024) : sm100::sdesc_sw128(smem_base, 16, 1024);
        const uint64_t b_desc0 = TR::b_mn ? sm100::sdesc_sw128(smem_base + C::A_BYTES, 8192, 1024)
                                          : sm100::sdesc_sw128(smem_base + C::A_BYTES, 16, 1024);
        constexpr uint64_t A_KSTEP = TR::a_mn ? (2048 >> 4) : (32 >> 4);
        constexpr uint64_t B_KSTEP = TR::b_mn ? (2048 >> 4) : (32 >> 4);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        bool issued_any = false;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const Tile tl = decode_tile<OP, BN>(t, args, s_off, s_start);
            if (tl.kb == 0) continue;   // empty K range: the epilogue writes zeros
            const bool got_acc = sm100::mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort, args.err, wait_ns);
            if (__any_sync(0xFFFFFFFFu, !got_acc)) { ok = false; break; }
            sm100::tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < tl.kb; ++kb) {
                const bool got = sm100::mbar_wait(&full_bar[stage], phase, abort, args.err, wait_ns);
                if (__any_sync(0xFFFFFFFFu, !got)) { ok = false; break; }
                const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                const uint32_t sb = sa + C::A_BYTES;
                int kk_end = TR::BK / UMMA_K;   // K slices of 16 rows this stage contributes
                if constexpr (TR::k_grouped) {
                    // the group ends inside this stage: only the 16-row slices holding its rows
                    // are multiplied, and the rows of the last one past the group's end (they
                    // belong to the next group) are zeroed in every operand box
                    const int valid = tl.k_rows - kb * TR::BK;
                    if (valid < TR::BK) {
                        kk_end = (valid + UMMA_K - 1) / UMMA_K;
                        const int zrows = kk_end * UMMA_K - valid;
                        if (zrows > 0) {
                            uint8_t *pa = smem + stage * C::STAGE_BYTES;
                            const int nbox = 2 + BN / 64;
                            for (int i = lane; i < nbox * zrows * 8; i += 32) {
                                const int box = i / (zrows * 8);
                                const int rem = i - box * zrows * 8;
                                const int row = valid + rem / 8, c16 = rem % 8;
                                *reinterpret_cast<uint4 *>(pa + box * 8192 + row * 128 + c16 * 16) =
                                    make_uint4(0, 0, 0, 0);
                            }
                            sm100::fence_proxy_async_smem();
                        }
                        __syncwarp();
                    }
                }
                sm100::tc_fence_after();
                // descriptors of this stage computed by the whole warp (warp-uniform values);
                // one elected lane issues
                const uint64_t ad = a_desc0 + (uint64_t)stage * (C::STAGE_BYTES >> 4);
                const uint64_t bd = b_desc0 + (uint64_t)stage * (C::STAGE_BYTES >> 4);
                if constexpr (TR::mx) {
                    const uint32_t ssf = sb + C::B_BYTES;
                    const uint32_t tsf = tmem_base + C::SF_COL0 + stage * C::SF_COLS;
                    if (sm100::elect_one()) {
                        // scales of this stage: smem atoms -> TMEM slot of the stage, then 4 MMAs of
                        // K = 32 with scale ids 0..3 (the 4 bytes of each TMEM scale word)
                        sm100::tmem_cp_32x128b_x4(tsf, sm100::sdesc_plain(ssf));
#pragma unroll
                        for (int j = 0; j < BN / 128; ++j)
                            sm100::tmem_cp_32x128b_x4(tsf + 4 + 4 * j, sm100::sdesc_plain(ssf + 512 + 512 * j));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            sm100::mma_mxf8(d_tmem, ad + kk * A_KSTEP, bd + kk * B_KSTEP,
                                            IDESC | sm100::idesc_sf_ids(kk, kk), tsf, tsf + 4, (kb | kk) != 0 ? 1u : 0u);
                        sm100::mma_commit(&empty_bar[stage]);
                    }
                } else {
                    if (sm100::elect_one()) {
                        if (kk_end == TR::BK / UMMA_K) {
#pragma unroll
                            for (int kk = 0; kk < TR::BK / UMMA_K; ++kk)
                                sm100::mma_bf16(d_tmem, ad + kk * A_KSTEP, bd + kk * B_KSTEP, IDESC,
                                                (kb | kk) != 0 ? 1u : 0u);
                        } else {
                            for (int kk = 0; kk < kk_end; ++kk)
                                sm100::mma_bf16(d_tmem, ad + kk * A_KSTEP, bd + kk * B_KSTEP, IDESC,
                                                (kb | kk) != 0 ? 1u : 0u);
                        }
                        sm100::mma_commit(&empty_bar[stage]);
                    }
                }
                issued_any = true;
                __syncwarp();
                if (++stage == S) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (sm100::elect_one()) sm100::mma_commit(&tfull_bar[acc]);
            __syncwarp();
            if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
        }
        if (!ok && issued_any && sm100::elect_one()) {
            // drain: wait for the MMAs already issued before TMEM is released
            sm100::mma_commit(&drain_bar);
            int dummy = 0;
            sm100::mbar_wait(&drain_bar, 0, &dummy, nullptr, 10000000ull);
        }
        __syncwarp();
    } else {
        // ============================================================ epilogue
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int r = q * 32 + lane;       // accumulator row of this thread
        const int ew = warp - 2;           // epilogue warp
        const int sub = ew >> 2;           // which of the quarter's warps (eight epilogue warps)
        constexpr int NSUB = C::EPI / 4;
        // Output staging of this warp: two 2 KB slots of 32 rows x 64 bytes in the 64-byte
        // swizzle (16-byte chunk j of row i at chunk j ^ ((i / 2) % 4): conflict-free
        // 16-byte writes), each written back by one TMA store while the other fills.
        uint8_t *stg = smem + S * C::STAGE_BYTES + ew * C::SLOTS * 2048;
        const uint32_t stg_s = smem_base + S * C::STAGE_BYTES + ew * C::SLOTS * 2048;
        int slot = 0;
        auto slot_open = [&]() {
            if (lane == 0) sm100::bulk_wait_read<C::SLOTS - 1>();   // the store that last used this slot has read it
            __syncwarp();
        };
        auto slot_put = [&](int j, uint4 v) {
            *reinterpret_cast<uint4 *>(stg + slot * 2048 + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
        };
        auto slot_store = [&](const CUtensorMap *tm, int col, int64_t row0) {
            sm100::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                sm100::tma_store_2d(tm, stg_s + slot * 2048, col, (int)row0);
                sm100::bulk_commit();
            }
            slot = slot + 1 == C::SLOTS ? 0 : slot + 1;
        };
        auto stage_bf16x32 = [&](const float (&v)[32], const CUtensorMap *tm, int col, int64_t row0) {
            slot_open();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 pk;
                __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
                slot_put(j, pk);
            }
            slot_store(tm, col, row0);
        };
        auto stage_f32x32 = [&](const uint32_t (&d)[32], const CUtensorMap *tm, int col, int64_t row0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                slot_open();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    slot_put(j, make_uint4(d[16 * h + 4 * j], d[16 * h + 4 * j + 1], d[16 * h + 4 * j + 2],
                                           d[16 * h + 4 * j + 3]));
                slot_store(tm, col + 16 * h, row0);
            }
        };
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const Tile tl = decode_tile<OP, BN>(t, args, s_off, s_start);
            if constexpr (TR::k_grouped) {
                const int row = tl.m0 + r;
                const size_t eoff = (size_t)tl.e * (size_t)args.expert_stride;
                if (tl.kb == 0) {
                    // expert with no routes: its weight gradient is exactly zero
                    for (int c = 32 * sub; c < BN; c += 32 * NSUB) {
                        const int n = tl.n0 + c;
                        if (n >= args.N) break;
                        const bool second = OP == Op::WGRAD_GATEUP && n >= args.n_split;
                        const size_t off = eoff + (size_t)row * (second ? args.ld1 : args.ld0) +
                                           (second ? n - args.n_split : n);
                        uint4 *d4 = args.w_bf16 ? reinterpret_cast<uint4 *>((second ? args.out1 : args.out0) + off)
                                                : reinterpret_cast<uint4 *>((second ? args.out1_f32 : args.out_f32) + off);
                        const int nq = args.w_bf16 ? 4 : 8;   // 32 columns: 64 or 128 bytes
                        for (int q4 = 0; q4 < nq; ++q4) d4[q4] = make_uint4(0, 0, 0, 0);
                    }
                    continue;
                }
            }
            const bool got = sm100::mbar_wait(&tfull_bar[acc], acc_phase, abort, args.err, wait_ns);
            if (__any_sync(0xFFFFFFFFu, !got)) break;
            sm100::tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            // M-grouped: this warp's 32 rows go out through TMA when all of them belong to the
            // group (a store box never crosses into the next group's rows); else row by row
            const int64_t wrow0 = (int64_t)tl.m0 + q * 32;
            const bool whole = wrow0 + 32 <= tl.m_end && wrow0 + 32 <= args.rows_cap;

            if constexpr (TR::swiglu) {
                const int64_t row = tl.m0 + r;
                const bool valid = row < tl.m_end && row < args.rows_cap;
                float rw = 1.0f;
                if (args.route_w) {
                    const int src = valid ? args.src_of_row[row] : -1;
                    rw = src >= 0 ? args.route_w[src] : 0.0f;
                }
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    uint32_t g[32], u[32];
                    sm100::tmem_ld32(tacc + c, g);
                    sm100::tmem_ld32(tacc + BN / 2 + c, u);
                    sm100::tmem_ld_wait();
                    const int n = tl.n0 + c;
                    if (n < args.N && (whole || valid)) {
                        float hv[32];
                        if (args.clamp) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float gc = fminf(fmaxf(__uint_as_float(g[i]), args.gate_lo), args.gate_hi);
                                const float uc = fminf(fmaxf(__uint_as_float(u[i]), args.up_lo), args.up_hi);
                                hv[i] = silu_f(gc) * uc * rw;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                hv[i] = silu_f(__uint_as_float(g[i])) * __uint_as_float(u[i]) * rw;
                        }
                        if constexpr (OP == Op::FC1_MX) {
                            // h quantised along F: this thread's 32 columns are one MX block; two
                            // blocks (64 bytes of codes) fill a staging row
                            const int X = mx::scale_exp(mx::amax32(hv));
                            uint4 lo, hi;
                            mx::quantize32(hv, X, lo, hi);
                            if (whole) {
                                const int half = (c >> 5) & 1;
                                if (half == 0) slot_open();
                                slot_put(2 * half, lo);
                                slot_put(2 * half + 1, hi);
                                if (half == 1) slot_store(&tmC0, n - 32, wrow0);
                            } else {
                                uint4 *dq = reinterpret_cast<uint4 *>(args.out_q + row * args.ld0 + n);
                                dq[0] = lo;
                                dq[1] = hi;
                            }
                            args.out_sf[mx::tile_sf_offset(tl.mtile, args.N / 128, r, n / 32)] = (uint8_t)(X + 127);
                            if (args.out1) {   // bf16 stash of g | u for the straight-through backward
                                float gv[32], uv[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    gv[i] = __uint_as_float(g[i]);
                                    uv[i] = __uint_as_float(u[i]);
                                }
                                store_bf16x32(args.out1 + row * args.ld1 + n, gv);
                                store_bf16x32(args.out1 + row * args.ld1 + args.N + n, uv);
                            }
                        } else {
                            float gv[32], uv[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                gv[i] = __uint_as_float(g[i]);
                                uv[i] = __uint_as_float(u[i]);
                            }
                            if (whole) {
                                stage_bf16x32(hv, &tmC0, n, wrow0);
                                if (args.out1) {
                                    stage_bf16x32(gv, &tmC1, n, wrow0);
                                    stage_bf16x32(uv, &tmC1, args.N + n, wrow0);
                                }
                            } else {
                                store_bf16x32(args.out0 + row * args.ld0 + n, hv);
                                if (args.out1) {
                                    store_bf16x32(args.out1 + row * args.ld1 + n, gv);
                                    store_bf16x32(args.out1 + row * args.ld1 + args.N + n, uv);
                                }
                            }
                        }
                    }
                }
            } else if constexpr (OP == Op::DGRAD_DSWIGLU) {
                const int64_t row = tl.m0 + r;
                const bool valid = row < tl.m_end && row < args.rows_cap;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t d[32];
                    sm100::tmem_ld32(tacc + c, d);
                    sm100::tmem_ld_wait();
                    const int n = tl.n0 + c;
                    if (n < args.N && (whole || valid)) {
                        float gv[32], uv[32], dg[32], du[32];
                        load_bf16x32(args.aux + row * args.ld_aux + n, gv);
                        load_bf16x32(args.aux + row * args.ld_aux + args.N + n, uv);
                        if (args.clamp) {   // clamped inputs; zero derivative outside the bounds
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float dh = __uint_as_float(d[i]);
                                const float G = gv[i], U = uv[i];
                                const float gc = fminf(fmaxf(G, args.gate_lo), args.gate_hi);
                                const float uc = fminf(fmaxf(U, args.up_lo), args.up_hi);
                                const float s = sigmoid_fast(gc);
                                const bool gin = G >= args.gate_lo && G <= args.gate_hi;
                                const bool uin = U >= args.up_lo && U <= args.up_hi;
                                dg[i] = gin ? dh * uc * s * (1.0f + gc * (1.0f - s)) : 0.0f;
                                du[i] = uin ? dh * gc * s : 0.0f;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float dh = __uint_as_float(d[i]);
                                const float s = sigmoid_fast(gv[i]);
                                dg[i] = dh * uv[i] * s * (1.0f + gv[i] * (1.0f - s));
                                du[i] = dh * gv[i] * s;
                            }
                        }
                        if (whole) {
                            stage_bf16x32(dg, &tmC0, n, wrow0);
                            stage_bf16x32(du, &tmC0, args.N + n, wrow0);
                        } else {
                            store_bf16x32(args.out0 + row * args.ld0 + n, dg);
                            store_bf16x32(args.out0 + row * args.ld0 + args.N + n, du);
                        }
                    }
                }
            } else if constexpr (TR::k_grouped) {   // fp32 weight gradient of expert e
                // rows of the [E * M, N] view of the expert-stacked gradient
                const int64_t grow0 = (int64_t)tl.e * args.M + tl.m0 + q * 32;
#pragma unroll 1
                for (int c = 32 * sub; c < BN; c += 32 * NSUB) {
                    uint32_t d[32];
                    sm100::tmem_ld32(tacc + c, d);
                    sm100::tmem_ld_wait();
                    const int n = tl.n0 + c;
                    if (n < args.N) {
                        const bool second = OP == Op::WGRAD_GATEUP && n >= args.n_split;
                        if (args.w_bf16) {
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(d[i]);
                            stage_bf16x32(v, second ? &tmC1 : &tmC0, second ? n - args.n_split : n, grow0);
                        } else {
                            stage_f32x32(d, second ? &tmC1 : &tmC0, second ? n - args.n_split : n, grow0);
                        }
                    }
                }
            } else {   // FC2, FC2_MX (y_perm: bf16 rows) and DGRAD_FC1 (dx_perm: fp32 rows)
                static_assert(OP == Op::FC2 || OP == Op::FC2_MX || OP == Op::DGRAD_FC1, "unhandled op");
                const int64_t row = tl.m0 + r;
                const bool valid = row < tl.m_end && row < args.rows_cap;
                float rw = 1.0f;
                if (args.route_w) {
                    const int src = valid ? args.src_of_row[row] : -1;
                    rw = src >= 0 ? args.route_w[src] : 0.0f;
                }
#pragma unroll 1
                for (int c = 32 * sub; c < BN; c += 32 * NSUB) {
                    uint32_t d[32];
                    sm100::tmem_ld32(tacc + c, d);
                    sm100::tmem_ld_wait();
                    if (args.route_w) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) d[i] = __float_as_uint(__uint_as_float(d[i]) * rw);
                    }
                    const int n = tl.n0 + c;
                    if (n < args.N) {
                        if constexpr (OP == Op::FC2 || OP == Op::FC2_MX) {
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(d[i]);
                            if (whole) stage_bf16x32(v, &tmC0, n, wrow0);
                            else if (valid) store_bf16x32(args.out0 + row * args.ld0 + n, v);
                        } else {
                            if (whole) stage_f32x32(d, &tmC0, n, wrow0);
                            else if (valid) store_f32x32(args.out_f32 + row * args.ld0 + n, d);
                        }
                    }
                }
            }
            sm100::tc_fence_before();
            sm100::mbar_arrive(&tempty_bar[acc]);
            if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
        }
        // every TMA store of this warp has finished before the CTA can exit
        if (lane == 0) sm100::bulk_wait_all();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    sm100::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        sm100::tc_fence_after();
        sm100::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace gg
}  // namespace moe
