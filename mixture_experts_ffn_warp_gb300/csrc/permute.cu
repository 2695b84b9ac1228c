// permute.cu -- A2: sync-free permutation of tokens into expert-contiguous rows.
//
// Two launches on one stream, no host round trip:
//   1. count:   each 2048-route chunk counts its routes per expert and gives
//               every route its stable rank among the chunk's routes to the
//               same expert (bit-sliced warp ballots + per-warp running counts); the last
//               block to finish turns the chunk counts into group sizes,
//               (aligned) group offsets and each chunk's first row per expert.  Up to
//               32768 routes one thread-block cluster does the same with the counts
//               exchanged in distributed shared memory, and writes the final rows;
//   2. scatter: one warp per token writes dst_of_route / src_of_row (unless the
//               cluster pass wrote them) and copies the token's row once from HBM
//               into its k destinations with 16-byte loads and stores.
// (One-GPU counterpart of the expert-major dispatch layout with device-side
// group sizes: "[JAX] Expert Parallelism: JAX primitives + VJPs", commit log;
// "MoE training optimization": problem sizes supplied from device buffers.)
#include "carveout.cuh"
#include "common.cuh"

namespace moe {
namespace {

constexpr int kScatterWarps = 8;
// Largest [chunks][E] count matrix the final scan stages in shared memory: 39 KB, within the
// 48 KB a block may use without opt-in next to the counting kernel's static arrays (8.7 KB).
constexpr int64_t kScanSmemInts = 9984;

// Group sizes, aligned offsets, each chunk's first row per expert (in place of
// the chunk counts) and, if mtile_start != nullptr, each group's first 128-row
// M-tile: one block (>= 256 threads), each thread owning up to 4 consecutive experts.
// s_mat (nullable): shared memory for the whole [chunks][E] count matrix, which is then
// read from and written back to global memory once, coalesced, instead of one column
// per thread.
__device__ void scan_groups(int32_t *chunk_counts, int64_t chunks, int E, int align, int32_t *group_sizes,
                            int32_t *group_offsets, int32_t *mtile_start, int32_t *s_mat) {
    __shared__ int32_t s_wsum[32], s_wtile[32];
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n = chunks * E;
    if (s_mat) {
        for (int64_t i = tid; i < n; i += nt) s_mat[i] = __ldcg(chunk_counts + i);
        __syncthreads();
    }
    const int per = (E + nt - 1) / nt;
    const int e0 = tid * per;
    int tot[4] = {0, 0, 0, 0};
    int pad_sum = 0, tile_sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = e0 + i;
        if (i < per && e < E) {
            if (s_mat) {
                for (int64_t c = 0; c < chunks; ++c) tot[i] += s_mat[c * E + e];
            } else {
                for (int64_t c0 = 0; c0 < chunks; c0 += 8) {   // 8 loads in flight
                    int v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v[u] = c0 + u < chunks ? __ldcg(chunk_counts + (c0 + u) * E + e) : 0;
#pragma unroll
                    for (int u = 0; u < 8; ++u) tot[i] += v[u];
                }
            }
            const int padded = (tot[i] + align - 1) / align * align;
            pad_sum += padded;
            tile_sum += (padded + 127) / 128;
        }
    }
    int incl = pad_sum, tincl = tile_sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off), ot = __shfl_up_sync(0xFFFFFFFFu, tincl, off);
        if (lane >= off) { incl += o; tincl += ot; }
    }
    if (lane == 31) { s_wsum[warp] = incl; s_wtile[warp] = tincl; }
    __syncthreads();
    if (warp == 0) {
        const int nw = (nt + 31) / 32;
        int v = lane < nw ? s_wsum[lane] : 0, vt = lane < nw ? s_wtile[lane] : 0;
        int vi = v, vti = vt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, vi, off), ot = __shfl_up_sync(0xFFFFFFFFu, vti, off);
            if (lane >= off) { vi += o; vti += ot; }
        }
        if (lane < nw) { s_wsum[lane] = vi - v; s_wtile[lane] = vti - vt; }
    }
    __syncthreads();
    int run = incl - pad_sum + s_wsum[warp];
    int trun = tincl - tile_sum + s_wtile[warp];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = e0 + i;
        if (i < per && e < E) {
            group_sizes[e] = tot[i];
            group_offsets[e] = run;
            if (mtile_start) mtile_start[e] = trun;
            int r2 = run;
            if (s_mat) {
                for (int64_t c = 0; c < chunks; ++c) {
                    const int v = s_mat[c * E + e];
                    s_mat[c * E + e] = r2;
                    r2 += v;
                }
            } else {
                for (int64_t c0 = 0; c0 < chunks; c0 += 8) {   // 8 loads in flight, then the stores
                    int v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v[u] = c0 + u < chunks ? __ldcg(chunk_counts + (c0 + u) * E + e) : 0;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (c0 + u < chunks) chunk_counts[(c0 + u) * E + e] = r2;
                        r2 += v[u];
                    }
                }
            }
            const int padded = (tot[i] + align - 1) / align * align;
            run += padded;
            trun += (padded + 127) / 128;
            if (e == E - 1) {
                group_offsets[E] = run;
                if (mtile_start) mtile_start[E] = trun;
            }
        }
    }
    if (s_mat) {
        __syncthreads();
        for (int64_t i = tid; i < n; i += nt) chunk_counts[i] = s_mat[i];
    }
}

// Column split of a [C][E] int matrix in shared memory over the block (E <= blockDim.x):
// thread (e = tid % E, j = tid / E) with j < J = min(blockDim.x / E, 32) takes rows
// [c0, c1) of column e, so the lanes of a warp read consecutive columns (no bank
// conflicts); the J partial sums of a column meet in s_part.  Returns the column's
// exclusive prefix before row c0 and its total.
struct ColSplit {
    int e, j, c0, c1, pre, tot;
    bool act;
};

__device__ ColSplit column_split(const int32_t *s_mat, int C, int E, int32_t *s_part) {
    ColSplit r;
    const int nt = blockDim.x, tid = threadIdx.x;
    const int J = nt / E < 32 ? nt / E : 32;
    r.e = tid % E;
    r.j = tid / E;
    r.act = r.j < J;
    const int per = (C + J - 1) / J;
    r.c0 = r.j * per < C ? r.j * per : C;
    r.c1 = r.c0 + per < C ? r.c0 + per : C;
    int seg = 0;
    if (r.act)
        for (int c = r.c0; c < r.c1; ++c) seg += s_mat[c * E + r.e];
    if (r.act) s_part[r.j * E + r.e] = seg;
    __syncthreads();
    r.pre = 0;
    r.tot = 0;
    if (r.act) {
        for (int q = 0; q < J; ++q) {
            const int v = s_part[q * E + r.e];
            if (q < r.j) r.pre += v;
            r.tot += v;
        }
    }
    __syncthreads();   // s_part may be reused
    return r;
}

// scan_groups for a count matrix staged in shared memory, with E <= blockDim.x (column
// split as above; the exclusive scan over the experts is a block scan).  Same results as
// scan_groups.
__device__ void scan_groups_smem(int32_t *chunk_counts, int C, int E, int align, int32_t *group_sizes,
                                 int32_t *group_offsets, int32_t *mtile_start, int32_t *s_mat) {
    __shared__ int32_t s_wsum[32], s_wtile[32], s_first[1025], s_part[1024];
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = C * E;
    for (int base = 0; base < n; base += 8 * nt) {   // 8 loads in flight per thread, then the stores
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * nt + tid;
            v[u] = i < n ? __ldcg(chunk_counts + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * nt + tid;
            if (i < n) s_mat[i] = v[u];
        }
    }
    __syncthreads();
    const ColSplit cs = column_split(s_mat, C, E, s_part);
    // exclusive scan over the experts: thread e (j == 0) holds expert e's padded size
    const bool head = cs.act && cs.j == 0;
    const int padded = head ? (cs.tot + align - 1) / align * align : 0;
    const int tiles = head ? (padded + 127) / 128 : 0;
    int pi = padded, ti = tiles;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, pi, off), ot = __shfl_up_sync(0xFFFFFFFFu, ti, off);
        if (lane >= off) { pi += o; ti += ot; }
    }
    if (lane == 31) { s_wsum[warp] = pi; s_wtile[warp] = ti; }
    __syncthreads();
    if (warp == 0) {
        const int nw = (nt + 31) / 32;
        const int v = lane < nw ? s_wsum[lane] : 0, vt = lane < nw ? s_wtile[lane] : 0;
        int vi = v, vti = vt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, vi, off), ot = __shfl_up_sync(0xFFFFFFFFu, vti, off);
            if (lane >= off) { vi += o; vti += ot; }
        }
        if (lane < nw) { s_wsum[lane] = vi - v; s_wtile[lane] = vti - vt; }
    }
    __syncthreads();
    if (head) {
        const int e = cs.e;
        const int off0 = pi - padded + s_wsum[warp], t0 = ti - tiles + s_wtile[warp];
        group_sizes[e] = cs.tot;
        group_offsets[e] = off0;
        if (mtile_start) mtile_start[e] = t0;
        s_first[e] = off0;
        if (e == E - 1) {
            group_offsets[E] = off0 + padded;
            if (mtile_start) mtile_start[E] = t0 + tiles;
        }
    }
    __syncthreads();
    // each chunk's first row per expert, in place of the counts
    if (cs.act) {
        int run = s_first[cs.e] + cs.pre;
        for (int c = cs.c0; c < cs.c1; ++c) {
            const int v = s_mat[c * E + cs.e];
            s_mat[c * E + cs.e] = run;
            run += v;
        }
    }
    __syncthreads();
    for (int i = tid; i < n; i += nt) chunk_counts[i] = s_mat[i];
}

// Stable ranks of one warp's 32 * kPermSteps consecutive routes from w0: ev[step] = the
// expert of route w0 + 32 step + lane (-1: dropped, invalid or past R), rk[step] = its rank
// among this warp's earlier routes to the same expert, counted into cnt[E] (the warp's
// running counts, zero on entry).  Lanes holding the same id are found by AND-ing the
// ballots of each bit of e + 1.
__device__ __forceinline__ void rank_warp_routes(const int32_t *__restrict__ topk_idx, int64_t R, int64_t w0, int E,
                                                 int32_t *cnt, int (&ev)[kPermSteps], int (&rk)[kPermSteps],
                                                 uint32_t *err) {
    const int lane = threadIdx.x & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int id_bits = 32 - __clz(E);
    // all of this warp's route ids first (independent loads), then the ranks from registers
#pragma unroll
    for (int step = 0; step < kPermSteps; ++step) {
        const int64_t r = w0 + step * 32 + lane;
        ev[step] = r < R ? __ldg(topk_idx + r) : -1;
    }
#pragma unroll
    for (int step = 0; step < kPermSteps; ++step) {
        int e = ev[step];
        if (e < -1 || e >= E) {
            raise_device_error(err, MOE_DEVERR_BAD_EXPERT_ID);
            e = -1;
        }
        ev[step] = e;
        unsigned peers = 0xFFFFFFFFu;
        const unsigned v = (unsigned)(e + 1);   // in [0, E]
        for (int b = 0; b < id_bits; ++b) {
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, (v >> b) & 1u);
            peers &= ((v >> b) & 1u) ? bal : ~bal;
        }
        int rank = -1;
        if (e >= 0) rank = cnt[e] + __popc(peers & lt_mask);
        __syncwarp();
        if (e >= 0 && (peers & lt_mask) == 0) cnt[e] += __popc(peers);   // leader of the peer group
        __syncwarp();
        rk[step] = rank;
    }
}

// Counting pass: per 2048-route chunk, stable ranks (warp ballots + per-warp running
// counts) and per-expert chunk counts; the last block to finish runs scan_groups,
// so that offsets are ready when the kernel ends (no separate scan launch).
__global__ void __launch_bounds__(kPermWarps * 32)
permute_count_kernel(const int32_t *__restrict__ topk_idx, int64_t R, int E, int align,
                     int32_t *__restrict__ local_rank, int32_t *__restrict__ chunk_counts,
                     int32_t *__restrict__ group_sizes, int32_t *__restrict__ group_offsets,
                     int32_t *__restrict__ mtile_start, int scan_in_smem, uint32_t *done, uint32_t *err) {
    pdl_wait();
    pdl_trigger();   // the scatter's CTAs may start loading token rows on the idle SMs
    // [kPermWarps][E] running counts; in the last block, the [chunks][E] count matrix when
    // scan_in_smem (the launch then sizes this array for it)
    extern __shared__ int32_t s_cnt[];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();

    const int64_t chunk0 = (int64_t)blockIdx.x * kPermChunk;
    const int64_t w0 = chunk0 + (int64_t)warp * 32 * kPermSteps;
    int ev[kPermSteps], rk[kPermSteps];
    rank_warp_routes(topk_idx, R, w0, E, s_cnt + warp * E, ev, rk, err);
    __syncthreads();
    // exclusive scan over warps per expert -> rank offset of each warp; chunk totals
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < kPermWarps; ++w) {
            int c = s_cnt[w * E + e];
            s_cnt[w * E + e] = run;
            run += c;
        }
        chunk_counts[(int64_t)blockIdx.x * E + e] = run;
    }
    __syncthreads();
    // add the warp offsets to this chunk's ranks
#pragma unroll
    for (int step = 0; step < kPermSteps; ++step) {
        const int64_t r = w0 + step * 32 + lane;
        if (r < R) local_rank[r] = rk[step] >= 0 ? rk[step] + s_cnt[warp * E + ev[step]] : -1;
    }
    // the last block to finish turns all chunk counts into offsets
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (scan_in_smem && E <= (int)blockDim.x)
        scan_groups_smem(chunk_counts, gridDim.x, E, align, group_sizes, group_offsets, mtile_start, s_cnt);
    else
        scan_groups(chunk_counts, gridDim.x, E, align, group_sizes, group_offsets, mtile_start,
                    scan_in_smem ? s_cnt : nullptr);
    if (threadIdx.x == 0) *done = 0u;
}

// The scan alone, for an empty problem (no counting blocks).
__global__ void __launch_bounds__(256)
permute_scan_kernel(int32_t *__restrict__ chunk_counts, int64_t chunks, int E, int align,
                    int32_t *__restrict__ group_sizes, int32_t *__restrict__ group_offsets,
                    int32_t *__restrict__ mtile_start) {
    pdl_wait();
    scan_groups(chunk_counts, chunks, E, align, group_sizes, group_offsets, mtile_start, nullptr);
}

// ---- counting pass in one thread-block cluster (R <= kClusterRoutes) ----
// The CTAs of one cluster exchange their per-expert counts through distributed shared
// memory instead of global memory, a fence and a finished-blocks counter, and every CTA
// writes the final rows of its own routes: the scatter then only reads them.  Measured on
// GB300 (route + permute, L2 flushed): fine_grained 33.8 -> 32.0 us, mixtral 44 -> 43 us,
// tiny 13.3 -> 11.3 us; with 32 warps a CTA (65536 routes) the eight SMs rank more slowly
// than the chunked pass's 32 CTAs (DeepSeek-V3 shape, quantising: 142 -> 146 us), hence
// the limit of 16 warps.
constexpr int kClusterCtas = 8;                                          // portable cluster size
constexpr int kClusterMaxWarps = 16;
constexpr int64_t kClusterRoutes = (int64_t)kClusterCtas * kClusterMaxWarps * 32 * kPermSteps;   // 32768

__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() {   // release: this CTA's shared writes / reads are done
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {     // acquire: the other CTAs' writes are visible
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Load of an int in CTA `rank`'s shared memory, at the address of `p` in this CTA's.
__device__ __forceinline__ int ld_cluster_s32(const int32_t *p, uint32_t rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t ra;
    int v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

// CTA c of the cluster owns routes [c P, (c + 1) P), P = 32 kPermSteps warps (blockDim.x >= 256).
// Dynamic shared memory: [warps][E] per-warp counts, then [E] this CTA's totals and [E] its first
// row per expert.  dst_of_route gets the final rows (-1: dropped), src_of_row their routes.
__global__ void __launch_bounds__(kClusterMaxWarps * 32)
permute_count_cluster_kernel(const int32_t *__restrict__ topk_idx, int64_t R, int E, int align, int64_t rows_cap,
                             int32_t *__restrict__ dst_of_route, int32_t *__restrict__ src_of_row,
                             int32_t *__restrict__ group_sizes, int32_t *__restrict__ group_offsets,
                             int32_t *__restrict__ mtile_start, uint32_t *err) {
    pdl_wait();
    pdl_trigger();   // the scatter's CTAs may start loading token rows on the idle SMs
    extern __shared__ int32_t s_dyn[];
    __shared__ int32_t s_wsum[32], s_wtile[32];
    const int nt = blockDim.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, W = nt >> 5;
    const uint32_t me = cta_rank_in_cluster(), C = gridDim.x;
    int32_t *s_cnt = s_dyn, *s_tot = s_dyn + W * E, *s_first = s_tot + E;
    for (int i = tid; i < W * E; i += nt) s_cnt[i] = 0;
    __syncthreads();

    const int64_t w0 = (int64_t)me * W * 32 * kPermSteps + (int64_t)warp * 32 * kPermSteps;
    int ev[kPermSteps], rk[kPermSteps];
    rank_warp_routes(topk_idx, R, w0, E, s_cnt + warp * E, ev, rk, err);
    __syncthreads();
    // exclusive scan over warps per expert -> rank offset of each warp; this CTA's totals
    for (int e = tid; e < E; e += nt) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            const int c = s_cnt[w * E + e];
            s_cnt[w * E + e] = run;
            run += c;
        }
        s_tot[e] = run;
    }
    cluster_arrive();
    cluster_wait();   // every CTA's totals are visible

    // per expert (up to 4 consecutive ones a thread): routes in earlier CTAs and in all
    const int per = (E + nt - 1) / nt;
    const int e0 = tid * per;
    int pre[4] = {0, 0, 0, 0}, tot[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = e0 + i;
        if (i < per && e < E) {
            int v[kClusterCtas];
#pragma unroll
            for (int c = 0; c < kClusterCtas; ++c) v[c] = c < (int)C ? ld_cluster_s32(s_tot + e, c) : 0;
#pragma unroll
            for (int c = 0; c < kClusterCtas; ++c) {
                if (c < (int)me) pre[i] += v[c];
                tot[i] += v[c];
            }
        }
    }
    cluster_arrive();   // done reading the other CTAs' totals (they wait for this before exiting)
    int pad_sum = 0, tile_sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i < per && e0 + i < E) {
            const int padded = (tot[i] + align - 1) / align * align;
            pad_sum += padded;
            tile_sum += (padded + 127) / 128;
        }
    }
    // exclusive scan of the padded sizes (and 128-row tile counts) over the experts
    int incl = pad_sum, tincl = tile_sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off), ot = __shfl_up_sync(0xFFFFFFFFu, tincl, off);
        if (lane >= off) { incl += o; tincl += ot; }
    }
    if (lane == 31) { s_wsum[warp] = incl; s_wtile[warp] = tincl; }
    __syncthreads();
    if (warp == 0) {
        const int v = lane < W ? s_wsum[lane] : 0, vt = lane < W ? s_wtile[lane] : 0;
        int vi = v, vti = vt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, vi, off), ot = __shfl_up_sync(0xFFFFFFFFu, vti, off);
            if (lane >= off) { vi += o; vti += ot; }
        }
        if (lane < W) { s_wsum[lane] = vi - v; s_wtile[lane] = vti - vt; }
    }
    __syncthreads();
    int run = incl - pad_sum + s_wsum[warp], trun = tincl - tile_sum + s_wtile[warp];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = e0 + i;
        if (i < per && e < E) {
            s_first[e] = run + pre[i];
            if (me == 0) {
                group_sizes[e] = tot[i];
                group_offsets[e] = run;
                if (mtile_start) mtile_start[e] = trun;
            }
            const int padded = (tot[i] + align - 1) / align * align;
            run += padded;
            trun += (padded + 127) / 128;
            if (me == 0 && e == E - 1) {
                group_offsets[E] = run;
                if (mtile_start) mtile_start[E] = trun;
            }
        }
    }
    __syncthreads();
    // final rows of this CTA's routes
#pragma unroll
    for (int step = 0; step < kPermSteps; ++step) {
        const int64_t r = w0 + step * 32 + lane;
        if (r < R) {
            int dst = -1;
            const int e = ev[step];
            if (e >= 0) {
                const int64_t row = (int64_t)s_first[e] + s_cnt[warp * E + e] + rk[step];
                if (row < rows_cap) {
                    dst = (int)row;
                    src_of_row[row] = (int32_t)r;
                } else {
                    raise_device_error(err, MOE_DEVERR_CAPACITY);
                }
            }
            dst_of_route[r] = dst;
        }
    }
    cluster_wait();   // no CTA leaves while another may still read its totals
}

// Warps per CTA of the cluster counting pass for R routes, 0 when R does not fit it
// (dyn_smem_max: the dynamic shared memory a CTA may take).
int cluster_count_warps(int64_t R, int E, size_t dyn_smem_max) {
    if (R <= 0) return 0;
    const int64_t ctas = (R + kPermChunk - 1) / kPermChunk < kClusterCtas ? (R + kPermChunk - 1) / kPermChunk
                                                                            : kClusterCtas;
    int64_t w = (R + ctas * 32 * kPermSteps - 1) / (ctas * 32 * kPermSteps);
    if (w < kPermWarps) w = kPermWarps;
    if (w > kClusterMaxWarps || R > kClusterRoutes) return 0;
    if ((size_t)(w * E + 2 * E) * sizeof(int32_t) > dyn_smem_max) return 0;
    return (int)w;
}

// Counting pass with the scan in its last block (or the scan alone for R = 0).  When the
// routes fit one cluster (cluster_count_warps > 0) the cluster pass runs instead, writes the
// final dst_of_route and src_of_row, and *final_rows is set: the scatter then takes the rows
// as they are (chunk_first = nullptr).  Otherwise dst_of_route holds chunk-local ranks.
moe_status_t count_and_scan(const int32_t *topk_idx, int64_t R, int E, int align, int64_t rows_cap,
                            int32_t *dst_of_route, int32_t *src_of_row, int32_t *counts, int32_t *group_sizes,
                            int32_t *group_offsets, int32_t *mtile, uint32_t *done, uint32_t *err, cudaStream_t s,
                            bool *final_rows) {
    int32_t *local_rank = dst_of_route;
    const int64_t chunks = perm_chunks(R);
    *final_rows = false;
    // The cluster pass takes all the shared memory a CTA may have, so that no scatter CTA
    // (launched early, loading its token rows) shares an SM with it: measured on GB300, the
    // counting CTAs' shared-memory and global accesses otherwise queue behind those loads.
    // Where the cluster cannot be launched (its attribute refused, or no eight whole SMs of one
    // GPC available to this context) the chunked pass below runs instead.
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    const size_t dyn = optin > 1024 ? (size_t)optin - 1024 : 0;   // (static arrays: 256 bytes)
    const int w = cluster_count_warps(R, E, dyn);
    if (w > 0) {
        if (cudaFuncSetAttribute(permute_count_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dyn) != cudaSuccess) {
            (void)cudaGetLastError();   // refused: not this call's error, the chunked pass runs
            goto chunked;
        }
        const int ctas = (int)(chunks < kClusterCtas ? chunks : kClusterCtas);
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)ctas);
        cfg.blockDim = dim3((unsigned)(w * 32));
        cfg.dynamicSmemBytes = dyn;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)ctas;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (cudaLaunchKernelEx(&cfg, permute_count_cluster_kernel, topk_idx, R, E, align, rows_cap, dst_of_route,
                               src_of_row, group_sizes, group_offsets, mtile, err) == cudaSuccess) {
            *final_rows = true;
            return launch_status();
        }
        (void)cudaGetLastError();   // refused: not this call's error, the chunked pass runs
    }
chunked:
    if (chunks > 0) {
        // the final scan stages the count matrix in shared memory when it fits
        const int64_t mat = chunks * E;
        const int scan_in_smem = mat <= kScanSmemInts ? 1 : 0;
        const int64_t smem_ints = scan_in_smem && mat > (int64_t)kPermWarps * E ? mat : (int64_t)kPermWarps * E;
        launch_k(permute_count_kernel, dim3((unsigned)chunks), dim3(kPermWarps * 32),
                 (size_t)smem_ints * sizeof(int32_t), s, topk_idx, R, E, align, local_rank, counts, group_sizes,
                 group_offsets, mtile, scan_in_smem, done, err);
    } else {
        launch_k(permute_scan_kernel, dim3(1), dim3(256), 0, s, counts, 0, E, align, group_sizes, group_offsets,
                 mtile);
    }
    return launch_status();
}

// One warp per token: maps, then the row copied once into its k rows (KMAX >= k).  The
// kernel runs after the counting pass, which triggers it early: the token row's first
// 32 * PRE 16-byte vectors are loaded before the wait (x was complete before the counting
// pass passed its own wait; the loads go to the L2, the point of coherence, past the SM's L1),
// the maps after it.  PRE = 8 (4 KB rows: H <= 2048), 16 for wider rows.  Blocks from
// token_blocks on (one per expert, aligned groups only) fill expert e's padding rows instead:
// src_of_row = -1 and zero data.
template <int KMAX, int PRE>
__global__ void __launch_bounds__(kScatterWarps * 32)
permute_scatter_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                       int64_t T, int k, int E, int row_vecs,
                       const int32_t *__restrict__ chunk_first, int32_t *__restrict__ dst_of_route,
                       int32_t *__restrict__ src_of_row, uint4 *__restrict__ x_perm,
                       int64_t rows_cap, const int32_t *__restrict__ group_sizes,
                       const int32_t *__restrict__ group_offsets, int64_t token_blocks, uint32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kScatterWarps + (threadIdx.x >> 5);
    const uint4 *src = x + (t < T ? t : 0) * row_vecs;
    uint4 pre[PRE];
    if (t < T) {
#pragma unroll
        for (int u = 0; u < PRE; ++u)
            if (lane + 32 * u < row_vecs) pre[u] = __ldcg(src + lane + 32 * u);   // from the L2, not L1
    }
    pdl_wait();
    if ((int64_t)blockIdx.x >= token_blocks) {   // an expert's padding rows
        const int e = (int)(blockIdx.x - token_blocks);
        const int64_t first = (int64_t)group_offsets[e] + group_sizes[e];
        const int64_t last = group_offsets[e + 1] < rows_cap ? group_offsets[e + 1] : rows_cap;
        for (int64_t row = first; row < last; ++row) {
            if (threadIdx.x == 0) src_of_row[row] = -1;
            for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) x_perm[row * row_vecs + v] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    if (t >= T) return;
    int my_dst = -1;
    if (lane < k) {
        const int64_t r = t * k + lane;
        if (!chunk_first) {
            my_dst = dst_of_route[r];         // final row written by the cluster count pass
        } else {
            const int rank = dst_of_route[r];     // local rank written by the count pass
            if (rank >= 0) {
                const int e = topk_idx[r];
                const int64_t row = (int64_t)chunk_first[(r / kPermChunk) * E + e] + rank;
                if (row < rows_cap) {
                    my_dst = (int)row;
                    src_of_row[row] = (int32_t)r;
                } else {
                    raise_device_error(err, MOE_DEVERR_CAPACITY);
                }
            }
            dst_of_route[r] = my_dst;
        }
    }
    int dst[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dst[j] = j < k ? __shfl_sync(0xFFFFFFFFu, my_dst, j) : -1;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j < k && dst[j] >= 0) {
            uint4 *d = x_perm + (int64_t)dst[j] * row_vecs;
#pragma unroll
            for (int u = 0; u < PRE; ++u)
                if (lane + 32 * u < row_vecs) d[lane + 32 * u] = pre[u];
        }
    }
    constexpr int U = 4;   // 16-byte vectors in flight per lane
    for (int v0 = lane + 32 * PRE; v0 < row_vecs; v0 += 32 * U) {
        uint4 val[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + 32 * u < row_vecs) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < k && dst[j] >= 0) {
                uint4 *d = x_perm + (int64_t)dst[j] * row_vecs;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (v0 + 32 * u < row_vecs) d[v0 + 32 * u] = val[u];
            }
        }
    }
}

// The scatter of T tokens, plus one block per expert filling its padding rows when `pad`.
void launch_scatter(cudaStream_t s, const uint4 *x, const int32_t *topk_idx, int64_t T, int k, int E, int row_vecs,
                    const int32_t *chunk_first, int32_t *dst_of_route, int32_t *src_of_row, uint4 *x_perm,
                    int64_t rows_cap, const int32_t *group_sizes, const int32_t *group_offsets, bool pad,
                    uint32_t *err) {
    const int64_t tb = (T + kScatterWarps - 1) / kScatterWarps;
    const unsigned blocks = (unsigned)(tb + (pad ? E : 0));
#define MOE_SCATTER(KM)                                                                                        \
    (prefer_max_smem_carveout<permute_scatter_kernel<KM, 16>>(),                                               \
     prefer_max_smem_carveout<permute_scatter_kernel<KM, 8>>(),                                                \
     row_vecs > 256                                                                                            \
         ? launch_k(permute_scatter_kernel<KM, 16>, dim3(blocks), dim3(kScatterWarps * 32), 0, s, x, topk_idx,  \
                    T, k, E, row_vecs, chunk_first, dst_of_route, src_of_row, x_perm, rows_cap, group_sizes,     \
                    group_offsets, tb, err)                                                                      \
         : launch_k(permute_scatter_kernel<KM, 8>, dim3(blocks), dim3(kScatterWarps * 32), 0, s, x, topk_idx,   \
                    T, k, E, row_vecs, chunk_first, dst_of_route, src_of_row, x_perm, rows_cap, group_sizes,     \
                    group_offsets, tb, err))
    if (k <= 1) MOE_SCATTER(1);
    else if (k <= 2) MOE_SCATTER(2);
    else if (k <= 4) MOE_SCATTER(4);
    else if (k <= 8) MOE_SCATTER(8);
    else if (k <= 16) MOE_SCATTER(16);
    else MOE_SCATTER(32);
#undef MOE_SCATTER
}


}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute(const moe_bf16_t *x, const int32_t *topk_idx, int64_t T, int H,
                                    int E, int k, int align, moe_bf16_t *x_perm, int64_t rows_cap,
                                    int32_t *dst_of_route, int32_t *src_of_row,
                                    int32_t *group_sizes, int32_t *group_offsets, void *ws,
                                    size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_permute");
    using namespace moe;
    if (T < 0 || H < 1 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || k < 1 || k > 32 || align < 1 || align > 1024 || H % 8 != 0)
        return MOE_ERR_UNSUPPORTED;
    if (!group_sizes || !group_offsets) return MOE_ERR_INVALID_ARG;
    const int64_t R = T * (int64_t)k;
    if (rows_cap < R + (int64_t)E * (align - 1)) return MOE_ERR_INVALID_ARG;
    if (rows_cap >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !topk_idx || !x_perm || !dst_of_route || !src_of_row))
        return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({x, x_perm})) return MOE_ERR_UNSUPPORTED;
    const size_t need = moe_workspace_bytes(T, E, k);
    if (!ws || ws_bytes < need || need == 0) return MOE_ERR_WORKSPACE;

    cudaStream_t s = (cudaStream_t)stream;
    uint32_t *err = ws_error_word(ws);
    int32_t *counts = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kWsHeaderBytes);
    const int64_t chunks = perm_chunks(R);
    bool final_rows = false;
    if (count_and_scan(topk_idx, R, E, align, rows_cap, dst_of_route, src_of_row, counts, group_sizes, group_offsets,
                       nullptr, ws_done_counter(ws), err, s, &final_rows) != MOE_OK)
        return MOE_ERR_CUDA;
    const int row_vecs = H / 8;
    if (T > 0) {   // (with no tokens there are no padding rows either)
        launch_scatter(s, reinterpret_cast<const uint4 *>(x), topk_idx, T, k, E, row_vecs,
                       final_rows ? nullptr : counts, dst_of_route,
                       src_of_row, reinterpret_cast<uint4 *>(x_perm), rows_cap, group_sizes, group_offsets,
                       align > 1, err);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// moe_permute_static_scratch: the same permutation for callers that cannot
// allocate device memory.  Its scratch (error word + per-chunk expert counts)
// is a fixed array in this library's device image instead of a workspace.
// ---------------------------------------------------------------------------

#include <mutex>

#include <cudaTypedefs.h>

namespace moe {
namespace {

// 256 KiB: a 256-byte header (error word at offset 0) and room for
// (256 KiB - 256) / 4 = 65472 per-chunk counts, i.e. chunks * E <= 65472
// with 2048 routes per chunk.  Every GPU that loads the library keeps this
// array resident until the process exits.
constexpr size_t kStaticScratchBytes = 256 * 1024;
static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 128;
std::mutex g_scratch_lock;
struct ScratchSlot {
    unsigned long long ctx_id;   // the context the address belongs to (0: none yet)
    void *addr;                  // device address of the array in that context
};
ScratchSlot g_scratch[kMaxScratchDevices];

// Id of the calling thread's current CUDA context (cuCtxGetId: unique within the process
// and never reused, so a context created after a cudaDeviceReset gets a new one); false
// when no context is current yet.  Driver entry points fetched once, under the lock.
bool current_context_id(unsigned long long *id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    if (!get_current || !get_id) {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r1) != cudaSuccess ||
            r1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) != cudaSuccess ||
            r2 != cudaDriverEntryPointSuccess)
            return false;
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(q);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// Device address of the array in the current device's current context.  The host-side
// name is only a stand-in and must not reach a kernel; the address is looked up with
// cudaGetSymbolAddress the first time a context calls, and again whenever the device's
// context changes (a cudaDeviceReset, or a caller that made another context current),
// since the module then lives elsewhere.
moe_status_t static_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxScratchDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_scratch_lock);
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    if (have_ctx && g_scratch[dev].addr && g_scratch[dev].ctx_id == ctx) {
        *out = g_scratch[dev].addr;
        return MOE_OK;
    }
    void *p = nullptr;   // the lookup also makes the device's primary context current if none was
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    if (!have_ctx && !current_context_id(&ctx)) return MOE_ERR_CUDA;
    g_scratch[dev].ctx_id = ctx;
    g_scratch[dev].addr = p;
    *out = p;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_static_scratch(const moe_bf16_t *x, const int32_t *topk_idx, int64_t T,
                                                   int H, int E, int k, int align, moe_bf16_t *x_perm,
                                                   int64_t rows_cap, int32_t *dst_of_route,
                                                   int32_t *src_of_row, int32_t *group_sizes,
                                                   int32_t *group_offsets, uint32_t *error_word,
                                                   moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_permute_static_scratch");
    using namespace moe;
    if (T < 0 || H < 1 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || k < 1 || k > 32 || align < 1 || align > 1024 || H % 8 != 0)
        return MOE_ERR_UNSUPPORTED;
    if (!group_sizes || !group_offsets) return MOE_ERR_INVALID_ARG;
    const int64_t R = T * (int64_t)k;
    if (rows_cap < R + (int64_t)E * (align - 1)) return MOE_ERR_INVALID_ARG;
    if (rows_cap >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !topk_idx || !x_perm || !dst_of_route || !src_of_row))
        return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({x, x_perm})) return MOE_ERR_UNSUPPORTED;
    const int64_t chunks = perm_chunks(R);
    if (kWsHeaderBytes + (size_t)chunks * (size_t)E * sizeof(int32_t) > kStaticScratchBytes)
        return MOE_ERR_UNSUPPORTED;   // problem needs more than the fixed scratch array

    void *scratch = nullptr;
    moe_status_t st = static_scratch(&scratch);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t *err = static_cast<uint32_t *>(scratch);
    int32_t *counts = reinterpret_cast<int32_t *>(static_cast<char *>(scratch) + kWsHeaderBytes);
    // the error word and the finished-blocks counter start at zero on every call; the
    // counts are fully rewritten
    if (cudaMemsetAsync(err, 0, 2 * sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    bool final_rows = false;
    if (count_and_scan(topk_idx, R, E, align, rows_cap, dst_of_route, src_of_row, counts, group_sizes, group_offsets,
                       nullptr, err + 1, err, s, &final_rows) != MOE_OK)
        return MOE_ERR_CUDA;
    const int row_vecs = H / 8;
    if (T > 0) {   // (with no tokens there are no padding rows either)
        launch_scatter(s, reinterpret_cast<const uint4 *>(x), topk_idx, T, k, E, row_vecs,
                       final_rows ? nullptr : counts, dst_of_route,
                       src_of_row, reinterpret_cast<uint4 *>(x_perm), rows_cap, group_sizes, group_offsets,
                       align > 1, err);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    if (error_word &&
        cudaMemcpyAsync(error_word, err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// moe_permute_mxfp8: the same permutation with the rows quantised to MXFP8 on
// the way (x is read once; each route gets E4M3 bytes and its scales in the
// MMA tile layout of its group).  ("[Draft][JAX] MoE block optimization",
// diagram: quantise before gather.)
// ---------------------------------------------------------------------------

#include "mx.cuh"

namespace moe {
namespace {

// KMAX >= k: the per-token route arrays stay in registers of that size.
template <int KMAX>
__global__ void __launch_bounds__(kScatterWarps * 32)
permute_scatter_mx_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx, int64_t T, int k,
                          int E, int H, const int32_t *__restrict__ chunk_first,
                          const int32_t *__restrict__ group_offsets, const int32_t *__restrict__ mtile_start,
                          int32_t *__restrict__ dst_of_route, int32_t *__restrict__ src_of_row,
                          uint8_t *__restrict__ x_q, uint8_t *__restrict__ x_sf, int64_t rows_cap, uint32_t *err) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kScatterWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_dst = -1, my_tile = 0, my_m = 0;
    if (lane < k) {
        const int64_t r = t * k + lane;
        if (!chunk_first) {
            my_dst = dst_of_route[r];         // final row written by the cluster count pass
            if (my_dst >= 0) {
                const int e = topk_idx[r];
                const int i = my_dst - group_offsets[e];
                my_tile = mtile_start[e] + i / 128;
                my_m = i % 128;
            }
        } else {
            const int rank = dst_of_route[r];     // local rank written by the count pass
            if (rank >= 0) {
                const int e = topk_idx[r];
                const int64_t row = (int64_t)chunk_first[(r / kPermChunk) * E + e] + rank;
                if (row < rows_cap) {
                    my_dst = (int)row;
                    src_of_row[row] = (int32_t)r;
                    const int i = (int)(row - group_offsets[e]);
                    my_tile = mtile_start[e] + i / 128;
                    my_m = i % 128;
                } else {
                    raise_device_error(err, MOE_DEVERR_CAPACITY);
                }
            }
            dst_of_route[r] = my_dst;
        }
    }
    int dst[KMAX], tile[KMAX], mm[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        dst[j] = j < k ? __shfl_sync(0xFFFFFFFFu, my_dst, j) : -1;
        tile[j] = __shfl_sync(0xFFFFFFFFu, my_tile, j);
        mm[j] = __shfl_sync(0xFFFFFFFFu, my_m, j);
    }
    // Four lanes share one 32-element block (8 bf16 each), so every load and every
    // code store of the warp is 512 / 256 contiguous bytes; the block maximum takes
    // two shuffles and one lane in four packs its group's scale bytes into a word.
    const int kb128 = H / 128;
    const uint4 *src = x + t * (H / 8);
    constexpr int U = 4;                       // 256-element slices in flight per lane
    for (int base = 0; base < H; base += 256 * U) {
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e0 = base + u * 256 + lane * 8;
            raw[u] = e0 < H ? __ldg(src + e0 / 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e0 = base + u * 256 + lane * 8;
            float v[8];
            const __nv_bfloat162 *hp = reinterpret_cast<const __nv_bfloat162 *>(&raw[u]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(hp[i]);
                v[2 * i] = f.x;
                v[2 * i + 1] = f.y;
            }
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
            const int X = mx::scale_exp(a);
            const uint2 q = mx::quantize8(v, X);
            // scale bytes of the 4 blocks of this half-warp (blocks kb0 .. kb0+3), one word
            const uint32_t byte = (uint32_t)(X + 127);
            const int g0 = lane & 16;
            const uint32_t word = __shfl_sync(0xFFFFFFFFu, byte, g0) | (__shfl_sync(0xFFFFFFFFu, byte, g0 + 4) << 8) |
                                  (__shfl_sync(0xFFFFFFFFu, byte, g0 + 8) << 16) |
                                  (__shfl_sync(0xFFFFFFFFu, byte, g0 + 12) << 24);
            if (e0 < H) {
                const int kb0 = (base + u * 256) / 32 + (lane >> 4) * 4;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < k && dst[j] >= 0) {
                        *reinterpret_cast<uint2 *>(x_q + (int64_t)dst[j] * H + e0) = q;
                        if ((lane & 15) == 0)
                            *reinterpret_cast<uint32_t *>(x_sf + mx::tile_sf_offset(tile[j], kb128, mm[j], kb0)) = word;
                    }
                }
            }
        }
    }
}

// The quantising scatter (KMAX >= k).
moe_status_t launch_scatter_mx(cudaStream_t s, const moe_bf16_t *x, const int32_t *topk_idx, int64_t T, int k, int E,
                               int H, const int32_t *counts, const int32_t *group_offsets,
                               const int32_t *mtile, int32_t *dst_of_route, int32_t *src_of_row, uint8_t *x_q,
                               uint8_t *x_sf, int64_t rows_cap, uint32_t *err) {
    const int64_t blocks = (T + kScatterWarps - 1) / kScatterWarps;
#define MOE_SCATTER_MX(KM)                                                                                   \
    launch_k(permute_scatter_mx_kernel<KM>, dim3((unsigned)blocks), dim3(kScatterWarps * 32), 0, s,               \
             reinterpret_cast<const uint4 *>(x), topk_idx, T, k, E, H, counts, group_offsets, mtile, \
             dst_of_route, src_of_row, x_q, x_sf, rows_cap, err)
    if (k <= 1) MOE_SCATTER_MX(1);
    else if (k <= 2) MOE_SCATTER_MX(2);
    else if (k <= 4) MOE_SCATTER_MX(4);
    else if (k <= 8) MOE_SCATTER_MX(8);
    else if (k <= 16) MOE_SCATTER_MX(16);
    else MOE_SCATTER_MX(32);
#undef MOE_SCATTER_MX
    return launch_status();
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_mxfp8(const moe_bf16_t *x, const int32_t *topk_idx, int64_t T, int H, int E,
                                          int k, uint8_t *x_q, uint8_t *x_sf, int64_t rows_cap,
                                          int32_t *dst_of_route, int32_t *src_of_row, int32_t *group_sizes,
                                          int32_t *group_offsets, void *ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX_RANGE("moe_permute_mxfp8");
    using namespace moe;
    if (T < 0 || H < 1 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || k < 1 || k > 32 || H % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!group_sizes || !group_offsets) return MOE_ERR_INVALID_ARG;
    const int64_t R = T * (int64_t)k;
    if (rows_cap < R) return MOE_ERR_INVALID_ARG;
    if (rows_cap >= 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !topk_idx || !x_q || !x_sf || !dst_of_route || !src_of_row)) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(x_q) % 8 ||
        reinterpret_cast<uintptr_t>(x_sf) % 4)
        return MOE_ERR_UNSUPPORTED;
    const size_t need = moe_workspace_bytes(T, E, k);
    if (!ws || ws_bytes < need || need == 0) return MOE_ERR_WORKSPACE;

    cudaStream_t s = (cudaStream_t)stream;
    uint32_t *err = ws_error_word(ws);
    const int64_t chunks = perm_chunks(R);
    int32_t *counts = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kWsHeaderBytes);
    int32_t *mtile = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kWsHeaderBytes + ws_counts_bytes(chunks, E));
    bool final_rows = false;
    if (count_and_scan(topk_idx, R, E, 1, rows_cap, dst_of_route, src_of_row, counts, group_sizes, group_offsets, mtile,
                       ws_done_counter(ws), err, s, &final_rows) != MOE_OK)
        return MOE_ERR_CUDA;
    if (T > 0 && launch_scatter_mx(s, x, topk_idx, T, k, E, H, final_rows ? nullptr : counts, group_offsets, mtile,
                                   dst_of_route, src_of_row, x_q, x_sf, rows_cap, err) != MOE_OK)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
