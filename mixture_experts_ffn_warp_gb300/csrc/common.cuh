// common.cuh -- shared host/device helpers of the CUDA path (not part of the ABI).
#pragma once

#include <initializer_list>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Workspace layout: [0, 256) header (uint32 error word at offset 0), then the
// permutation's per-chunk expert counts.
constexpr size_t kWsHeaderBytes = 256;

// Routes per chunk of the permutation's counting pass.
constexpr int kPermWarps = 8;
constexpr int kPermSteps = 8;
constexpr int kPermChunk = kPermWarps * 32 * kPermSteps;   // 2048 routes

inline int64_t perm_chunks(int64_t R) { return (R + kPermChunk - 1) / kPermChunk; }

// True when every pointer is 16-byte aligned (null counts as aligned): the row kernels move
// 16-byte vectors, so an entry point returns MOE_ERR_UNSUPPORTED before launching on anything else.
inline bool all_aligned16(std::initializer_list<const void *> ps) {
    for (const void *p : ps)
        if (reinterpret_cast<uintptr_t>(p) % 16) return false;
    return true;
}

// Workspace layout after the header: per-chunk expert counts, then (for the
// MXFP8 path) each group's first 128-row M-tile id, [E+1] int32.
inline size_t ws_counts_bytes(int64_t chunks, int E) {
    return ((size_t)chunks * (size_t)E * sizeof(int32_t) + 15) / 16 * 16;
}
inline size_t ws_mtile_bytes(int E) { return ((size_t)(E + 1) * sizeof(int32_t) + 15) / 16 * 16; }

// mtile_start[g] = sum over g' < g of ceil(rows(g') / 128) from group offsets (one block, G <= 1024).
__global__ void mtile_prefix_kernel(const int32_t *__restrict__ group_offsets, int G, int32_t *__restrict__ mtile_start);

// NVTX range around each entry point of the C ABI (named after the call), so that a
// timeline tool shows which call enqueued which kernels.  Without a tool attached an NVTX
// call returns at once.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define MOE_NVTX_RANGE(name) ::moe::NvtxRange moe_nvtx_range_(name)

inline uint32_t *ws_error_word(void *ws) { return reinterpret_cast<uint32_t *>(ws); }

// Limit of the GEMM pipelines' device spin waits (their mbarrier waits), in ns: the
// workspace header's uint32 at offset 8 (0 = the default, 2 s), set with
// moe_workspace_set_wait_limit.  A wait past it sets MOE_DEVERR_TIMEOUT and the kernel
// winds down (it lets its issued copies and MMAs finish, frees TMEM and exits).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
inline uint32_t *ws_wait_limit(void *ws) { return reinterpret_cast<uint32_t *>(ws) + 2; }
// Read by the kernels after their programmatic-launch wait (the error word is header word 0).
__device__ __forceinline__ uint64_t device_wait_limit(const uint32_t *err) {
    const uint32_t v = err ? __ldcg(err + 2) : 0u;
    return v ? (uint64_t)v : kDefaultWaitNs;
}
// Blocks of the permutation's counting pass that have finished (header offset 4); the last
// one to finish runs the scan and sets it back to zero.
inline uint32_t *ws_done_counter(void *ws) { return reinterpret_cast<uint32_t *>(ws) + 1; }

inline moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Status of the last launch on this thread (clears the sticky-free error).
inline moe_status_t launch_status() { return cuda_status(cudaGetLastError()); }

int device_sm_count();

// Per-device launch set-up of one kernel (its shared-memory attribute, an occupancy
// query), done once per device and read by every later launch on it.  Indexed by device
// ordinal and filled under a mutex, so that host threads driving different GPUs through
// the library never race on it.
struct PerDeviceOnce {
    static constexpr int kMaxDevices = 128;
    std::mutex lock;
    bool done[kMaxDevices] = {};
    int value[kMaxDevices] = {};

    // The value for the current device, computing it with init(&value) -> moe_status_t
    // the first time; init failing leaves the device unset (retried by the next launch).
    template <typename Init>
    moe_status_t get(Init &&init, int *out) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
        if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
        std::lock_guard<std::mutex> g(lock);
        if (!done[dev]) {
            int v = 0;
            const moe_status_t st = init(&v);
            if (st != MOE_OK) return st;
            value[dev] = v;
            done[dev] = true;
        }
        *out = value[dev];
        return MOE_OK;
    }
};

// out[t] = bf16(sum_j w[t,j] * y[dst[t,j]]) over fp32 rows of y (w == nullptr: weights 1).
cudaError_t combine_rows(const float *y, const int32_t *dst, const float *w, int64_t T, int H, int k,
                         moe_bf16_t *out, cudaStream_t s);

__device__ __forceinline__ void raise_device_error(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// Bounds-check builds (-DMOE_BOUNDS_CHECK; compute-sanitizer is not available for this
// library's tests): a GEMM first checks the group offsets it read from device memory -- the
// one data-dependent extent its loads, MMAs and stores trust -- and on a violation raises
// MOE_DEVERR_BOUNDS and computes nothing.  Called by one whole warp over s_off[0..G]; true
// when 0 <= s_off[0] <= ... <= s_off[G] <= rows_cap.  Always true in other builds.
__device__ __forceinline__ bool group_offsets_in_bounds(const int *s_off, int G, int64_t rows_cap, int lane,
                                                        uint32_t *err) {
#ifdef MOE_BOUNDS_CHECK
    bool bad = false;
    for (int i = lane; i <= G; i += 32) {
        const int v = s_off[i];
        if (v < 0 || v > rows_cap || (i < G && v > s_off[i + 1])) bad = true;
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (bad && lane == 0) raise_device_error(err, MOE_DEVERR_BOUNDS);
    return !bad;
#else
    (void)s_off; (void)G; (void)rows_cap; (void)lane; (void)err;
    return true;
#endif
}

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream serialization, so the
// GPU may schedule it as the kernel before it on the stream drains, instead of after that
// kernel has fully completed.  Each kernel calls pdl_wait() before its first global-memory
// access and before any early return: griddepcontrol.wait blocks until the preceding grid
// has completed and its writes are visible, so nothing a kernel reads or writes can race
// with earlier work on the stream.  Only on-chip set-up (mbarriers, TMEM allocation,
// tensor-map prefetch) runs before it.  Only the permutation's counting pass triggers its
// dependent early (griddepcontrol.launch_dependents, right after its own wait): it runs a
// few CTAs, so the scatter's CTAs fill the idle SMs and load their token rows meanwhile.
// Measured on the forward chain, an early trigger in every kernel let the next grid's CTAs
// occupy SMs during the whole kernel and cost more than it saved, while the implicit
// trigger at CTA exit removes most of the launch gap.  Without the launch attribute the
// wait is a no-op and the launch behaves as an ordinary one.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream be scheduled before this one ends.  Called after
// pdl_wait(), so a dependent that starts early knows that every grid before this one has
// completed: what those grids wrote may be read before the dependent's own wait.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Kernel launch with programmatic stream serialization (arguments are converted to the
// kernel's parameter types).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

}  // namespace moe
