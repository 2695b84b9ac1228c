// gemm_launch.cuh -- host launch of one grouped GEMM op (persistent grid, one CTA per SM).
// a, b0, b1: operand load maps; c0, c1: the epilogue's output store maps.
#pragma once

#include "grouped_gemm.cuh"
#include "tmap.cuh"

namespace moe {
namespace gg {

template <Op OP, int BN>
moe_status_t launch(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1, const CUtensorMap &c0,
                    const CUtensorMap &c1, const Args &args, int64_t tiles_bound, cudaStream_t s) {
    using C = Cfg<OP, BN>;
    if (tiles_bound <= 0) return MOE_OK;
    auto kern = grouped_gemm_kernel<OP, BN>;
    static PerDeviceOnce once;   // per device: the smem attribute set
    int unused = 0;
    const moe_status_t st = once.get(
        [&](int *) {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) ==
                           cudaSuccess
                       ? MOE_OK
                       : MOE_ERR_CUDA;
        },
        &unused);
    if (st != MOE_OK) return st;
    const int64_t sms = device_sm_count();
    const int grid = (int)(tiles_bound < sms ? tiles_bound : sms);
    launch_k(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, s, a, b0, b1, c0, c1, args);
    return launch_status();
}

}  // namespace gg
}  // namespace moe
