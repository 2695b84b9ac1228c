// carveout.cuh -- shared-memory carveout preference for the kernels around the permutation.
//
// The permutation's cluster counting pass takes all of an SM's shared memory.  An SM whose
// L1 / shared-memory split was last set for a kernel that asked for little shared memory
// must be reconfigured (drained, its L1 flushed) before such a CTA can start there.  The
// router, which runs just before the counting pass, and the bf16 scatter, which runs beside
// and after it, therefore ask for the largest carveout (they use no shared memory and read
// their rows past the L1): measured on GB300 (route + permute, L2 flushed): fine_grained
// 33.8 -> 31.7 us, mixtral 44.0 -> 42.0 us.  The quantising scatter reads its rows through
// the L1 and keeps the default split (with the largest carveout: 127 -> 135 us on the
// DeepSeek-V3 shape).
#pragma once

#include "common.cuh"

namespace moe {

// Sets the preference once per device and kernel; a refusal only leaves the default split.
template <auto KERN>
inline void prefer_max_smem_carveout() {
    static PerDeviceOnce once;
    int applied = 0;
    const moe_status_t st = once.get(
        [](int *v) {
            *v = 1;
            return cudaFuncSetAttribute(KERN, cudaFuncAttributePreferredSharedMemoryCarveout,
                                        (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess
                       ? MOE_OK
                       : MOE_ERR_CUDA;
        },
        &applied);
    if (st != MOE_OK) (void)cudaGetLastError();
}

}  // namespace moe
