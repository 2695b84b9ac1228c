// abi.cu -- status strings, workspace management and the device error word.
#include "common.cuh"

namespace moe {

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

// One word of a workspace header written in stream order (capturable, no host copy).
__global__ void set_word_kernel(uint32_t *word, uint32_t value) {
    pdl_wait();
    *word = value;
}

}  // namespace moe

extern "C" {

const char *moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_DATA: return "MOE_ERR_DEVICE_DATA";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    }
    return "MOE_ERR_UNKNOWN";
}

int moe_abi_version(void) { return 1; }

size_t moe_workspace_bytes(int64_t T, int E, int k) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32) return 0;
    int64_t chunks = moe::perm_chunks(T * (int64_t)k);
    return moe::kWsHeaderBytes + moe::ws_counts_bytes(chunks, E) + moe::ws_mtile_bytes(E);
}

size_t moe_mx_tile_scale_bytes(int64_t rows_cap, int E, int K) {
    if (rows_cap < 0 || E < 1 || K < 128 || K % 128 != 0) return 0;
    return (size_t)((rows_cap + 127) / 128 + E) * (size_t)(K / 128) * 512;
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ws || ws_bytes < moe::kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    return moe::cuda_status(cudaMemsetAsync(ws, 0, moe::kWsHeaderBytes, (cudaStream_t)stream));
}

moe_status_t moe_workspace_set_wait_limit(void *ws, size_t ws_bytes, uint32_t limit_ns, moe_stream_t stream) {
    if (!ws || ws_bytes < moe::kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    moe::launch_k(moe::set_word_kernel, dim3(1), dim3(1), 0, (cudaStream_t)stream, moe::ws_wait_limit(ws), limit_ns);
    return moe::launch_status();
}

moe_status_t moe_read_device_error(const void *ws, moe_stream_t stream, uint32_t *out) {
    if (!ws || !out) return MOE_ERR_INVALID_ARG;
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    *out = v;
    return v ? MOE_ERR_DEVICE_DATA : MOE_OK;
}

}  // extern "C"
