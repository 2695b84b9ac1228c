// tmap.cuh -- host-side TMA tensor-map encoding (driver entry point fetched at run time).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// The driver's encoder, fetched once (a function-local static: initialised by one thread).
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return nullptr;
    }();
    return fn;
}

// Tiled map over a row-major tensor of `dtype` elements of `elem_bytes`
// bytes: dims[0] is the contiguous dimension; strides_bytes[i] is the byte
// stride of dims[i+1].  128-byte swizzle unless given, zero fill out of bounds.
inline bool encode_tmap(CUtensorMap *m, CUtensorMapDataType dtype, int rank, const void *base,
                        const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = tmap_encoder();
    if (!fn) return false;
    if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
    CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D bf16 matrix [outer, inner] with row pitch `ld` elements.
inline bool tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld,
                         uint32_t box_inner, uint32_t box_outer) {
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {ld * 2};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box);
}

// 3-D bf16 tensor [d2, d1, d0] (d0 contiguous), densely packed.
inline bool tmap_bf16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint32_t box0, uint32_t box1) {
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const uint32_t box[3] = {box0, box1, 1};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box);
}

// A row-major bf16 matrix [rows, cols] (row pitch ld elements, cols % 64 == 0) seen as the
// 3-D tensor [cols / 64][rows][64] -- dimension 2 steps 64 columns (128 bytes) --, with
// boxes {64, box_rows, 2}: one load brings two adjacent 64-column chunks of box_rows rows,
// chunk after chunk, each a 128-byte-swizzled block (the MN-major operand layout with
// chunks box_rows * 128 bytes apart).
inline bool tmap_bf16_col_chunks(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld,
                                 uint32_t box_rows) {
    const uint64_t dims[3] = {64, rows, cols / 64};
    const uint64_t strides[2] = {ld * 2, 128};
    const uint32_t box[3] = {64, box_rows, 2};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box);
}

// Store map of the GEMM epilogue: 2-D row-major [outer, inner] of `elem_bytes`-byte
// elements (bf16, fp32 or bytes), row pitch `ld` elements; boxes of 64 bytes x 32 rows
// in the 64-byte swizzle (the epilogue's staging slots).
inline bool tmap_store_2d(CUtensorMap *m, const void *base, int elem_bytes, uint64_t inner, uint64_t outer,
                          uint64_t ld) {
    const CUtensorMapDataType dt = elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {ld * (uint64_t)elem_bytes};
    const uint32_t box[2] = {(uint32_t)(64 / elem_bytes), 32};
    return encode_tmap(m, dt, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Store map without swizzle: 2-D row-major [outer, inner] of `elem_bytes`-byte elements
// (bf16, fp32 or bytes), row pitch `ld` elements, boxes of box_inner x box_rows (dense rows in
// shared memory).
inline bool tmap_store_plain(CUtensorMap *m, const void *base, int elem_bytes, uint64_t inner, uint64_t outer,
                             uint64_t ld, uint32_t box_inner, uint32_t box_rows) {
    const CUtensorMapDataType dt = elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {ld * (uint64_t)elem_bytes};
    const uint32_t box[2] = {box_inner, box_rows};
    return encode_tmap(m, dt, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 2-D byte matrix [outer, inner] with row pitch `ld` bytes (E4M3 data).
inline bool tmap_u8_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld,
                       uint32_t box_inner, uint32_t box_outer) {
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {ld};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box);
}

// 3-D byte tensor [d2, d1, d0] (d0 contiguous), densely packed.
inline bool tmap_u8_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                       uint32_t box1) {
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t strides[2] = {d0, d0 * d1};
    const uint32_t box[3] = {box0, box1, 1};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box);
}

// Blocks of `row_bytes`-byte rows stored one after another (the pre-swizzled MXFP8 weight
// blocks, rows of 128 bytes; the 512-byte scale atoms, rows of 16 bytes) as a 2-D byte
// tensor [rows, row_bytes] without swizzle, boxes of box_rows rows: a load copies the bytes
// as they are.
inline bool tmap_u8_rows(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
    const uint64_t dims[2] = {row_bytes, rows};
    const uint64_t strides[1] = {row_bytes};
    const uint32_t box[2] = {(uint32_t)row_bytes, box_rows};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// MXFP8 row scales in the tile layout ([tile][K/128] atoms of 32 x 16 bytes) as the 4-D byte
// tensor [tiles][K/128][32][16]; a box holds the atoms of one K block of two consecutive
// tiles (1 KB), tiles past the end read as zeros.
inline bool tmap_sf_tile_pairs(CUtensorMap *m, const void *base, uint64_t kblocks, uint64_t tiles) {
    const uint64_t dims[4] = {16, 32, kblocks, tiles};
    const uint64_t strides[3] = {16, 512, kblocks * 512};
    const uint32_t box[4] = {16, 32, 1, 2};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace moe
