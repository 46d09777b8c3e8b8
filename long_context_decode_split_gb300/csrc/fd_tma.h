// fd_tma.h -- host side of the tiled TMA copies: 2-D tensor maps over a row
// matrix [rows, row_bytes] with 64-row x 128-byte boxes and the 128-byte
// swizzle.  In shared memory a box is 64 rows of 128 bytes; the 16-byte chunk
// c of row r sits at chunk position c ^ (r % 8) (box base 1024-byte aligned),
// which spreads the 8 rows that one tensor-core fragment load touches over
// all 32 banks.  The encoder is reached through the runtime's driver entry
// point, so the library needs no link against libcuda.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace fd {

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

inline EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        tried = true;
    }
    return fn;
}

// Tensor map for `rows` rows of `row_bytes` bytes, read as boxes of box_rows
// (64 unless given) rows x min(row_bytes, 128) bytes: row_bytes a multiple of 128 uses the 128-byte
// swizzle, row_bytes == 64 the 64-byte swizzle (chunk c of row r at
// position c ^ ((r / 2) % 4)), row_bytes == 32 no swizzle.  Elements are
// taken as 16-bit values, so the first coordinate counts 2-byte units; byte
// rows work the same way.  Returns false when the encoder is unavailable or
// rejects the arguments.
inline bool make_row_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_bytes,
                         uint32_t box_rows = 64) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc || rows == 0) return false;
    if (row_bytes % 128 != 0 && row_bytes != 64 && row_bytes != 32) return false;
    const uint32_t box_bytes = row_bytes >= 128 ? 128 : row_bytes;
    const cuuint64_t dims[2] = {row_bytes / 2, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes / 2, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                    : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over a plain vector of `n` elements of `elem_bytes` (4 or 2)
// bytes, read as boxes of `box` elements (box * elem_bytes a multiple of 16,
// box <= 256) without swizzle.  A copy must start at an index whose byte
// offset is a multiple of 16; elements past the end read as zero.
inline bool make_vec_map(CUtensorMap* map, const void* base, uint64_t n, uint32_t box, uint32_t elem_bytes = 4) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc || n == 0 || box == 0 || box > 256 || (elem_bytes != 4 && elem_bytes != 2) ||
        (box * elem_bytes) % 16 != 0)
        return false;
    const cuuint64_t dims[1] = {n};
    const cuuint64_t strides[1] = {n * elem_bytes};  // not read for a rank-1 map
    const cuuint32_t boxd[1] = {box};
    const cuuint32_t estr[1] = {1};
    const CUresult r = enc(map, elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 1,
                           const_cast<void*>(base), dims, strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace fd
