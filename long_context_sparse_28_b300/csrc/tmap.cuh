// Host-side construction of TMA tensor maps (2-D, tiled) through the driver entry point, so the
// library needs no link-time dependency on the driver library.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace csahca {

// Encodes a 2-D tiled map over `rows` rows of `inner` elements (row pitch `pitch` bytes), box
// `box_inner` x `box_rows`, 128-byte swizzle, zero fill out of bounds.  Returns false when the
// driver entry point is missing or rejects the parameters (the caller then takes another path).
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t pitch, uint32_t box_inner, uint32_t box_rows);

// The same with the swizzle mode given (CU_TENSOR_MAP_SWIZZLE_NONE lands the box as dense rows)
// and only the 16-byte base alignment TMA itself asks for (a map may start inside a row).
bool encode_tmap_2d_sw(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t pitch, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// Encodes an N-D tiled map (N <= 5): dims[0] elements innermost, strides[i] = byte stride of
// dims[i + 1] (any order: a map may visit rows in a permuted order), box[i] per dimension,
// 128-byte swizzle.  False when the driver rejects it.
bool encode_tmap_nd(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box);

}  // namespace csahca
