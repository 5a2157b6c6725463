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

}  // namespace csahca
