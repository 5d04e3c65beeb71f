// Host helpers shared by the TMA-fed kernels: tensor-map encoding through the
// driver entry point, and the SM count of the current device.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace moe {

// Row-major tensor of `rank` (2 or 3) dims, dims[0] innermost, elements of
// esize bytes (2 = bf16 / f16, 1 = byte codes); box of box_cols x box_rows
// (x 1); 128-byte swizzle unless swizzle is false (the box then lands densely,
// row after row); out-of-range elements read as zero.
bool tmap_encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, int esize, uint32_t box_cols,
                 uint32_t box_rows, bool swizzle = true);

int device_sm_count();

}  // namespace moe
