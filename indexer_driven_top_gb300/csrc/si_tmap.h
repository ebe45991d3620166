// si_tmap.h -- host-side creation of TMA tensor maps (driver entry point
// fetched through the runtime, so libsi does not link libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace si {

// 2-D map over a row-major byte matrix [rows, row_bytes] with row stride
// `stride` bytes; boxes of `box_rows` x `box_bytes`, written to shared memory
// with the 128-byte swizzle.  Returns cudaErrorInvalidValue if the driver
// rejects the description.
cudaError_t make_tmap_2d_u8_sw128(CUtensorMap *map, const void *base, uint64_t row_bytes,
                                  uint64_t rows, uint64_t stride, uint32_t box_bytes,
                                  uint32_t box_rows);

}  // namespace si
