// tmap.h -- TMA tensor maps of the library's [slices][T][64] bf16 tensors.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fibattn {

// Rows of one box: every tiled copy moves 64 rows of 64 bf16 (8 KB).
constexpr int kTmaBoxRows = 64;

// Encodes a 3D map {64, T, slices} over a contiguous [slices][T][64] bf16 tensor: box
// {64, 64, 1}, 128-byte swizzle, zero fill outside [0, T) so that a box never reads across
// a slice boundary. Returns 0 (CUDA_SUCCESS) or the driver's CUresult (-1 when the entry
// point is missing). The driver needs a current context on the calling thread: callers
// make a runtime call that binds the device's primary context first.
int make_bf16_rows_map(CUtensorMap* m, const void* base, int64_t slices, int32_t T);

// The same map over rows of d bf16 (d a multiple of 64): the box still spans 64 columns, a
// copy takes the columns [x, x + 64) at an x that is a multiple of 64.
int make_bf16_rows_map_d(CUtensorMap* m, const void* base, int64_t slices, int32_t T, int32_t d);

// The same map with an 8-row box (1 KB): the rows just past a 128-row tile.
int make_bf16_rows8_map(CUtensorMap* m, const void* base, int64_t slices, int32_t T);

}  // namespace fibattn
