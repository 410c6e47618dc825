// tmap.cuh - TMA tensor maps over row-major matrices (built on the host with
// the driver's cuTensorMapEncodeTiled, fetched once through the runtime's
// entry-point query). Shared by the tensor-core GEMMs.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace moe {

// 2-D bf16 map over a row-major [rows, cols] matrix, box [box_rows][box_cols]
// (box_cols * 2 bytes = 128, the swizzle span), 128-byte swizzle, zero fill
// outside the matrix.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                 uint32_t box_rows);

// 2-D map over a row-major [rows, cols] output, box [32 rows][32 cols]: fp32
// with the 128-byte swizzle, or bf16 with the 64-byte swizzle. Stores
// outside the matrix are clipped.
bool make_map_2d_out(CUtensorMap* m, void* base, uint64_t rows, uint64_t cols, bool f32);

}  // namespace moe
