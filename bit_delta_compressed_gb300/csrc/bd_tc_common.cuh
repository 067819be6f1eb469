// bd_tc_common.cuh -- host helpers shared by the tensor-core paths.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "bd_paths.cuh"

namespace bd {

// 2-D bf16 row-major [rows, cols] tensor map with a box of box_rows x 64
// columns (128 bytes: one 128-byte swizzle atom per row).  Returns false if
// the driver entry point is unavailable or rejects the description.
bool make_tmap_bf16_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows);

// 2-D byte matrix [rows, cols_bytes] with a box of box_rows x 128 bytes and
// the 128-byte swizzle (call after make_tmap_bf16_sw128 has resolved the
// driver entry point).
bool make_tmap_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols_bytes,
                        uint32_t box_rows);

// Packed sign bits [rows, words] u32 with a box of box_rows x 4 words (16
// bytes per row), no swizzle.
bool make_tmap_bits(CUtensorMap* map, const void* base, uint64_t rows, uint64_t words, uint32_t box_rows);

// Opt a kernel into `bytes` of dynamic shared memory (once per device).
bool set_smem_attr(const void* kernel, int bytes, int slot);

}  // namespace bd
