// Host helpers that build TMA tensor maps through the driver entry point
// (no link against libcuda).  Internal to the library.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace pkv {

// The pool [num_blocks][num_kv_heads][16][128] bf16 viewed as 2-D rows of
// 128 elements; box = 16 rows x 64 columns with 128-byte swizzle (one
// 64-column half of one (block, head) tile).  False if rows >= 2^31 or the
// driver refuses.
bool encode_pool_map_bf16(CUtensorMap* map, const void* base, int64_t rows);

// The fp8 pool [num_blocks][num_kv_heads][16][128] bytes as 2-D rows of 128
// bytes; box = 16 rows x 128 bytes (one whole (block, head) tile) with
// 128-byte swizzle.
bool encode_pool_map_u8(CUtensorMap* map, const void* base, int64_t rows);

// q or out [n][heads][128] bf16 as a 3-D map; box = 64 x 1 x 128 rows, 128-byte swizzle.
bool encode_rows_map_bf16(CUtensorMap* map, const void* base, int64_t n, int heads);

}  // namespace pkv
