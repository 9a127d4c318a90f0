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

// The latent pool [num_blocks][16][128] bf16, one whole block per box: a 4-D
// view (column x of 64, row y of 8, half z of 2, 8-row group w) with box
// 64 x 8 x 2 x 2 and 128-byte swizzle.  A block lands in shared memory as
// [row group][half][8 rows][128 B], so every 8 rows x 64 columns form one
// 1 KiB swizzle atom.  False if 2 * num_blocks >= 2^31 or the driver refuses.
bool encode_latent_block_map(CUtensorMap* map, const void* base, int64_t num_blocks);

// Rows of 128 bf16 (e.g. [sequences * 32 heads][128]); box = 32 rows x 64
// columns, 128-byte swizzle.
bool encode_rows32_map_bf16(CUtensorMap* map, const void* base, int64_t rows);

}  // namespace pkv
