// kv_append: scatter each new token's key and value rows into the paged
// pools ("KV cache and continuous batching: 1,000 people ask AI", section
// "What does a KV cache keep?": a decode step appends the new key and value
// to the cache before attending).
//
// k_new, v_new [T][Hkv][D] -> pools [num_blocks][Hkv][16][D] at
// slot = block * 16 + row.  One thread moves one 16-byte chunk of one row of
// K and the same chunk of V, so reads of k_new/v_new are fully coalesced and
// every destination row is written by D*size/16 adjacent threads.  The copy
// is bit-exact.  slot < 0 is padding and is skipped; a slot beyond the pool
// is skipped and reported in the error word.
#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  const int chunks = a.row_bytes / 16;
  const int64_t total = a.num_tokens * a.num_kv_heads * chunks;
  const int64_t pool_slots = a.num_blocks * kBlockSize;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / chunks;
    const int c = (int)(i - row * chunks);
    const int64_t t = row / a.num_kv_heads;
    const int h = (int)(row - t * a.num_kv_heads);
    const int64_t slot = __ldg(a.slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      record_error(a.err, DEVERR_SLOT_RANGE);
      continue;
    }
    const int64_t blk = slot / kBlockSize, r = slot - blk * kBlockSize;
    const int64_t dst = ((blk * a.num_kv_heads + h) * kBlockSize + r) * a.row_bytes + c * 16;
    const int64_t src = row * a.row_bytes + c * 16;
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.k_new) + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.v_new) + src));
    *reinterpret_cast<uint4*>(static_cast<char*>(a.k_cache) + dst) = kv;
    *reinterpret_cast<uint4*>(static_cast<char*>(a.v_cache) + dst) = vv;
  }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
  const int64_t total = a.num_tokens * a.num_kv_heads * (a.row_bytes / 16);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  kv_append_kernel<<<(int)blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv
