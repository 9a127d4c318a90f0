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
// is skipped and reported in the error word.  With v_new null only the first
// pool is written (the latent cache has one pool).
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
    *reinterpret_cast<uint4*>(static_cast<char*>(a.k_cache) + dst) = kv;
    if (a.v_new) {   // null for a single pool (the latent cache)
      const uint4 vv = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.v_new) + src));
      *reinterpret_cast<uint4*>(static_cast<char*>(a.v_cache) + dst) = vv;
    }
  }
}

// One thread quantises 16 elements (one 16-byte chunk of the fp8 row) of K
// and of V: code = E4M3(x / scale[head]), the division in IEEE fp32.
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(const AppendFp8Args a) {
  const int chunks = a.head_dim / 16;
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
    const int64_t dst = ((blk * a.num_kv_heads + h) * kBlockSize + r) * a.head_dim + c * 16;
    const int64_t src = row * a.head_dim + c * 16;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint4* sp = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(which ? a.v_new : a.k_new) + src);
      const uint4 w0 = __ldg(sp), w1 = __ldg(sp + 1);
      const float sc = __ldg((which ? a.v_scale : a.k_scale) + h);
      const uint32_t in[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      uint32_t out[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint16_t p0 = f32x2_to_e4m3x2(__fdiv_rn(bf16lo(in[2 * j]), sc),
                                            __fdiv_rn(bf16hi(in[2 * j]), sc));
        const uint16_t p1 = f32x2_to_e4m3x2(__fdiv_rn(bf16lo(in[2 * j + 1]), sc),
                                            __fdiv_rn(bf16hi(in[2 * j + 1]), sc));
        out[j] = (uint32_t)p0 | ((uint32_t)p1 << 16);
      }
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(which ? a.v_cache : a.k_cache) + dst) =
          make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
}

}  // namespace

cudaError_t launch_kv_append_fp8(const AppendFp8Args& a, cudaStream_t stream) {
  const int64_t total = a.num_tokens * a.num_kv_heads * (a.head_dim / 16);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  kv_append_fp8_kernel<<<(int)blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
  const int64_t total = a.num_tokens * a.num_kv_heads * (a.row_bytes / 16);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  kv_append_kernel<<<(int)blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv
