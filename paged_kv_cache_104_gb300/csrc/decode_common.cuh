// Work planning shared by the decode kernels: a ragged batch becomes a flat
// list of (sequence, KV head, split) units through a prefix sum of splits
// per sequence, built in shared memory by every CTA.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace pkv {

struct Unit {
  int b, g, s, ns, tok_begin, tok_end;
};

// Length of row b (0 if the row is invalid; then err is set by the planner).
__device__ __forceinline__ int row_len(const DecodeArgs& a, int b) {
  return a.chunk_prior >= 0 ? a.chunk_prior + b + 1 : a.seq_lens[b];
}

// Build cu[0..B] (units per sequence, prefix-summed) with warp 0.
__device__ __forceinline__ void plan_units(const DecodeArgs& a, int* cu) {
  const int lane = threadIdx.x & 31;
  constexpr unsigned kAll = 0xffffffffu;
  if (threadIdx.x < 32) {
    int carry = 0;
    if (lane == 0) cu[0] = 0;
    const int limit = min(a.max_seq_len, a.max_blocks_per_seq * kBlockSize);
    for (int base = 0; base < a.num_seqs; base += 32) {
      const int b = base + lane;
      int units = 0;
      if (b < a.num_seqs) {
        const int n = row_len(a, b);
        if (n < 1 || n > limit) {
          record_error(a.err, DEVERR_SEQLEN_RANGE);
        } else {
          units = a.num_kv_heads * ((n + a.split_tokens - 1) / a.split_tokens);
        }
      }
      int x = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kAll, x, o);
        if (lane >= o) x += y;
      }
      if (b < a.num_seqs) cu[b + 1] = carry + x;
      carry += __shfl_sync(kAll, x, 31);
    }
  }
}

__device__ __forceinline__ Unit find_unit(const DecodeArgs& a, const int* cu, int w) {
  // largest b with cu[b] <= w  (cu is non-decreasing, cu[0] = 0 <= w < cu[B])
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= w) lo = mid; else hi = mid - 1;
  }
  Unit u;
  u.b = lo;
  const int rem = w - cu[lo];
  u.ns = (cu[lo + 1] - cu[lo]) / a.num_kv_heads;
  u.g = rem / u.ns;
  u.s = rem - u.g * u.ns;
  const int n = row_len(a, lo);
  u.tok_begin = u.s * a.split_tokens;
  u.tok_end = min(n, u.tok_begin + a.split_tokens);
  return u;
}

}  // namespace pkv
