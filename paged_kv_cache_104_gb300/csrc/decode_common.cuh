// Work planning shared by the decode kernels: a ragged batch becomes a flat
// list of (sequence, KV head, split) units through a prefix sum of splits
// per sequence, built in shared memory by every CTA.  The bf16 decode can
// instead walk a balanced plan: the same prefix sum over stages (the
// kernel's load granule), cut into one equal share of stages per CTA.
#pragma once

#include <climits>

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

// Build cu[0..B] with warp 0: per sequence, num_kv_heads times the number of
// split_tokens-token splits (stage_tok = 0) or of stage_tok-token stages
// plus `pad` stages that hold no tokens, prefix-summed.  The padding stands
// for the fixed cost of a piece (loading its queries, writing its result):
// a CTA whose share starts many short sequences then gets fewer tokens.
// lens (optional, shared memory): every sequence's length is kept there too,
// so the walk does not read it from global memory at each unit.
__device__ __forceinline__ void plan_units(const DecodeArgs& a, int* cu, int stage_tok = 0,
                                           int pad = 0, int* lens = nullptr) {
  const int lane = threadIdx.x & 31;
  constexpr unsigned kAll = 0xffffffffu;
  if (threadIdx.x < 32) {
    int carry = 0;
    if (lane == 0) cu[0] = 0;
    const int limit = min(a.max_seq_len, a.max_blocks_per_seq * kBlockSize);
    // eight windows of 32 lengths are requested before the first is scanned,
    // so their load latencies overlap
    for (int base = 0; base < a.num_seqs; base += 256) {
      int n[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int b = base + 32 * k + lane;
        n[k] = b < a.num_seqs ? row_len(a, b) : 0;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (base + 32 * k >= a.num_seqs) break;
        const int b = base + 32 * k + lane;
        int units = 0;
        if (b < a.num_seqs) {
          if (n[k] < 1 || n[k] > limit) {
            record_error(a.err, DEVERR_SEQLEN_RANGE);
          } else {
            const int per = stage_tok > 0 ? stage_tok : a.split_tokens;
            units = a.num_kv_heads * ((n[k] + per - 1) / per + (stage_tok > 0 ? pad : 0));
          }
        }
        int x = units;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kAll, x, o);
          if (lane >= o) x += y;
        }
        if (b < a.num_seqs) {
          cu[b + 1] = carry + x;
          if (lens) lens[b] = n[k];
        }
        carry += __shfl_sync(kAll, x, 31);
      }
    }
  }
}

__device__ __forceinline__ Unit find_unit(const DecodeArgs& a, const int* cu, int w,
                                          const int* lens = nullptr) {
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
  const int n = lens ? lens[lo] : row_len(a, lo);
  u.tok_begin = u.s * a.split_tokens;
  u.tok_end = min(n, u.tok_begin + a.split_tokens);
  return u;
}

// Largest b with cu[b] <= w (cu non-decreasing, cu[0] = 0 <= w < cu[B]).
__device__ __forceinline__ int seq_of(const DecodeArgs& a, const int* cu, int64_t w) {
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= w) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// A CTA's walk over its work.  Split walk: units blockIdx.x, + gridDim.x, ...
// Balanced walk: CTA c takes stages [c S / C, (c + 1) S / C) of the S stages
// of cu (C = gridDim.x), cut where (sequence, KV head) streams change; each
// such piece is a unit whose s is its index among the pieces of its stream
// and ns their number (the CTAs its stages fall to).
struct Walk {
  bool balanced;
  const int* lens;   // sequence lengths in shared memory, or null (read seq_lens)
  int total;     // units (split walk) or stages (balanced walk)
  int w;         // split walk: next unit
  int64_t pos;   // balanced walk: next stage, and the end of this CTA's share
  int64_t end;
};

// The balanced walk needs a workspace for the piece counts and shares of at
// least kSplitTokens tokens of stages per CTA (so no stream is cut into more
// pieces than the workspace has partial slots); otherwise the split walk.

// True if the stage prefix sums of this call fit an int: every counted
// sequence has at most max_seq_len tokens (longer ones are rejected).
inline bool stage_plan_fits(const DecodeArgs& a, int stage_tok, int pad = 0) {
  return (int64_t)a.num_seqs * a.num_kv_heads *
             ((a.max_seq_len + stage_tok - 1) / stage_tok + pad) <
         (int64_t)INT_MAX;
}

// The CTA whose share holds stage p.  Units of work are cut where streams
// change, so every role of every CTA evaluates this at each of its units:
// 32-bit division when the operands fit (they do for any realistic batch), as
// a 64-bit division takes hundreds of cycles.
__device__ __forceinline__ int cta_of_stage(int64_t p, int64_t total) {
  const uint64_t num = (uint64_t)(p + 1) * gridDim.x - 1;
  if ((num >> 32) == 0 && ((uint64_t)total >> 32) == 0)
    return (int)((uint32_t)num / (uint32_t)total);
  return (int)(num / (uint64_t)total);
}

__device__ __forceinline__ Walk walk_begin(const DecodeArgs& a, const int* cu, bool balanced,
                                           const int* lens = nullptr) {
  Walk k;
  k.balanced = balanced;
  k.lens = lens;
  k.total = cu[a.num_seqs];
  k.w = blockIdx.x;
  k.pos = (int64_t)blockIdx.x * k.total / gridDim.x;
  k.end = (int64_t)(blockIdx.x + 1) * k.total / gridDim.x;
  return k;
}

// Next unit of this CTA (false when done).  stage_tok: tokens per stage;
// pad: the empty stages plan_units put after every stream (a CTA's share
// may end, or lie entirely, inside them: those are skipped).
__device__ __forceinline__ bool walk_next(const DecodeArgs& a, const int* cu, int stage_tok,
                                          Walk& k, Unit& u, int pad = 0) {
  if (!k.balanced) {
    if (k.w >= k.total) return false;
    u = find_unit(a, cu, k.w, k.lens);
    k.w += gridDim.x;
    return true;
  }
  while (k.pos < k.end) {
    const int b = seq_of(a, cu, k.pos);
    const int nst = (cu[b + 1] - cu[b]) / a.num_kv_heads;   // stages of one stream
    const int real = nst - pad;                              // the stream's own stages
    const int rem = (int)(k.pos - cu[b]);
    const int g = rem / nst;
    const int st0 = rem - g * nst;
    const int64_t s_begin = (int64_t)cu[b] + (int64_t)g * nst, s_end = s_begin + real;
    if (st0 >= real) {   // inside the padding: nothing to do up to the next stream
      k.pos = min(k.end, s_begin + nst);
      continue;
    }
    const int len = (int)(min(k.end, s_end) - k.pos);
    const int c0 = cta_of_stage(s_begin, k.total);
    u.b = b;
    u.g = g;
    u.s = (int)blockIdx.x - c0;
    u.ns = cta_of_stage(s_end - 1, k.total) - c0 + 1;
    u.tok_begin = st0 * stage_tok;
    u.tok_end = min(k.lens ? k.lens[b] : row_len(a, b), (st0 + len) * stage_tok);
    k.pos += len;
    return true;
  }
  return false;
}

}  // namespace pkv
