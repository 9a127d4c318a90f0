// Prefix caching over the paged KV cache: chained block hashes and a
// hash -> physical block index ("The KV cache and prefix caching", section
// "A prefix already in the cache can skip its prefill").
//
// The pages fix the rules this follows:
//  * the prompt is hashed block by block, 16 tokens per block;
//  * a block's identifier covers its own tokens together with the identifier
//    of the block before it (chaining), so two sequences agree on a block's
//    identifier only if they agree on every token up to and including it,
//    and a match is always a contiguous prefix starting at position 0;
//  * hits are counted in whole blocks, so the last partial block is always
//    recomputed.
// The pages name no hash function; this uses 64-bit FNV-1a (Fowler, Noll and
// Vo), fed the previous identifier as 8 little-endian bytes and then each
// token id as 4 little-endian bytes.  The first block's "previous identifier"
// is the caller's parent value (0 for a fresh prompt).
//
// Host code only; the index lives in host memory and is not thread-safe.
#include <stdint.h>
#include <stdlib.h>

#include <new>
#include <unordered_map>

#include "pagedkv.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

inline uint64_t fnv1a_byte(uint64_t h, uint8_t b) { return (h ^ b) * kFnvPrime; }

uint64_t block_hash(uint64_t parent, const int32_t* tokens, int block_size) {
  uint64_t h = kFnvOffset;
  for (int i = 0; i < 8; ++i) h = fnv1a_byte(h, (uint8_t)(parent >> (8 * i)));
  for (int t = 0; t < block_size; ++t) {
    const uint32_t v = (uint32_t)tokens[t];
    for (int i = 0; i < 4; ++i) h = fnv1a_byte(h, (uint8_t)(v >> (8 * i)));
  }
  return h;
}

}  // namespace

struct pkv_prefix_cache {
  std::unordered_map<uint64_t, int32_t> map;
};

extern "C" {

uint64_t pkv_fnv1a64(const void* data, size_t len) {
  uint64_t h = kFnvOffset;
  const uint8_t* p = static_cast<const uint8_t*>(data);
  for (size_t i = 0; i < len; ++i) h = fnv1a_byte(h, p[i]);
  return h;
}

int64_t pkv_prefix_hash_blocks(const int32_t* tokens, int64_t num_tokens, int block_size,
                               uint64_t parent, uint64_t* out_hashes) {
  if (num_tokens < 0 || block_size < 1 || (num_tokens > 0 && (!tokens || !out_hashes))) return -1;
  const int64_t n = num_tokens / block_size;
  uint64_t h = parent;
  for (int64_t b = 0; b < n; ++b) {
    h = block_hash(h, tokens + b * block_size, block_size);
    out_hashes[b] = h;
  }
  return n;
}

pkv_prefix_cache* pkv_prefix_cache_create(void) {
  return new (std::nothrow) pkv_prefix_cache();
}

void pkv_prefix_cache_destroy(pkv_prefix_cache* cache) { delete cache; }

int64_t pkv_prefix_cache_size(const pkv_prefix_cache* cache) {
  return cache ? (int64_t)cache->map.size() : -1;
}

pkv_status pkv_prefix_cache_insert(pkv_prefix_cache* cache, const uint64_t* hashes,
                                   const int32_t* block_ids, int64_t n) {
  if (!cache || n < 0 || (n > 0 && (!hashes || !block_ids))) return PKV_EINVAL;
  try {
    for (int64_t i = 0; i < n; ++i) {
      if (block_ids[i] < 0) return PKV_EINVAL;
      cache->map.emplace(hashes[i], block_ids[i]);  // an existing entry is kept
    }
  } catch (...) {
    return PKV_ERANGE;
  }
  return PKV_OK;
}

pkv_status pkv_prefix_cache_evict(pkv_prefix_cache* cache, const uint64_t* hashes, int64_t n) {
  if (!cache || n < 0 || (n > 0 && !hashes)) return PKV_EINVAL;
  for (int64_t i = 0; i < n; ++i) cache->map.erase(hashes[i]);
  return PKV_OK;
}

int64_t pkv_prefix_cache_match(const pkv_prefix_cache* cache, const uint64_t* hashes, int64_t n,
                               int32_t* out_block_ids) {
  if (!cache || n < 0 || (n > 0 && !hashes)) return -1;
  int64_t m = 0;
  for (; m < n; ++m) {
    auto it = cache->map.find(hashes[m]);
    if (it == cache->map.end()) break;
    if (out_block_ids) out_block_ids[m] = it->second;
  }
  return m;
}

int64_t pkv_prefix_plan(const pkv_prefix_cache* cache, const int32_t* tokens, int64_t num_tokens,
                        int block_size, int32_t* out_block_ids, uint64_t* out_hashes) {
  if (!cache || num_tokens < 1 || block_size < 1 || !tokens || !out_hashes) return -1;
  const int64_t n = pkv_prefix_hash_blocks(tokens, num_tokens, block_size, 0, out_hashes);
  if (n < 0) return -1;
  // at least the prompt's last token is recomputed, so a whole-block prompt
  // that is fully cached still gets a query for its first output token
  const int64_t usable = (num_tokens - 1) / block_size;
  const int64_t m = pkv_prefix_cache_match(cache, out_hashes, usable < n ? usable : n, out_block_ids);
  return m < 0 ? -1 : m * block_size;
}

}  // extern "C"
