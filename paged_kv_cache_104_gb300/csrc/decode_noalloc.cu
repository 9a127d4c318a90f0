// pkv_paged_decode_attention_noalloc: paged decode attention for callers
// that cannot allocate device memory.
//
// Some callers of this library have no way to hand it a workspace: an
// inference engine that reserves all device memory in its own pool at
// start-up and forbids any later cudaMalloc (a stray allocation can fail
// under memory pressure, fragment the pool, or synchronise the device in the
// middle of a step), or a plugin interface that passes only input and output
// pointers.  For them this entry point uses a scratch buffer that lives
// inside the library itself: a file-scope device array of
// PKV_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library
// holds until the process exits.
//
// The array is shared by all calls and keeps the last call's contents.  The
// split partials written there need no clearing: every partial the merge
// reads is written earlier in the same call.  Two calls whose kernels
// overlap on the GPU (different streams, or different host threads on one
// device) race on the array and give wrong results; serialise them.
//
// The first call on a device resolves the array's device address with
// cudaGetSymbolAddress (host code only sees a host-side stand-in for the
// array, which a kernel must never be given).  Make that first call before
// capturing any stream.  After a device reset the next call resolves the
// address again, in the new context; that call, too, belongs before any
// capture.
#include <cuda_runtime.h>

#include <mutex>

#include "host_cache.h"
#include "pagedkv.h"

namespace {

constexpr int kMaxDevicesNA = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Per device: the array's device address and the context it was resolved in.
struct ScratchAddr {
  uint64_t ctx;
  void* addr;
};
ScratchAddr g_scratch_addr[kMaxDevicesNA];
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device.  Resolved on the
// first call with that device current, and again when the context has
// changed since (a device reset destroys the primary context, and with it the
// array; the address resolved before it would point into freed memory).
pkv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNA) return PKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& s = g_scratch_addr[dev];
  const uint64_t ctx = pkv::current_context_id();
  if (!s.addr || ctx == 0 || ctx != s.ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PKV_ECUDA;
    s.addr = p;
    s.ctx = pkv::current_context_id();
  }
  *out = s.addr;
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
    int max_seq_len, int64_t num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, float scale, pkv_dtype dtype, pkv_stream_t stream) {
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len);
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERANGE;
  void* scratch = nullptr;
  if (need > 0) {
    const pkv_status st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
  }
  return pkv_paged_decode_attention(out, q, k_cache, v_cache, block_table, seq_lens, num_seqs,
                                    max_blocks_per_seq, max_seq_len, num_blocks, num_q_heads,
                                    num_kv_heads, head_dim, block_size, scale, scratch,
                                    need > 0 ? (size_t)PKV_NOALLOC_SCRATCH_BYTES : 0, dtype,
                                    stream);
}
