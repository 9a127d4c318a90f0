// C ABI of libpagedkv.so: argument validation, workspace layout, dispatch to
// the kernel launchers, and the per-device error word.  The declarations and
// their contracts are in include/pagedkv.h.
#include <climits>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "host_cache.h"
#include "launch.h"
#include "pagedkv.h"

namespace {

constexpr int kMaxDevices = 64;

// One error word per device: kernels record the first device-side error here.
__device__ int g_pkv_error_word;

// Per device: the context the cached state was resolved in, the device-side
// address of the error word and the SM count.  Resolved on the first call
// with that device current, and again after the context changes (a device
// reset destroys the primary context and the module with it).  Guarded by a
// mutex: host threads may make their first calls at the same time.
struct DeviceState {
  uint64_t ctx;
  int* err;
  int num_sms;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pkv_dtype d) { return d == PKV_BF16 ? 2 : 4; }

bool dtype_ok(pkv_dtype d) { return d == PKV_F32 || d == PKV_BF16; }

pkv_status device_state(int** err, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceState& s = g_dev[dev];
  uint64_t ctx = pkv::current_context_id();
  if (!s.err || ctx == 0 || ctx != s.ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_error_word) != cudaSuccess) return PKV_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ECUDA;
    s.num_sms = sms;
    s.err = static_cast<int*>(p);
    s.ctx = pkv::current_context_id();   // now that the runtime made one current
  }
  *err = s.err;
  *num_sms = s.num_sms;
  return PKV_OK;
}

int max_splits_for(int max_seq_len) {
  return (max_seq_len + pkv::kSplitTokens - 1) / pkv::kSplitTokens;
}

// Partial slots per (sequence, query head) row: a sequence of n tokens gives
// at most ceil(n / kSplitTokens) partials in 512-token splits, and at most
// one more in the bf16 decode's balanced walk (each CTA's share of at least
// 512 tokens may start inside a sequence).  One slot: no partials at all.
int partial_slots_for(int max_seq_len) {
  const int s = max_splits_for(max_seq_len);
  return s <= 1 ? 1 : s + 1;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The decode workspace, in order: fp32 partial rows [rows][head_dim], their
// (m, l) pairs [rows][2], and the partial count per (sequence, head) [count],
// rows = num_seqs * num_q_heads * partial slots.
struct Partials {
  float* acc;
  float* ml;
  int* np;
};
Partials carve_partials(void* workspace, size_t rows, int head_dim) {
  char* ws = static_cast<char*>(workspace);
  const size_t acc_b = align256(rows * head_dim * sizeof(float));
  const size_t ml_b = align256(rows * 2 * sizeof(float));
  return {reinterpret_cast<float*>(ws), reinterpret_cast<float*>(ws + acc_b),
          reinterpret_cast<int*>(ws + acc_b + ml_b)};
}

// Shape checks shared by decode and prefill.
pkv_status check_heads(int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       pkv_dtype dtype) {
  if (!dtype_ok(dtype)) return PKV_EDTYPE;
  if (num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1) return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (block_size != pkv::kBlockSize) return PKV_EUNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (!pkv::decode_supported(dtype == PKV_BF16, head_dim, group) &&
      !pkv::decode_mma_supported(dtype == PKV_BF16, head_dim, group))
    return PKV_EUNSUPPORTED;
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_abi_version(void) { return 2; }

}  // extern "C"

namespace {
// the span record of later side-by-side calls (pkv_set_span_buffer)
std::atomic<unsigned long long*> g_span_buf{nullptr};
}  // namespace

extern "C" {

pkv_status pkv_set_span_buffer(unsigned long long* buf) {
  if (reinterpret_cast<uintptr_t>(buf) & 7u) return PKV_EINVAL;
  g_span_buf.store(buf);
  return PKV_OK;
}

const char* pkv_status_str(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument";
    case PKV_EDTYPE: return "unknown dtype";
    case PKV_ERANGE: return "size out of range";
    case PKV_ECUDA: return "CUDA runtime error";
    case PKV_EUNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

pkv_status pkv_get_device_error(int* code, int clear) {
  if (!code) return PKV_EINVAL;
  int* err = nullptr;
  int sms = 0;
  pkv_status st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ECUDA;
  if (cudaMemcpy(code, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ECUDA;
  if (clear && cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return PKV_ECUDA;
  return PKV_OK;
}

pkv_status pkv_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                         int num_kv_heads, int head_dim, int block_size, pkv_dtype dtype,
                         pkv_stream_t stream) {
  if (!dtype_ok(dtype)) return PKV_EDTYPE;
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1)
    return PKV_EINVAL;
  if (block_size != pkv::kBlockSize) return PKV_EUNSUPPORTED;
  const int row_bytes = head_dim * elem_bytes(dtype);
  if (row_bytes % 16 != 0) return PKV_EUNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_EINVAL;
  int* err = nullptr;
  int sms = 0;
  pkv_status st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  pkv::AppendArgs a{k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
                    num_kv_heads, row_bytes, err};
  return pkv::launch_kv_append(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ECUDA;
}

size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_seq_len) {
  if (num_seqs < 1 || num_q_heads < 1 || head_dim < 1 || max_seq_len < 1) return 0;
  const int s = partial_slots_for(max_seq_len);
  if (s <= 1) return 0;
  const size_t rows = (size_t)num_seqs * num_q_heads * s;
  return align256(rows * head_dim * sizeof(float)) + align256(rows * 2 * sizeof(float)) +
         align256((size_t)num_seqs * num_q_heads * sizeof(int));
}

}  // extern "C"

namespace {

// Shared by paged_decode_attention and its fused-append form (k_new != null).
// Validates a decode call and fills its launch arguments; launches nothing.
pkv_status decode_prepare(pkv::DecodeArgs* out_args, int* out_sms, void* out, const void* q,
                          const void* k_new, const void* v_new, const void* k_cache,
                          const void* v_cache, const int32_t* block_table,
                          const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
                          int max_seq_len, int64_t num_blocks, int num_q_heads, int num_kv_heads,
                          int head_dim, int block_size, float scale, void* workspace,
                          size_t workspace_bytes, pkv_dtype dtype) {
  pkv_status st = check_heads(num_q_heads, num_kv_heads, head_dim, block_size, dtype);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_blocks_per_seq < 1 || max_seq_len < 1 || num_blocks < 1)
    return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > PKV_MAX_SEQS) return PKV_ERANGE;
  if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * block_size) return PKV_EINVAL;
  if (!isfinite(scale)) return PKV_EINVAL;
  if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PKV_EINVAL;
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len);
  if (workspace_bytes < need) return PKV_ERANGE;
  if ((int64_t)num_seqs * num_kv_heads * max_splits_for(max_seq_len) >= (int64_t)INT_MAX)
    return PKV_ERANGE;  // the kernels' unit list is indexed by int
  if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))) return PKV_EINVAL;
  int* err = nullptr;
  int sms = 0;
  st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  const int s = partial_slots_for(max_seq_len);
  const Partials part = carve_partials(workspace, (size_t)num_seqs * num_q_heads * s, head_dim);
  pkv::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.ws_acc = need ? part.acc : nullptr;
  a.ws_ml = need ? part.ml : nullptr;
  a.ws_np = need ? part.np : nullptr;
  a.err = err;
  a.num_seqs = num_seqs;
  a.bt_stride = max_blocks_per_seq;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.max_splits = s;
  a.split_tokens = pkv::kSplitTokens;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.chunk_prior = -1;
  a.is_bf16 = dtype == PKV_BF16;
  a.k_new = k_new;
  a.v_new = v_new;
  *out_args = a;
  *out_sms = sms;
  return PKV_OK;
}

// Launches a prepared decode; sm_budget bounds its persistent grid, and
// dependent launches it as the programmatic dependent of the stream's
// previous kernel (tensor-core path only).
pkv_status decode_launch(const pkv::DecodeArgs& a, int sm_budget, bool dependent,
                         cudaStream_t s_) {
  if (a.num_seqs == 0) return PKV_OK;   // nothing was prepared: an empty batch
  const cudaError_t e =
      pkv::decode_mma_supported(a.is_bf16, a.head_dim, a.num_q_heads / a.num_kv_heads)
          ? pkv::launch_paged_decode_mma(a, sm_budget, s_, dependent)
          : pkv::launch_paged_decode(a, sm_budget, s_);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

pkv_status decode_impl(void* out, const void* q, const void* k_new, const void* v_new,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
                       int max_seq_len, int64_t num_blocks, int num_q_heads, int num_kv_heads,
                       int head_dim, int block_size, float scale, void* workspace,
                       size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream) {
  pkv::DecodeArgs a{};
  int sms = 0;
  const pkv_status st = decode_prepare(&a, &sms, out, q, k_new, v_new, k_cache, v_cache,
                                       block_table, seq_lens, num_seqs, max_blocks_per_seq,
                                       max_seq_len, num_blocks, num_q_heads, num_kv_heads,
                                       head_dim, block_size, scale, workspace, workspace_bytes,
                                       dtype);
  if (st != PKV_OK) return st;
  return decode_launch(a, sms, false, reinterpret_cast<cudaStream_t>(stream));
}

// Validates a chunked-prefill call; launches nothing.
pkv_status prefill_check(const void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table_row, int max_blocks, int prior_len,
                         int chunk_len, int64_t num_blocks, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, float scale, pkv_dtype dtype) {
  pkv_status st = check_heads(num_q_heads, num_kv_heads, head_dim, block_size, dtype);
  if (st != PKV_OK) return st;
  if (max_blocks < 1 || prior_len < 0 || chunk_len < 0 || num_blocks < 1) return PKV_EINVAL;
  if (chunk_len == 0) return PKV_OK;
  if ((int64_t)prior_len + chunk_len > (int64_t)max_blocks * block_size) return PKV_EINVAL;
  if (!isfinite(scale)) return PKV_EINVAL;
  if (!out || !q || !k_cache || !v_cache || !block_table_row) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_table_row) & 3u))
    return PKV_EINVAL;
  if (!(dtype == PKV_BF16 && head_dim == 128) && chunk_len > PKV_MAX_SEQS) return PKV_ERANGE;
  return PKV_OK;
}

// Launches a checked chunked prefill (chunk_len > 0).  persistent_ctas > 0
// asks the two-head tensor-core kernel for that many persistent CTAs.
pkv_status prefill_launch(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table_row, int max_blocks, int prior_len,
                          int chunk_len, int64_t num_blocks, int num_q_heads, int num_kv_heads,
                          int head_dim, float scale, pkv_dtype dtype, int persistent_ctas,
                          cudaStream_t s) {
  int* err = nullptr;
  int sms = 0;
  pkv_status st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  if (dtype == PKV_BF16 && head_dim == 128) {
    pkv::PrefillArgs a{out, q, k_cache, v_cache, block_table_row, max_blocks, prior_len, chunk_len,
                       num_blocks, num_q_heads, num_kv_heads, scale, err};
    return pkv::launch_prefill_pair(a, s, persistent_ctas) == cudaSuccess ? PKV_OK : PKV_ECUDA;
  }
  // CUDA-core path: every chunk row is one query over its causal prefix, run
  // as a single split so no workspace is needed.
  const int total = prior_len + chunk_len;
  pkv::DecodeArgs a{};
  a.out = const_cast<void*>(out);
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table_row;
  a.seq_lens = nullptr;
  a.err = err;
  a.num_seqs = chunk_len;
  a.bt_stride = 0;
  a.max_blocks_per_seq = max_blocks;
  a.max_seq_len = total;
  a.max_splits = 1;
  a.split_tokens = ((total + pkv::kSplitTokens - 1) / pkv::kSplitTokens) * pkv::kSplitTokens;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.chunk_prior = prior_len;
  a.is_bf16 = dtype == PKV_BF16;
  return pkv::launch_paged_decode(a, sms, s) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_decode_attention(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_table,
                                      const int32_t* seq_lens, int num_seqs,
                                      int max_blocks_per_seq, int max_seq_len,
                                      int64_t num_blocks, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, float scale,
                                      void* workspace, size_t workspace_bytes, pkv_dtype dtype,
                                      pkv_stream_t stream) {
  return decode_impl(out, q, nullptr, nullptr, k_cache, v_cache, block_table, seq_lens, num_seqs,
                     max_blocks_per_seq, max_seq_len, num_blocks, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, workspace, workspace_bytes, dtype, stream);
}

pkv_status pkv_paged_decode_attention_append(void* out, const void* q, const void* k_new,
                                             const void* v_new, void* k_cache, void* v_cache,
                                             const int32_t* block_table, const int32_t* seq_lens,
                                             int num_seqs, int max_blocks_per_seq,
                                             int max_seq_len, int64_t num_blocks,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int block_size, float scale, void* workspace,
                                             size_t workspace_bytes, pkv_dtype dtype,
                                             pkv_stream_t stream) {
  if (!dtype_ok(dtype)) return PKV_EDTYPE;
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (!pkv::decode_mma_supported(dtype == PKV_BF16, head_dim, num_q_heads / num_kv_heads))
    return PKV_EUNSUPPORTED;
  if (num_seqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
    return PKV_EINVAL;
  return decode_impl(out, q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, num_seqs,
                     max_blocks_per_seq, max_seq_len, num_blocks, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, workspace, workspace_bytes, dtype, stream);
}

pkv_status pkv_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const float* k_scale, const float* v_scale,
                             const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                             int num_kv_heads, int head_dim, int block_size, pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1)
    return PKV_EINVAL;
  if (block_size != pkv::kBlockSize || head_dim % 16 != 0) return PKV_EUNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
    return PKV_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return PKV_EINVAL;
  int* err = nullptr;
  int sms = 0;
  pkv_status st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  pkv::AppendFp8Args a{k_new, v_new, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                       num_tokens, num_blocks, num_kv_heads, head_dim, err};
  return pkv::launch_kv_append_fp8(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ECUDA;
}

pkv_status pkv_paged_decode_attention_fp8(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const float* k_scale,
                                          const float* v_scale, const int32_t* block_table,
                                          const int32_t* seq_lens, int num_seqs,
                                          int max_blocks_per_seq, int max_seq_len,
                                          int64_t num_blocks, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, float scale,
                                          void* workspace, size_t workspace_bytes,
                                          pkv_stream_t stream) {
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || head_dim < 1 ||
      block_size < 1)
    return PKV_EINVAL;
  if (block_size != pkv::kBlockSize ||
      !pkv::decode_mma_supported(1, head_dim, num_q_heads / num_kv_heads))
    return PKV_EUNSUPPORTED;
  if (num_seqs < 0 || max_blocks_per_seq < 1 || max_seq_len < 1 || num_blocks < 1)
    return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > PKV_MAX_SEQS) return PKV_ERANGE;
  if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * block_size) return PKV_EINVAL;
  if (!isfinite(scale)) return PKV_EINVAL;
  if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens || !k_scale || !v_scale)
    return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return PKV_EINVAL;
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len);
  if (workspace_bytes < need) return PKV_ERANGE;
  if ((int64_t)num_seqs * num_kv_heads * max_splits_for(max_seq_len) >= (int64_t)INT_MAX)
    return PKV_ERANGE;  // the kernels' unit list is indexed by int
  if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))) return PKV_EINVAL;
  int* err = nullptr;
  int sms = 0;
  pkv_status st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  const int s = partial_slots_for(max_seq_len);
  const Partials part = carve_partials(workspace, (size_t)num_seqs * num_q_heads * s, head_dim);
  pkv::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.ws_acc = need ? part.acc : nullptr;
  a.ws_ml = need ? part.ml : nullptr;
  a.ws_np = need ? part.np : nullptr;
  a.err = err;
  a.num_seqs = num_seqs;
  a.bt_stride = max_blocks_per_seq;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.max_splits = s;
  a.split_tokens = pkv::kSplitTokens;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.chunk_prior = -1;
  a.is_bf16 = 1;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return pkv::launch_paged_decode_fp8(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ECUDA;
}

pkv_status pkv_latent_append(const void* c_new, void* c_cache, const int64_t* slot_mapping,
                             int64_t num_tokens, int64_t num_blocks, int rank, int block_size,
                             pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || rank < 1 || block_size < 1) return PKV_EINVAL;
  if (block_size != pkv::kBlockSize || (rank * 2) % 16 != 0) return PKV_EUNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!c_new || !c_cache || !slot_mapping) return PKV_EINVAL;
  if (!aligned16(c_new) || !aligned16(c_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_EINVAL;
  int* err = nullptr;
  int sms = 0;
  pkv_status st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  pkv::AppendArgs a{c_new, nullptr, c_cache, nullptr, slot_mapping, num_tokens, num_blocks, 1,
                    rank * 2, err};
  return pkv::launch_kv_append(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ECUDA;
}

size_t pkv_mla_workspace_bytes(int num_seqs, int num_q_heads, int rank, int max_seq_len) {
  if (num_seqs < 1 || num_q_heads < 1 || rank < 1 || max_seq_len < 1) return 0;
  const size_t vec = align256((size_t)num_seqs * num_q_heads * rank * 2);
  return 2 * vec + pkv_decode_workspace_bytes(num_seqs, num_q_heads, rank, max_seq_len);
}

}  // extern "C"

namespace {

// The latent decode call; c_new (optional): each sequence's new latent,
// appended by the query absorption's launch.
pkv_status mla_decode(void* out, const void* q, const void* c_new, const void* w_k,
                      const void* w_v, void* c_cache, const int32_t* block_table,
                      const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
                      int max_seq_len, int64_t num_blocks, int num_q_heads, int head_dim, int rank,
                      int block_size, float scale, void* workspace, size_t workspace_bytes,
                      pkv_stream_t stream) {
  if (num_q_heads < 1 || head_dim < 1 || rank < 1 || block_size < 1) return PKV_EINVAL;
  if (block_size != pkv::kBlockSize || num_q_heads != 32 || head_dim != 128 || rank != 128)
    return PKV_EUNSUPPORTED;
  if (num_seqs < 0 || max_blocks_per_seq < 1 || max_seq_len < 1 || num_blocks < 1) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > PKV_MAX_SEQS) return PKV_ERANGE;
  if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * block_size) return PKV_EINVAL;
  if (!isfinite(scale)) return PKV_EINVAL;
  if (!out || !q || !w_k || !w_v || !c_cache || !block_table || !seq_lens || !workspace)
    return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(w_k) || !aligned16(w_v) ||
      !aligned16(c_cache) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_EINVAL;
  if (workspace_bytes < pkv_mla_workspace_bytes(num_seqs, num_q_heads, rank, max_seq_len))
    return PKV_ERANGE;
  if ((int64_t)num_seqs * max_splits_for(max_seq_len) >= (int64_t)INT_MAX)
    return PKV_ERANGE;  // the kernel's unit list is indexed by int
  int* err = nullptr;
  int sms = 0;
  pkv_status st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t vec = align256((size_t)num_seqs * num_q_heads * rank * 2);
  char* ws = static_cast<char*>(workspace);
  void* q_lat = ws;          // absorbed queries [B][Hq][rank] bf16
  void* z = ws + vec;        // attention over the latent [B][Hq][rank] bf16
  char* part = ws + 2 * vec;
  // 1) q~_h = W_K[h]^T q_h (and, given c_new, each sequence's new latent
  //    placed at position seq_lens[b] - 1)
  const pkv::LatentAppend app{c_new, c_cache, block_table, seq_lens, max_blocks_per_seq,
                              (int)std::min<int64_t>(max_seq_len,
                                                     (int64_t)max_blocks_per_seq * block_size),
                              num_blocks, err};
  if (pkv::launch_gemm_heads(q_lat, q, w_k, num_seqs, num_q_heads, s, c_new ? &app : nullptr) !=
      cudaSuccess)
    return PKV_ECUDA;
  // 2) z_h = softmax(scale q~_h . C^T) C over the latent pool
  const int splits = partial_slots_for(max_seq_len);
  const Partials pp = carve_partials(part, (size_t)num_seqs * num_q_heads * splits, rank);
  pkv::DecodeArgs a{};
  a.out = z;
  a.q = q_lat;
  a.k_cache = c_cache;
  a.v_cache = c_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.ws_acc = pp.acc;
  a.ws_ml = pp.ml;
  a.ws_np = splits > 1 ? pp.np : nullptr;
  a.err = err;
  a.num_seqs = num_seqs;
  a.bt_stride = max_blocks_per_seq;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.max_splits = splits;
  a.split_tokens = pkv::kSplitTokens;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = 1;
  a.head_dim = rank;
  a.scale = scale;
  a.chunk_prior = -1;
  a.is_bf16 = 1;
  // 3) merge of the partials fused with o_h = W_V[h] z_h
  if (pkv::launch_decode_mla(a, w_v, out, sms, s) != cudaSuccess) return PKV_ECUDA;
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_mla_decode_attention(void* out, const void* q, const void* w_k, const void* w_v,
                                    const void* c_cache, const int32_t* block_table,
                                    const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
                                    int max_seq_len, int64_t num_blocks, int num_q_heads,
                                    int head_dim, int rank, int block_size, float scale,
                                    void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  return mla_decode(out, q, nullptr, w_k, w_v, const_cast<void*>(c_cache), block_table, seq_lens,
                    num_seqs, max_blocks_per_seq, max_seq_len, num_blocks, num_q_heads, head_dim,
                    rank, block_size, scale, workspace, workspace_bytes, stream);
}

pkv_status pkv_mla_decode_attention_append(void* out, const void* q, const void* c_new,
                                           const void* w_k, const void* w_v, void* c_cache,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           int num_seqs, int max_blocks_per_seq, int max_seq_len,
                                           int64_t num_blocks, int num_q_heads, int head_dim,
                                           int rank, int block_size, float scale, void* workspace,
                                           size_t workspace_bytes, pkv_stream_t stream) {
  if (num_seqs > 0 && (!c_new || !aligned16(c_new))) return PKV_EINVAL;
  return mla_decode(out, q, c_new, w_k, w_v, c_cache, block_table, seq_lens, num_seqs,
                    max_blocks_per_seq, max_seq_len, num_blocks, num_q_heads, head_dim, rank,
                    block_size, scale, workspace, workspace_bytes, stream);
}

pkv_status pkv_chunked_prefill_attention(void* out, const void* q, const void* k_cache,
                                         const void* v_cache, const int32_t* block_table_row,
                                         int max_blocks, int prior_len, int chunk_len,
                                         int64_t num_blocks, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, float scale,
                                         pkv_dtype dtype, pkv_stream_t stream) {
  pkv_status st = prefill_check(out, q, k_cache, v_cache, block_table_row, max_blocks, prior_len,
                                chunk_len, num_blocks, num_q_heads, num_kv_heads, head_dim,
                                block_size, scale, dtype);
  if (st != PKV_OK || chunk_len == 0) return st;
  return prefill_launch(out, q, k_cache, v_cache, block_table_row, max_blocks, prior_len, chunk_len,
                        num_blocks, num_q_heads, num_kv_heads, head_dim, scale, dtype, 0,
                        reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_decode_prefill_attention(const pkv_decode_prefill_args* x, pkv_stream_t stream) {
  if (!x) return PKV_EINVAL;
  // validate both halves before anything is launched
  if (!dtype_ok(x->dtype)) return PKV_EDTYPE;
  if (x->num_q_heads < 1 || x->num_kv_heads < 1 || x->num_q_heads % x->num_kv_heads != 0)
    return PKV_EINVAL;
  if (!pkv::decode_mma_supported(x->dtype == PKV_BF16, x->head_dim,
                                 x->num_q_heads / x->num_kv_heads))
    return PKV_EUNSUPPORTED;
  if (x->num_seqs > 0 && (!x->k_new || !x->v_new || !aligned16(x->k_new) || !aligned16(x->v_new)))
    return PKV_EINVAL;
  pkv::DecodeArgs d{};
  int sms = 0;
  pkv_status st = decode_prepare(&d, &sms, x->decode_out, x->decode_q, x->k_new, x->v_new,
                                 x->k_cache, x->v_cache, x->block_table, x->seq_lens, x->num_seqs,
                                 x->max_blocks_per_seq, x->max_seq_len, x->num_blocks,
                                 x->num_q_heads, x->num_kv_heads, x->head_dim, x->block_size,
                                 x->scale, x->workspace, x->workspace_bytes, x->dtype);
  if (st != PKV_OK) return st;
  st = prefill_check(x->prefill_out, x->prefill_q, x->k_cache, x->v_cache, x->prefill_block_table,
                     x->prefill_max_blocks, x->prior_len, x->chunk_len, x->num_blocks,
                     x->num_q_heads, x->num_kv_heads, x->head_dim, x->block_size, x->scale,
                     x->dtype);
  if (st != PKV_OK) return st;
  if (x->prefill_sms < 0) return PKV_EINVAL;
  // the chunk's own keys and values: all three pointers or none
  const bool chunk_append = x->chunk_k_new || x->chunk_v_new || x->chunk_slot_mapping;
  if (chunk_append && x->chunk_len > 0 &&
      (!x->chunk_k_new || !x->chunk_v_new || !x->chunk_slot_mapping || !aligned16(x->chunk_k_new) ||
       !aligned16(x->chunk_v_new) || (reinterpret_cast<uintptr_t>(x->chunk_slot_mapping) & 7u)))
    return PKV_EINVAL;
  int* err = nullptr;
  st = device_state(&err, &sms);
  if (st != PKV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (chunk_append && x->chunk_len > 0) {
    // the chunk's rows first; the prefill (launched next, not as a
    // programmatic dependent) reads them
    pkv::AppendArgs ap{x->chunk_k_new, x->chunk_v_new, x->k_cache, x->v_cache,
                       x->chunk_slot_mapping, x->chunk_len, x->num_blocks, x->num_kv_heads,
                       x->head_dim * elem_bytes(x->dtype), err};
    if (pkv::launch_kv_append(ap, s) != cudaSuccess) return PKV_ECUDA;
  }
  const int p_sms = x->prefill_sms > 0 ? x->prefill_sms : sms / 4;
  pkv::PrefillArgs pa{x->prefill_out, x->prefill_q, x->k_cache, x->v_cache, x->prefill_block_table,
                      x->prefill_max_blocks, x->prior_len, x->chunk_len, x->num_blocks,
                      x->num_q_heads, x->num_kv_heads, x->scale, err};
  if (unsigned long long* span = g_span_buf.load()) {
    pa.span = span;
    d.span = span + 2;
  }
  const bool side_by_side = x->chunk_len > 0 && d.num_seqs > 0 && x->head_dim == 128 &&
                            x->dtype == PKV_BF16 && p_sms < sms &&
                            pkv::prefill_pair_persistent_ok(pa, p_sms);
  if (!side_by_side) {   // one after the other, each on the whole GPU
    if (x->chunk_len > 0) {
      st = prefill_launch(x->prefill_out, x->prefill_q, x->k_cache, x->v_cache,
                          x->prefill_block_table, x->prefill_max_blocks, x->prior_len,
                          x->chunk_len, x->num_blocks, x->num_q_heads, x->num_kv_heads,
                          x->head_dim, x->scale, x->dtype, 0, s);
      if (st != PKV_OK) return st;
    }
    return decode_launch(d, sms, false, s);
  }
  // the prefill's persistent CTAs take p_sms SMs; the decode, launched as its
  // programmatic dependent, runs on the others and finishes after it.  (The
  // prefill launched as the programmatic dependent of the chunk's append,
  // its gathers waiting for that grid, measured 20% slower per layer.)
  if (pkv::launch_prefill_pair(pa, s, p_sms) != cudaSuccess) return PKV_ECUDA;
  return decode_launch(d, sms - p_sms, true, s);
}

}  // extern "C"
