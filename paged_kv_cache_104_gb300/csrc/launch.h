// Internal launchers: one per kernel family, called by the C ABI layer
// (abi.cu) after it has validated every host-side argument.  Each returns a
// cudaError_t from the launch.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

constexpr int kBlockSize = 16;     // tokens per cache block (compiled)
constexpr int kSplitTokens = 512;  // decode tokens per split-K unit

struct AppendArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int64_t num_blocks;
  int num_kv_heads;
  int row_bytes;  // head_dim * element size
  int* err;
};
cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream);
// bf16 rows -> fp8 E4M3 codes of x / scale[head] (head_dim a multiple of 16)
struct AppendFp8Args {
  const void* k_new;   // bf16 [T][Hkv][D]
  const void* v_new;
  void* k_cache;       // uint8 [NB][Hkv][16][D]
  void* v_cache;
  const float* k_scale;  // [Hkv]
  const float* v_scale;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int64_t num_blocks;
  int num_kv_heads;
  int head_dim;
  int* err;
};
cudaError_t launch_kv_append_fp8(const AppendFp8Args& a, cudaStream_t stream);

struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* seq_lens;  // may be null in chunk mode
  float* ws_acc;            // [B][Hq][max_splits][D] fp32 (unused if max_splits == 1)
  float* ws_ml;             // [B][Hq][max_splits][2] fp32
  int* ws_np;               // [B][Hkv] partials per (sequence, KV head) (balanced walk)
  int* err;
  int num_seqs;
  int bt_stride;            // elements between block-table rows (0: all rows share one)
  int max_blocks_per_seq;
  int max_seq_len;          // host bound on every sequence length
  int max_splits;           // partial slots per row (>= partials of any row)
  int split_tokens;
  int64_t num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  float scale;
  int chunk_prior;          // -1: decode; >= 0: row b has length chunk_prior + b + 1
  int is_bf16;
  // fused append (decode_mma only): each sequence's new key/value [B][Hkv][D],
  // written at position seq_lens[b] - 1 before attending; null = no append
  const void* k_new;
  const void* v_new;
  // fp8 cache only: per-KV-head dequantisation scales [Hkv]
  const float* k_scale;
  const float* v_scale;
  // 1: the main kernel stores split partials with an L2 evict-last hint and
  // the merge drops each partial line from L2 once read (no write-back);
  // 0: plain stores.  Set by the bf16 decode launcher, except for per-head
  // stages beside a prefill, whose re-read K/V lives in L2: there the many
  // partials of 512-token splits made plain stores faster.
  int keep_partials;
  // 1: the balanced walk of the bf16, fp8 and latent decodes (set by their
  // launchers when ws_np is given and the decode runs alone, or, for the bf16
  // decode with grouped stages, also beside a prefill): the stages of all
  // sequences are cut into equal shares, one per CTA, and the main kernel
  // records in ws_np how many partials each (sequence, KV head) left for the
  // merge; 0: 512-token splits, the merge derives their count from seq_lens.
  int balanced;
  // 1: the kernel keeps every sequence's length in shared memory after its
  // unit prefix sums (set by a launcher that sized shared memory for it)
  int lens_in_smem;
  // 1: a split partial is stored as O / l in fp16 (head_dim 128: 256 B a
  // row, half the bytes of fp32 O) beside its fp32 (m, l); set by the bf16
  // and fp8 tensor-core decodes, whose outputs are bf16.  0: fp32 O.
  int partials_f16;
  // optional span record (the bf16 decode's main kernel): {earliest CTA
  // start, latest CTA end} in %globaltimer ns, by atomic min / max
  unsigned long long* span;
};
// True if (dtype, head_dim, group) has a compiled decode kernel.
bool decode_supported(int is_bf16, int head_dim, int group);
cudaError_t launch_paged_decode(const DecodeArgs& a, int num_sms, cudaStream_t stream);
// Tensor-core (mma.sync) decode for bf16, head_dim 128, group in {1,2,4,8,16};
// decode mode only (chunk_prior < 0).  Launches the split reduce when needed.
bool decode_mma_supported(int is_bf16, int head_dim, int group);
// dependent: launch as the programmatic dependent of the previous kernel in
// the stream (see launch_prefill_pair); the grid then also waits, at its end,
// for that kernel to complete.  num_sms bounds the persistent grid.
cudaError_t launch_paged_decode_mma(const DecodeArgs& a, int num_sms, cudaStream_t stream,
                                    bool dependent = false);
// fp8 (E4M3) cache, bf16 q/out, head_dim 128, group in {1,2,4,8,16}; uses
// DecodeArgs with k_scale / v_scale set.
cudaError_t launch_paged_decode_fp8(const DecodeArgs& a, int num_sms, cudaStream_t stream);
// Attention over a latent (MLA-style) cache and the output projection: one
// pool of rank-128 latents, 32 query heads, q already absorbed into a.q;
// a.k_cache is the latent pool, a.out receives z for sequences covered in one
// piece (the others leave partials); then the merge + up-projection writes
// o = W_V z into `out`.  The attention is launched as the programmatic
// dependent of the kernel before it in the stream (the query absorption),
// and waits for it before reading a.q or any latent.
cudaError_t launch_decode_mla(const DecodeArgs& a, const void* w_v, void* out, int num_sms,
                              cudaStream_t stream);
// The latent of each decode sequence's new token, placed by the query
// absorption's launch at position seq_lens[r] - 1 of row r's block table
// (rank 128, bf16, pool [num_blocks][16][128]).
struct LatentAppend {
  const void* c_new;        // [rows][128]
  void* c_cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int bt_stride;
  int max_len;              // lengths outside [1, max_len] are skipped
  int64_t num_blocks;
  int* err;
};
// y[r][h] = x[r][h] . W[h] (W[h] 128 x 128 bf16, stored [K][N]), bf16 in and
// out; with app set, the same launch also appends each row's new latent.
// Each CTA signals at its start that a programmatic dependent launch may
// begin.
cudaError_t launch_gemm_heads(void* y, const void* x, const void* w, int rows, int heads,
                              cudaStream_t stream, const LatentAppend* app = nullptr);
// The latent attention's merge of split partials fused with the output
// up-projection o_h = W_V[h] z_h (launched as the attention's programmatic
// dependent).
cudaError_t launch_merge_project(const DecodeArgs& a, const void* w_v, void* out,
                                 cudaStream_t stream);
// Merge of split partials for bf16 / head_dim 128 (used by the mma decode).
cudaError_t launch_decode_reduce_bf16_128(const DecodeArgs& a, cudaStream_t stream);

struct PrefillArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table_row;
  int max_blocks;
  int prior_len;
  int chunk_len;
  int64_t num_blocks;
  int num_q_heads;
  int num_kv_heads;
  float scale;
  int* err;
  // optional span record, as DecodeArgs::span (the tcgen05 prefill)
  unsigned long long* span = nullptr;
};
// tcgen05 path (bf16, head_dim 128, block_size 16): two streams of 128 query
// rows per CTA sharing each K/V tile -- two query heads of one KV head when
// the GQA group is even, else two consecutive query tiles of one head.
// persistent_ctas > 0: that many persistent CTAs run the work items (query
// tile x head pair), assigned longest first, and each signals at its start
// that a programmatically dependent launch may begin (so a kernel launched
// next with that attribute runs on the remaining SMs); 0: one CTA per item.
bool prefill_pair_persistent_ok(const PrefillArgs& a, int ctas);
cudaError_t launch_prefill_pair(const PrefillArgs& a, cudaStream_t stream, int persistent_ctas = 0);

}  // namespace pkv
