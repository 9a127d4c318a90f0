/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library
 * (libpagedkv.so).
 *
 * The library implements the per-step attention of continuous batching over
 * a block-paged KV cache:
 *   - kv_append: write each running sequence's new key and value into the
 *     cache ("KV cache and continuous batching: 1,000 people ask AI", section
 *     "What does a KV cache keep?"; "The KV cache and prefix caching",
 *     section "What prefill stores and decode reads": a decode step appends
 *     the new key and value to the cache);
 *   - paged_decode_attention: attend each sequence's new query over every
 *     key and value it has stored, under grouped-query attention, across a
 *     ragged batch (same sections; the cache is held in fixed-size blocks
 *     reached through a per-sequence block table, the PagedAttention layout);
 *   - chunked_prefill_attention: a capped chunk of prompt tokens attends
 *     causally over itself and the sequence's earlier cache ("The KV cache is
 *     not your bottleneck", section "The fix that mattered").
 *
 * Conventions shared by every call
 *   Layouts (row-major, element type given by `dtype`):
 *     k_cache, v_cache   [num_blocks][num_kv_heads][block_size][head_dim]
 *     block_table        int32 [num_seqs][max_blocks_per_seq]; entry j of a
 *                        row is the physical block holding the sequence's
 *                        tokens j*block_size .. j*block_size+block_size-1
 *     slot_mapping       int64, slot = physical_block*block_size + row
 *     q, out (decode)    [num_seqs][num_q_heads][head_dim]
 *     q, out (prefill)   [chunk_len][num_q_heads][head_dim]
 *   Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   seq_lens counts the tokens stored after this step's append, so each new
 *   query attends over its own key as well.
 *   Memory: every pointer except those named "host" is a device pointer the
 *   caller owns; the library allocates no memory and keeps no state between
 *   calls other than a per-device error word (and the scratch array of
 *   pkv_paged_decode_attention_noalloc).  Pointers must be 16-byte aligned.
 *   Streams: work is enqueued on `stream` (NULL = the legacy default stream)
 *   and the call returns without synchronising.
 *   Errors: argument errors are found on the host and returned before any
 *   launch.  Values that live in device memory (slots, block ids, sequence
 *   lengths) are checked by the kernels: an offending entry is skipped (no
 *   out-of-bounds access happens), its outputs are unspecified, and a code
 *   is recorded in the device error word (pkv_get_device_error).  Kernels
 *   never trap; every internal wait is bounded.
 *   Supported shapes: block_size 16; bf16 with head_dim 128, or fp32 with
 *   head_dim 16 or 128; num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 *   The library runs on sm_103 GPUs (GB300).
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = 1,       /* null pointer, negative size, misaligned pointer, inconsistent shape */
  PKV_EDTYPE = 2,       /* dtype not one of pkv_dtype */
  PKV_ERANGE = 3,       /* a size beyond a limit (workspace too small, too many sequences) */
  PKV_ECUDA = 4,        /* the CUDA runtime reported an error at launch */
  PKV_EUNSUPPORTED = 5  /* a shape this build has no kernel for */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Device error word values (pkv_get_device_error). */
#define PKV_DEVERR_NONE 0
#define PKV_DEVERR_SLOT_RANGE 1   /* kv_append: slot >= num_blocks*block_size (entry skipped) */
#define PKV_DEVERR_BLOCK_RANGE 2  /* block-table entry outside [0, num_blocks) (block 0 read instead) */
#define PKV_DEVERR_SEQLEN_RANGE 3 /* sequence length < 1 or beyond its bound (sequence skipped) */
#define PKV_DEVERR_TIMEOUT 4      /* an internal wait ran out of time (results unspecified) */
#define PKV_DEVERR_SMEM_LAYOUT 5  /* shared memory not laid out as a kernel needs (call skipped) */

/* Largest num_seqs accepted by paged_decode_attention. */
#define PKV_MAX_SEQS 8192

/*
 * kv_append -- write new keys and values into the paged pools (bit-exact copy).
 *   k_new, v_new   [num_tokens][num_kv_heads][head_dim], device, read
 *   k_cache, v_cache  pools, device, written in place at the given slots only
 *   slot_mapping   int64 [num_tokens], device; slot < 0 means padding (skipped)
 *   num_tokens >= 0 (0: no-op), num_blocks >= 1
 * Slots must be distinct; two tokens writing one slot leave either row there.
 */
pkv_status pkv_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t num_tokens, int64_t num_blocks,
                         int num_kv_heads, int head_dim, int block_size, pkv_dtype dtype,
                         pkv_stream_t stream);

/*
 * Bytes of device workspace paged_decode_attention needs for these sizes
 * (0 when no sequence can need more than one split, max_seq_len <= 512).
 * Otherwise: room for fp32 partials of ceil(max_seq_len / 512) + 1 slots
 * per (sequence, query head) row, each head_dim values plus a (max, sum)
 * pair, and one int per row for the partial count (the bf16 and fp8
 * tensor-core decodes store their partials as fp16 in half of that room).
 * Host-only, no GPU use.  The
 * workspace holds no state between calls: every value a call reads there it
 * wrote earlier in the same call, so it needs no clearing.
 */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_seq_len);

/*
 * paged_decode_attention -- one new query per sequence over its whole cache.
 *   out    [num_seqs][num_q_heads][head_dim], device, written
 *   q      [num_seqs][num_q_heads][head_dim], device, read
 *   block_table  int32 [num_seqs][max_blocks_per_seq], device
 *   seq_lens     int32 [num_seqs], device; 1 <= seq_lens[b] <= max_seq_len
 *   max_seq_len  host bound on every seq_lens entry (sizes the split grid)
 *   scale        softmax scale (usually 1/sqrt(head_dim))
 *   workspace    device scratch of at least pkv_decode_workspace_bytes(...)
 *                bytes (may be NULL when that is 0); overwritten
 *   1 <= num_seqs <= PKV_MAX_SEQS; max_seq_len <= max_blocks_per_seq*block_size
 * Output: out[b][h] = sum_j softmax_j(scale * q[b][h].k_j) v_j over the
 * seq_lens[b] stored tokens j of sequence b and KV head h/(Hq/Hkv), rounded
 * to the storage type.
 */
pkv_status pkv_paged_decode_attention(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_table,
                                      const int32_t *seq_lens, int num_seqs,
                                      int max_blocks_per_seq, int max_seq_len,
                                      int64_t num_blocks, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, float scale,
                                      void *workspace, size_t workspace_bytes, pkv_dtype dtype,
                                      pkv_stream_t stream);

/*
 * paged_decode_attention_append -- kv_append of each sequence's new token
 * fused into paged_decode_attention ("KV cache and continuous batching:
 * 1,000 people ask AI", section "What does a KV cache keep?": a decode step
 * appends the new key and value, then attends over everything stored).
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim], device: the new token of
 *                 sequence b, written at position seq_lens[b] - 1, i.e. into
 *                 physical block block_table[b][(seq_lens[b]-1)/block_size],
 *                 row (seq_lens[b]-1) % block_size, of both pools
 *   every other argument as for pkv_paged_decode_attention; the pools are
 *   written (that one row per sequence and KV head) as well as read.
 * Equivalent to pkv_kv_append of those rows followed by
 * pkv_paged_decode_attention, in one launch: the new row is placed into the
 * staged tile in shared memory and stored to the pool by the same CTA.
 * bf16 with head_dim 128 only (PKV_EUNSUPPORTED otherwise).
 */
pkv_status pkv_paged_decode_attention_append(void *out, const void *q, const void *k_new,
                                             const void *v_new, void *k_cache, void *v_cache,
                                             const int32_t *block_table, const int32_t *seq_lens,
                                             int num_seqs, int max_blocks_per_seq,
                                             int max_seq_len, int64_t num_blocks,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int block_size, float scale, void *workspace,
                                             size_t workspace_bytes, pkv_dtype dtype,
                                             pkv_stream_t stream);

/* Size of the scratch buffer pkv_paged_decode_attention_noalloc keeps inside
 * the library (32 MiB; held by every GPU that loads the library until exit). */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * paged_decode_attention_noalloc -- paged_decode_attention for callers that
 * cannot allocate device memory.  The pages have no counterpart to this call.
 *
 * Who needs it: an engine that reserves all device memory in its own pool at
 * start-up and allows no later cudaMalloc (a late allocation can fail under
 * memory pressure, fragment the pool or synchronise the device mid-step), or
 * a plugin interface that hands over only input and output pointers.  Such a
 * caller has no workspace to pass, so this call uses a scratch array that
 * lives in the library itself (PKV_NOALLOC_SCRATCH_BYTES) instead.
 *   Arguments, layouts and results are those of pkv_paged_decode_attention
 *   without workspace / workspace_bytes.  The caller still provides every
 *   input and output buffer.
 *   Returns PKV_ERANGE, before any launch, when
 *   pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len)
 *   exceeds PKV_NOALLOC_SCRATCH_BYTES.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress); make that first call before capturing any stream.
 *   After a device reset (cudaDeviceReset) the array is gone with the old
 *   context; the next call looks the address up again in the new one, so it
 *   too must come before any capture.
 *   All calls share the one array, which keeps the last call's contents (no
 *   part of it needs to start at zero).  Calls whose kernels overlap on the
 *   GPU -- on different streams or from different host threads -- race on it
 *   and produce wrong results; the caller must serialise them.
 */
pkv_status pkv_paged_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *block_table,
                                              const int32_t *seq_lens, int num_seqs,
                                              int max_blocks_per_seq, int max_seq_len,
                                              int64_t num_blocks, int num_q_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              float scale, pkv_dtype dtype, pkv_stream_t stream);

/*
 * chunked_prefill_attention -- a chunk of one sequence's prompt attends
 * causally over itself and the cache before it.
 *   out, q   [chunk_len][num_q_heads][head_dim], device
 *   block_table_row  int32 [max_blocks], device: the sequence's block table
 *   prior_len   tokens the sequence had before this chunk (host value)
 *   chunk_len   tokens in the chunk (host value, >= 0; 0 is a no-op)
 * The chunk's own keys and values must already be in the pools (kv_append
 * first).  Row i sits at position prior_len + i and sees keys
 * 0 .. prior_len + i.  Requires prior_len + chunk_len <= max_blocks*block_size.
 * bf16 with head_dim 128 runs on the tcgen05 tensor cores; other supported
 * shapes run a CUDA-core kernel.
 */
pkv_status pkv_chunked_prefill_attention(void *out, const void *q, const void *k_cache,
                                         const void *v_cache, const int32_t *block_table_row,
                                         int max_blocks, int prior_len, int chunk_len,
                                         int64_t num_blocks, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, float scale,
                                         pkv_dtype dtype, pkv_stream_t stream);

/*
 * decode_prefill_attention -- one layer of a continuous-batching step: the
 * batch's decode (as pkv_paged_decode_attention_append: each sequence's new
 * key/value appended, then one query per sequence over its cache) and one
 * prompt chunk's prefill (as pkv_chunked_prefill_attention), run side by side
 * on disjoint SMs of the GPU.  "The KV cache is not your bottleneck", section
 * "The fix that mattered", admits prompts in capped chunks that share each
 * step with the running decodes; this call gives them the tensor cores of
 * some SMs while the memory-bound decode streams the cache on the rest.
 *   All fields of pkv_decode_prefill_args mean what the same arguments of the
 *   two calls mean (decode_out/decode_q/k_new/v_new/block_table/seq_lens/
 *   num_seqs/max_blocks_per_seq/max_seq_len/workspace for the decode,
 *   prefill_out/prefill_q/prefill_block_table/prefill_max_blocks/prior_len/
 *   chunk_len for the prefill; pools, head counts, sizes, scale and dtype are
 *   shared).  The chunk's sequence must not be one of the decoded sequences.
 *   chunk_k_new, chunk_v_new  the chunk's own new keys and values
 *                [chunk_len][num_kv_heads][head_dim] (16-byte aligned), and
 *   chunk_slot_mapping        their slots (int64 [chunk_len], as for
 *                pkv_kv_append): the call first appends them (bit-exact, as
 *                pkv_kv_append would) and the prefill reads them.  All three
 *                null: the chunk's keys and values must already be in the
 *                pools.
 *   prefill_sms  SMs given to the prefill (0: a quarter of the GPU).  The
 *                best split makes both halves end together; it depends on
 *                the batch (the decode's cache bytes) and the chunk.
 * Results are those of the two calls made one after the other (bit for bit).
 * Both halves are checked before either is launched.  When the prefill
 * cannot run as persistent tensor-core CTAs (not bf16 with head_dim 128, more
 * than 512 work items -- a work item is 128 query rows of two heads of one KV
 * head, or 256 rows of one head when the GQA group is odd -- or prefill_sms
 * not below the SM count), the two run one after the other instead.  bf16
 * with head_dim 128 only for the decode (PKV_EUNSUPPORTED otherwise).
 */
typedef struct pkv_decode_prefill_args {
  void *decode_out;
  const void *decode_q;
  const void *k_new;
  const void *v_new;
  const int32_t *block_table;
  const int32_t *seq_lens;
  int num_seqs;
  int max_blocks_per_seq;
  int max_seq_len;
  void *workspace;
  size_t workspace_bytes;
  void *prefill_out;
  const void *prefill_q;
  const int32_t *prefill_block_table;
  int prefill_max_blocks;
  int prior_len;
  int chunk_len;
  void *k_cache;
  void *v_cache;
  int64_t num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  float scale;
  pkv_dtype dtype;
  int prefill_sms;
  const void *chunk_k_new;
  const void *chunk_v_new;
  const int64_t *chunk_slot_mapping;
} pkv_decode_prefill_args;

pkv_status pkv_decode_prefill_attention(const pkv_decode_prefill_args *args,
                                        pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * fp8 KV cache (E4M3 codes with a float scale per KV head).  "The KV cache is
 * not your bottleneck", section "What the profile said", names cache
 * quantisation; the pages give no format.  This library stores a key or value
 * element x of KV head h as code = E4M3(x / scale[h]) -- the OCP FP8 E4M3
 * format (bias 7, 3 mantissa bits, largest finite 448, no infinity), x/scale
 * computed in fp32, rounded to nearest even, finite values beyond 448 clamped
 * to 448 -- and reads it back as decode(code) * scale[h].  Pools are bytes
 * [num_blocks][num_kv_heads][block_size][head_dim]; scales are device float
 * [num_kv_heads]; new keys/values, q and out are bf16.
 * ------------------------------------------------------------------------- */

/* Quantise and scatter new keys and values (as pkv_kv_append otherwise;
 * head_dim a multiple of 16). */
pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const float *k_scale, const float *v_scale,
                             const int64_t *slot_mapping, int64_t num_tokens, int64_t num_blocks,
                             int num_kv_heads, int head_dim, int block_size, pkv_stream_t stream);

/* Decode attention over the fp8 pools (as pkv_paged_decode_attention with
 * q/out in bf16; head_dim 128; the same workspace size). */
pkv_status pkv_paged_decode_attention_fp8(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const float *k_scale,
                                          const float *v_scale, const int32_t *block_table,
                                          const int32_t *seq_lens, int num_seqs,
                                          int max_blocks_per_seq, int max_seq_len,
                                          int64_t num_blocks, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, float scale,
                                          void *workspace, size_t workspace_bytes,
                                          pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Latent (MLA-style) cache.  "The KV cache and prefix caching", section "What
 * prefill stores and decode reads", names multi-head latent attention: the
 * cache stores a low-rank projection instead of the keys and values.  This
 * library's reading: per token and layer one latent c of rank r (bf16) in a
 * pool [num_blocks][block_size][rank]; query head h sees the key W_K[h] c and
 * the value W_V[h] c, with W_K, W_V bf16 [num_q_heads][head_dim][rank].
 * ------------------------------------------------------------------------- */

/* Scatter c_new [T][rank] (bf16, device) into the latent pool at
 * slot_mapping (int64 [T]; slot = block * block_size + row; negative = skip;
 * beyond the pool = skipped and reported in the device error word).
 * rank * 2 bytes must be a multiple of 16.  Byte-exact copy. */
pkv_status pkv_latent_append(const void *c_new, void *c_cache, const int64_t *slot_mapping,
                             int64_t num_tokens, int64_t num_blocks, int rank, int block_size,
                             pkv_stream_t stream);

/* Device scratch pkv_mla_decode_attention needs (absorbed queries, the
 * attention over the latent, split partials). */
size_t pkv_mla_workspace_bytes(int num_seqs, int num_q_heads, int rank, int max_seq_len);

/* Decode over the latent cache: out[b][h] = sum_j softmax_j(scale * q[b][h] .
 * W_K[h] c_j) W_V[h] c_j over the seq_lens[b] latents of sequence b, read
 * through block_table (int32 [num_seqs][max_blocks_per_seq]).  q, out bf16
 * [num_seqs][num_q_heads][head_dim].  Computed with the projections absorbed:
 * q~ = W_K^T q, attention of q~ over the latents, then W_V applied to the
 * result.  Supported: num_q_heads 32, head_dim 128, rank 128, block_size 16
 * (PKV_EUNSUPPORTED otherwise).  workspace: 256-byte aligned, at least
 * pkv_mla_workspace_bytes(...) bytes (PKV_ERANGE if smaller). */
pkv_status pkv_mla_decode_attention(void *out, const void *q, const void *w_k, const void *w_v,
                                    const void *c_cache, const int32_t *block_table,
                                    const int32_t *seq_lens, int num_seqs, int max_blocks_per_seq,
                                    int max_seq_len, int64_t num_blocks, int num_q_heads,
                                    int head_dim, int rank, int block_size, float scale,
                                    void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* As pkv_mla_decode_attention, with each sequence's new latent appended in
 * the same call: c_new [num_seqs][rank] (bf16, 16-byte aligned) goes to
 * position seq_lens[b] - 1 of sequence b (its slot read from block_table), a
 * byte-exact copy, before any latent is read.  The result and the pool equal
 * those of pkv_latent_append at those slots followed by
 * pkv_mla_decode_attention.  A length outside [1, max_seq_len] leaves the
 * pool untouched for that sequence (the decode reports it); a block id
 * outside the pool is skipped and reported in the device error word. */
pkv_status pkv_mla_decode_attention_append(void *out, const void *q, const void *c_new,
                                           const void *w_k, const void *w_v, void *c_cache,
                                           const int32_t *block_table, const int32_t *seq_lens,
                                           int num_seqs, int max_blocks_per_seq, int max_seq_len,
                                           int64_t num_blocks, int num_q_heads, int head_dim,
                                           int rank, int block_size, float scale, void *workspace,
                                           size_t workspace_bytes, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Prefix caching (host-only): chained block hashes and a hash -> block index.
 * "The KV cache and prefix caching", section "A prefix already in the cache
 * can skip its prefill": the prompt is hashed block by block; a block's
 * identifier covers its tokens together with the identifier of the block
 * before it, so two sequences share a block identifier only if they agree on
 * every token up to and including that block; a hit is a contiguous prefix
 * starting at position 0, counted in whole blocks, so the last partial block
 * is always recomputed.  The pages name no hash; this library uses 64-bit
 * FNV-1a: h_b = FNV1a(le64(h_{b-1}) || le32(token_0) .. le32(token_{bs-1})),
 * h_{-1} = parent (0 for a fresh prompt).  These calls touch no GPU; the
 * index is host memory owned by the handle and is not thread-safe.
 * ------------------------------------------------------------------------- */

/* 64-bit FNV-1a of len bytes (offset basis 0xcbf29ce484222325, prime 0x100000001b3). */
uint64_t pkv_fnv1a64(const void *data, size_t len);

/* Chained hashes of the floor(num_tokens / block_size) full blocks of tokens
 * (host arrays) into out_hashes.  Returns that count, or -1 on bad arguments. */
int64_t pkv_prefix_hash_blocks(const int32_t *tokens, int64_t num_tokens, int block_size,
                               uint64_t parent, uint64_t *out_hashes);

typedef struct pkv_prefix_cache pkv_prefix_cache;

/* New empty index (NULL if host memory runs out); free with _destroy. */
pkv_prefix_cache *pkv_prefix_cache_create(void);
void pkv_prefix_cache_destroy(pkv_prefix_cache *cache);
/* Number of cached blocks, or -1 for a NULL handle. */
int64_t pkv_prefix_cache_size(const pkv_prefix_cache *cache);
/* Record that block hashes[i] is held in physical block block_ids[i] (>= 0);
 * an identifier already present keeps its block. */
pkv_status pkv_prefix_cache_insert(pkv_prefix_cache *cache, const uint64_t *hashes,
                                   const int32_t *block_ids, int64_t n);
/* Forget the given identifiers (absent ones are ignored). */
pkv_status pkv_prefix_cache_evict(pkv_prefix_cache *cache, const uint64_t *hashes, int64_t n);
/* Length of the longest prefix of hashes[0..n) that is cached; the matching
 * physical blocks go to out_block_ids (may be NULL).  -1 on bad arguments. */
int64_t pkv_prefix_cache_match(const pkv_prefix_cache *cache, const uint64_t *hashes, int64_t n,
                               int32_t *out_block_ids);
/* Plan a prefill: hashes every full block of the prompt into out_hashes
 * (floor(num_tokens / block_size) entries), matches the cached prefix, and
 * returns the number of prompt tokens whose keys and values can be reused --
 * whole blocks only, and at most num_tokens - 1 so the last token is always
 * computed.  The reused physical blocks go to out_block_ids.  The caller then
 * runs chunked_prefill_attention with prior_len = that count.  -1 on bad
 * arguments. */
int64_t pkv_prefix_plan(const pkv_prefix_cache *cache, const int32_t *tokens, int64_t num_tokens,
                        int block_size, int32_t *out_block_ids, uint64_t *out_hashes);

/*
 * Read the device error word of the current device into *code (host) and,
 * if clear != 0, reset it to PKV_DEVERR_NONE.  Synchronises the device.
 */
pkv_status pkv_get_device_error(int *code, int clear);

/*
 * l2_flush -- measurement helper, not part of the attention path.  Evicts
 * the L2 cache ahead of a timed launch whose inputs are small enough to stay
 * in it (the 16-sequence, 65-token decode batch holds 4.3 MB of keys and
 * values; GB300's L2 is 129 MB): timed without it, such a launch measures
 * the L2, not HBM.
 *   buf    device buffer, 16-byte aligned, owned by the caller; read only.
 *          Pass one several times larger than the L2.
 *   bytes  its size, a multiple of 16.
 *   sink   one device int the kernel may write (it never does in practice);
 *          it keeps the reads from being optimised away.
 * Reads the whole buffer with 16-byte loads on `stream`, which leaves the L2
 * holding clean lines of it, so the next launch evicts them without
 * write-backs.  PKV_EINVAL on a null or misaligned argument; PKV_ECUDA on a
 * launch error.
 */
pkv_status pkv_l2_flush(const void *buf, size_t bytes, int *sink, pkv_stream_t stream);

/*
 * set_span_buffer -- a measurement aid for pkv_decode_prefill_attention,
 * whose two halves overlap in time on one stream, so that events around the
 * call see only the pair.  With buf set (device memory, 8-byte aligned, four
 * uint64 the caller initialises to {UINT64_MAX, 0, UINT64_MAX, 0}), later
 * side-by-side calls record, with atomic min / max, the earliest CTA start
 * and the latest CTA end of the prefill (buf[0], buf[1]) and of the decode's
 * main kernel (buf[2], buf[3]), in %globaltimer nanoseconds.  NULL turns it
 * off (the default).  A process-wide setting, not thread-safe; PKV_EINVAL on
 * a misaligned pointer.  Host-only.
 */
pkv_status pkv_set_span_buffer(unsigned long long *buf);

/* Static description of a status code.  Host-only. */
const char *pkv_status_str(pkv_status status);

/* ABI version of this header (bumped on any incompatible change).  Host-only. */
int pkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
