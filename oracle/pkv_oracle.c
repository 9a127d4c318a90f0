/*
 * Plain, slow, fp64 CPU oracle for attention over a block-paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes, and where the pages state it:
 *  - "KV cache and continuous batching: 1,000 people ask AI", section
 *    "What does a KV cache keep?": a decode step computes the new token's
 *    key, value and query, appends key and value to the cache, and attends
 *    over everything stored.
 *  - "The KV cache and prefix caching", section "What prefill stores and
 *    decode reads": the same statement, plus grouped-query attention
 *    (several query heads share one key/value head) and the PagedAttention
 *    layout: fixed-size blocks with a per-sequence block table.
 *  - "The KV cache is not your bottleneck", section "The fix that mattered":
 *    prompts are admitted in capped chunks (chunked prefill).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *  - query head h reads KV head h / (Hq / Hkv)  (contiguous groups);
 *  - pool layout [num_blocks][Hkv][block_size][D];
 *  - the token at logical position p of a sequence lives in physical block
 *    block_table[p / block_size], row p % block_size;
 *  - seq_lens counts the tokens stored after this step's append, so the new
 *    query attends over its own key;
 *  - a prefill chunk row i (absolute position prior + i) sees keys
 *    0 .. prior + i inclusive.
 *
 * Method: each sequence's keys and values are first gathered by a walk over
 * its block table into contiguous fp64 arrays; attention is then the plain
 * definition softmax(scale * q.K^T) V, with the maximum subtracted before
 * the exponential, in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ERANGE 3
#define ORACLE_ENOMEM 7

/* Storage element -> fp64.  dtype 0: IEEE binary32; dtype 1: bfloat16, the
 * upper 16 bits of a binary32, so widening is exact; dtype 3: IEEE binary64
 * (used for pools already dequantised from another storage format). */
static double load_elem(const void *base, int64_t idx, int dtype) {
  if (dtype == 0) return (double)((const float *)base)[idx];
  if (dtype == 3) return ((const double *)base)[idx];
  uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* kv_append: for every new token t with slot >= 0, copy its key row and value
 * row of every KV head into the pools, byte for byte.  slot = physical block *
 * block_size + row in block.  A negative slot means padding: nothing is
 * written.  Returns ORACLE_ERANGE if a slot lies outside the pool. */
int pkv_oracle_kv_append(const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int64_t *slot_mapping,
                         int64_t num_tokens, int64_t num_blocks,
                         int num_kv_heads, int head_dim, int block_size,
                         int elem_bytes) {
  const int64_t row_bytes = (int64_t)head_dim * elem_bytes;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * block_size) return ORACLE_ERANGE;
    int64_t blk = slot / block_size, row = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      int64_t dst = ((blk * num_kv_heads + h) * block_size + row) * row_bytes;
      int64_t src = ((t * num_kv_heads) + h) * row_bytes;
      memcpy((char *)k_cache + dst, (const char *)k_new + src, (size_t)row_bytes);
      memcpy((char *)v_cache + dst, (const char *)v_new + src, (size_t)row_bytes);
    }
  }
  return ORACLE_OK;
}

/* Walk one sequence's block table and copy the first n tokens of KV head g
 * into contiguous arrays kc[n][D], vc[n][D]. */
static int gather_head(double *kc, double *vc, const void *k_cache,
                       const void *v_cache, const int32_t *bt_row, int64_t n,
                       int64_t num_blocks, int num_kv_heads, int g,
                       int head_dim, int block_size, int dtype) {
  for (int64_t p = 0; p < n; ++p) {
    int32_t blk = bt_row[p / block_size];
    if (blk < 0 || blk >= num_blocks) return ORACLE_ERANGE;
    int64_t base =
        (((int64_t)blk * num_kv_heads + g) * block_size + p % block_size) *
        head_dim;
    for (int d = 0; d < head_dim; ++d) {
      kc[p * head_dim + d] = load_elem(k_cache, base + d, dtype);
      vc[p * head_dim + d] = load_elem(v_cache, base + d, dtype);
    }
  }
  return ORACLE_OK;
}

/* One query row over n contiguous keys: out = softmax(scale q.k_j) v_j.
 * w is scratch of length n. */
static void attend(double *out, const double *q, const double *kc,
                   const double *vc, int64_t n, int head_dim, double scale,
                   double *w) {
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    double s = 0.0;
    for (int d = 0; d < head_dim; ++d) s += q[d] * kc[j * head_dim + d];
    w[j] = scale * s;
    if (w[j] > m) m = w[j];
  }
  double z = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    w[j] = exp(w[j] - m);
    z += w[j];
  }
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  for (int64_t j = 0; j < n; ++j)
    for (int d = 0; d < head_dim; ++d) out[d] += w[j] * vc[j * head_dim + d];
  for (int d = 0; d < head_dim; ++d) out[d] /= z;
}

/* Decode attention over the paged cache.
 *   q       [B][Hq][D]           (dtype)
 *   pools   [num_blocks][Hkv][block_size][D] (dtype)
 *   block_table [B][max_blocks], seq_lens [B] (tokens stored, >= 1)
 * If pairs is NULL, out is [B][Hq][D] fp64 for every (sequence, query head);
 * otherwise pairs holds npairs (sequence, query head) couples and out is
 * [npairs][D]. */
int pkv_oracle_decode(double *out, const void *q, const void *k_cache,
                      const void *v_cache, const int32_t *block_table,
                      const int32_t *seq_lens, int num_seqs, int max_blocks,
                      int64_t num_blocks, int num_q_heads, int num_kv_heads,
                      int head_dim, int block_size, double scale, int dtype,
                      const int32_t *pairs, int npairs) {
  if (num_q_heads % num_kv_heads != 0) return ORACLE_EINVAL;
  const int group = num_q_heads / num_kv_heads;
  const int64_t nwork = pairs ? npairs : (int64_t)num_seqs * num_q_heads;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t w = 0; w < nwork; ++w) {
    int b = pairs ? pairs[2 * w] : (int)(w / num_q_heads);
    int h = pairs ? pairs[2 * w + 1] : (int)(w % num_q_heads);
    if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads) {
      status = ORACLE_ERANGE;
      continue;
    }
    int64_t n = seq_lens[b];
    if (n < 1 || n > (int64_t)max_blocks * block_size) {
      status = ORACLE_ERANGE;
      continue;
    }
    double *kc = malloc(sizeof(double) * n * head_dim);
    double *vc = malloc(sizeof(double) * n * head_dim);
    double *sc = malloc(sizeof(double) * n);
    double *qd = malloc(sizeof(double) * head_dim);
    if (!kc || !vc || !sc || !qd) {
      status = ORACLE_ENOMEM;
    } else if (gather_head(kc, vc, k_cache, v_cache,
                           block_table + (int64_t)b * max_blocks, n, num_blocks,
                           num_kv_heads, h / group, head_dim, block_size,
                           dtype) != ORACLE_OK) {
      status = ORACLE_ERANGE;
    } else {
      for (int d = 0; d < head_dim; ++d)
        qd[d] = load_elem(q, ((int64_t)b * num_q_heads + h) * head_dim + d, dtype);
      attend(out + w * head_dim, qd, kc, vc, n, head_dim, scale, sc);
    }
    free(kc);
    free(vc);
    free(sc);
    free(qd);
  }
  return status;
}

/* Chunked prefill of one sequence: chunk row i (absolute position prior + i)
 * attends keys 0 .. prior + i of the sequence, read through bt_row.  The
 * chunk's own keys and values are already in the pools.
 *   q [chunk_len][Hq][D];  out [chunk_len][Hq][D] fp64, or [nrows][D] when
 *   rows (npairs (row, query head) couples) is given. */
int pkv_oracle_prefill(double *out, const void *q, const void *k_cache,
                       const void *v_cache, const int32_t *bt_row,
                       int max_blocks, int prior_len, int chunk_len,
                       int64_t num_blocks, int num_q_heads, int num_kv_heads,
                       int head_dim, int block_size, double scale, int dtype,
                       const int32_t *rows, int nrows) {
  if (num_q_heads % num_kv_heads != 0) return ORACLE_EINVAL;
  const int group = num_q_heads / num_kv_heads;
  const int64_t total = (int64_t)prior_len + chunk_len;
  if (total > (int64_t)max_blocks * block_size || chunk_len < 0 || prior_len < 0)
    return ORACLE_ERANGE;
  /* gather every KV head once: kc[g][total][D] */
  double *kc = malloc(sizeof(double) * num_kv_heads * total * head_dim + 8);
  double *vc = malloc(sizeof(double) * num_kv_heads * total * head_dim + 8);
  if (!kc || !vc) {
    free(kc);
    free(vc);
    return ORACLE_ENOMEM;
  }
  int status = ORACLE_OK;
  for (int g = 0; g < num_kv_heads && status == ORACLE_OK; ++g)
    status = gather_head(kc + (int64_t)g * total * head_dim,
                         vc + (int64_t)g * total * head_dim, k_cache, v_cache,
                         bt_row, total, num_blocks, num_kv_heads, g, head_dim,
                         block_size, dtype);
  const int64_t nwork = rows ? nrows : (int64_t)chunk_len * num_q_heads;
  if (status == ORACLE_OK) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t w = 0; w < nwork; ++w) {
      int i = rows ? rows[2 * w] : (int)(w / num_q_heads);
      int h = rows ? rows[2 * w + 1] : (int)(w % num_q_heads);
      if (i < 0 || i >= chunk_len || h < 0 || h >= num_q_heads) {
        status = ORACLE_ERANGE;
        continue;
      }
      int g = h / group;
      int64_t n = (int64_t)prior_len + i + 1;
      double *sc = malloc(sizeof(double) * n);
      double *qd = malloc(sizeof(double) * head_dim);
      if (!sc || !qd) {
        status = ORACLE_ENOMEM;
      } else {
        for (int d = 0; d < head_dim; ++d)
          qd[d] = load_elem(q, ((int64_t)i * num_q_heads + h) * head_dim + d, dtype);
        attend(out + w * head_dim, qd, kc + (int64_t)g * total * head_dim,
               vc + (int64_t)g * total * head_dim, n, head_dim, scale, sc);
      }
      free(sc);
      free(qd);
    }
  }
  free(kc);
  free(vc);
  return status;
}

/* Recompute path: full causal attention over one contiguous, unpaged
 * sequence, the computation a loop without a cache redoes at every step.
 *   q [T][Hq][D], k, v [T][Hkv][D]  ->  out [T][Hq][D] fp64
 * Row t attends keys 0 .. t. */
int pkv_oracle_causal_attention(double *out, const void *q, const void *k,
                                const void *v, int seq_len, int num_q_heads,
                                int num_kv_heads, int head_dim, double scale,
                                int dtype) {
  if (num_q_heads % num_kv_heads != 0) return ORACLE_EINVAL;
  const int group = num_q_heads / num_kv_heads;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int g = 0; g < num_kv_heads; ++g) {
    double *kc = malloc(sizeof(double) * seq_len * head_dim + 8);
    double *vc = malloc(sizeof(double) * seq_len * head_dim + 8);
    double *sc = malloc(sizeof(double) * seq_len + 8);
    double *qd = malloc(sizeof(double) * head_dim);
    if (!kc || !vc || !sc || !qd) {
      status = ORACLE_ENOMEM;
    } else {
      for (int64_t p = 0; p < seq_len; ++p)
        for (int d = 0; d < head_dim; ++d) {
          int64_t idx = (p * num_kv_heads + g) * head_dim + d;
          kc[p * head_dim + d] = load_elem(k, idx, dtype);
          vc[p * head_dim + d] = load_elem(v, idx, dtype);
        }
      for (int hh = 0; hh < group; ++hh) {
        int h = g * group + hh;
        for (int64_t t = 0; t < seq_len; ++t) {
          for (int d = 0; d < head_dim; ++d)
            qd[d] = load_elem(q, (t * num_q_heads + h) * head_dim + d, dtype);
          attend(out + (t * num_q_heads + h) * head_dim, qd, kc, vc, t + 1,
                 head_dim, scale, sc);
        }
      }
    }
    free(kc);
    free(vc);
    free(sc);
    free(qd);
  }
  return status;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int pkv_oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Set the number of OpenMP threads later calls use (no effect without
 * OpenMP).  Timing only: the results do not depend on it. */
void pkv_oracle_set_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
