// Paged grouped-query decode attention on CUDA cores for fp32 storage (the
// bf16 path runs on tensor-core tiles in decode_mma.cu), plus the reduce
// kernel that merges split-K partials for both.
//
// What it computes ("KV cache and continuous batching: 1,000 people ask AI",
// section "What does a KV cache keep?"; "The KV cache and prefix caching",
// section "What prefill stores and decode reads"): each sequence's new query
// attends, per query head, over every key and value the sequence has stored,
// out[b][h] = softmax(scale * q[b][h] . K[b][:, h/G]) V[b][:, h/G], where the
// cache is a pool of fixed 16-token blocks reached through a per-sequence
// block table and G query heads share one KV head.
//
// Design (one GPU, HBM-bound):
//  * Work unit = (sequence, KV head, split of kSplitTokens tokens).  All G
//    query heads of the group are resident, so each cached K/V byte is read
//    from HBM exactly once.  Units are enumerated from a per-CTA prefix sum of
//    splits per sequence, so a ragged batch becomes an even work list; a
//    persistent grid of 2 CTAs per SM walks it round-robin.
//  * One producer warp streams each block's 4 KiB K tile and V tile (layout
//    [block][kv_head][16][D], so a tile is contiguous) into a ring of shared
//    memory stages with 1-D TMA bulk copies completing on mbarriers.  It runs
//    ahead across unit boundaries, so the ring never drains between units.
//  * Four consumer warps split into key groups of D*size/16 lanes; a lane owns
//    one 16-byte column chunk of every key of its group.  Scores: per-lane
//    partial dot products for KPG keys x G heads, then a transposed butterfly
//    reduction (P-1 shuffles per score for P lanes instead of P log P).
//    Each key group keeps its own online-softmax state (running max in the
//    log2 domain, lazily raised only when it grows by more than 8, sum and
//    accumulator) so no cross-warp traffic happens inside the loop; the groups
//    are merged once per unit through shared memory.
//  * A unit that covers its whole sequence writes the output directly;
//    otherwise it writes (m, l, acc) partials and the reduce kernel merges
//    them: o = sum_s 2^(m_s-M) acc_s / sum_s 2^(m_s-M) l_s.
//  * Tokens beyond a sequence's end inside its last block are masked before
//    the softmax and skipped in P.V, so stale pool contents (even NaN) never
//    reach the output.
//  * Chunk mode (chunk_prior >= 0) reuses the kernel for a causal prefill
//    chunk: row b is a query at position chunk_prior + b whose keys are the
//    first chunk_prior + b + 1 tokens of one block-table row.
#include "common.cuh"
#include "decode_common.cuh"
#include "host_cache.h"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kConsumers = 128;
constexpr int kThreads = kConsumers + 32;
constexpr float kLazyRescale = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr unsigned kFull = 0xffffffffu;

template <typename T, int D, int G>
struct Cfg {
  static constexpr int CH = Elem<T>::kPer16B;       // elements per 16-byte chunk
  static constexpr int LPK = D / CH;                // lanes per key
  static constexpr int KG = kConsumers / LPK;       // key groups
  static constexpr int KPG0 = LPK / G;
  static constexpr int KPG = KPG0 > 4 ? KPG0 : 4;   // keys per group per stage
  static constexpr int V = KPG * G;                 // partial scores per lane
  static constexpr int R = V / LPK;                 // scores per lane after reduction
  static constexpr int STAGE_TOK = KG * KPG;
  static constexpr int BPS = STAGE_TOK / kBlockSize;  // blocks per stage
  static constexpr int ROW_BYTES = D * (int)sizeof(T);
  static constexpr int TILE_BYTES = kBlockSize * ROW_BYTES;
  static constexpr int HALF_STAGE = STAGE_TOK * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * HALF_STAGE;
  static constexpr int NST = STAGE_BYTES <= 16384 ? 6 : (STAGE_BYTES <= 32768 ? 3 : 2);
  static constexpr int RING_BYTES = NST * STAGE_BYTES;
  static constexpr int COMB_BYTES = KG * G * (D + 2) * 4;
  static constexpr int PBUF_BYTES = KG * (V + G) * 4;
  static constexpr int BAR_BYTES = 2 * NST * 8 + 16;
  static constexpr int FIXED_SMEM = RING_BYTES + COMB_BYTES + PBUF_BYTES + BAR_BYTES;
  static_assert(LPK >= 2 && LPK <= 32 && (LPK & (LPK - 1)) == 0, "lanes per key");
  static_assert(V % LPK == 0 && R >= 1 && R <= G && G % R == 0, "score layout");
  static_assert(STAGE_TOK % kBlockSize == 0, "stage holds whole blocks");
  static_assert(kSplitTokens % STAGE_TOK == 0, "split holds whole stages");
  static_assert(32 % BPS == 0, "a stage never straddles two block-id windows");
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(const DecodeArgs a) {
  using C = Cfg<T, D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  float* comb = reinterpret_cast<float*>(smem + C::RING_BYTES);       // [KG][G][D] acc
  float* comb_ml = comb + C::KG * G * D;                               // [KG][G][2]
  float* pbuf = reinterpret_cast<float*>(smem + C::RING_BYTES + C::COMB_BYTES);  // [KG][V+G]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES + C::COMB_BYTES + C::PBUF_BYTES);
  int* abort_flag = reinterpret_cast<int*>(bars + 2 * C::NST);
  int* cu = reinterpret_cast<int*>(smem + C::FIXED_SMEM);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + C::NST);

  if (tid == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kConsumers / 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  plan_units(a, cu);
  __syncthreads();
  const int total = cu[a.num_seqs];
  volatile int* vabort = abort_flag;

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer
    const T* kc = static_cast<const T*>(a.k_cache);
    const T* vc = static_cast<const T*>(a.v_cache);
    const uint64_t policy = policy_evict_first();
    uint32_t issued = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Unit u = find_unit(a, cu, w);
      const int blk0 = u.tok_begin / kBlockSize;
      const int nblk = (u.tok_end - 1) / kBlockSize - blk0 + 1;
      const int32_t* bt_row = a.block_table + (int64_t)u.b * a.bt_stride + blk0;
      int my_blk = 0;  // block id of unit block (window*32 + lane)
      const int nst = (nblk + C::BPS - 1) / C::BPS;
      for (int st = 0; st < nst; ++st, ++issued) {
        if ((st * C::BPS) % 32 == 0) {  // next window of 32 block ids, one per lane
          const int idx = st * C::BPS + lane;
          my_blk = 0;
          if (idx < nblk) {
            my_blk = __ldg(bt_row + idx);
            if (my_blk < 0 || (int64_t)my_blk >= a.num_blocks) {
              record_error(a.err, DEVERR_BLOCK_RANGE);
              my_blk = 0;  // read a valid block instead; the error word reports it
            }
          }
        }
        const int buf = issued % C::NST;
        const uint32_t phase = (issued / C::NST) & 1;
        if (lane == 0 && issued >= (uint32_t)C::NST && !*vabort) {
          if (!mbar_wait(empty0 + 8 * buf, phase ^ 1, a.err)) { *vabort = 1; }
        }
        __syncwarp();
        if (*vabort) { ok = false; break; }
        const int nb = min(C::BPS, nblk - st * C::BPS);
        int blks[C::BPS];
#pragma unroll
        for (int i = 0; i < C::BPS; ++i) blks[i] = __shfl_sync(kFull, my_blk, (st * C::BPS + i) & 31);
        if (lane == 0) {
          const uint32_t fb = full0 + 8 * buf;
          mbar_arrive_expect_tx(fb, (uint32_t)(nb * 2 * C::TILE_BYTES));
          const uint32_t kdst = smem_u32(ring + buf * C::STAGE_BYTES);
          const uint32_t vdst = kdst + C::HALF_STAGE;
#pragma unroll
          for (int i = 0; i < C::BPS; ++i) {
            if (i < nb) {
              const int64_t tile = ((int64_t)blks[i] * a.num_kv_heads + u.g) * (kBlockSize * D);
              bulk_g2s_hint(kdst + i * C::TILE_BYTES, kc + tile, C::TILE_BYTES, fb, policy);
              bulk_g2s_hint(vdst + i * C::TILE_BYTES, vc + tile, C::TILE_BYTES, fb, policy);
            }
          }
        }
      }
    }
    // On abort, let every copy already issued land before the CTA exits.
    if (!ok && lane == 0) {
      const uint32_t first = issued > (uint32_t)C::NST ? issued - C::NST : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait(full0 + 8 * (i % C::NST), (i / C::NST) & 1, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  constexpr int CH = C::CH, LPK = C::LPK, KPG = C::KPG, V = C::V, R = C::R;
  const int kg = tid / LPK;           // key group
  const int l = tid % LPK;            // lane within the key group = column chunk
  const int kb = kg * KPG;            // first key of the group inside a stage
  const int kk_l = (R * l) / G;       // key of this lane's reduced scores
  const int h0 = (R * l) % G;         // first head of this lane's reduced scores
  const T* qp = static_cast<const T*>(a.q);
  T* outp = static_cast<T*>(a.out);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  float* my_p = pbuf + kg * (V + G);
  float* my_alpha = my_p + V;
  uint32_t consumed = 0;

  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const Unit u = find_unit(a, cu, w);
    const int hq0 = u.g * G;
    float qf[G][CH];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 raw = *reinterpret_cast<const uint4*>(
          qp + ((int64_t)u.b * a.num_q_heads + hq0 + h) * D + l * CH);
      float f[CH];
      Elem<T>::unpack(raw, f);
#pragma unroll
      for (int e = 0; e < CH; ++e) qf[h][e] = f[e] * scale_log2;
    }
    float acc[G][CH];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < CH; ++e) acc[h][e] = 0.f;
    float m_run[R], l_run[R];
#pragma unroll
    for (int i = 0; i < R; ++i) { m_run[i] = -INFINITY; l_run[i] = 0.f; }

    const int nblk = (u.tok_end - 1) / kBlockSize - u.tok_begin / kBlockSize + 1;
    const int nst = (nblk + C::BPS - 1) / C::BPS;
    for (int st = 0; st < nst; ++st, ++consumed) {
      const int buf = consumed % C::NST;
      const uint32_t phase = (consumed / C::NST) & 1;
      if (!*vabort) {
        if (!mbar_wait(full0 + 8 * buf, phase, a.err)) *vabort = 1;
      }
      const unsigned char* kst = ring + buf * C::STAGE_BYTES;
      const unsigned char* vst = kst + C::HALF_STAGE;
      const int tok0 = u.tok_begin + st * C::STAGE_TOK + kb;   // token of key 0 of the group
      const int nvalid = min(KPG, max(0, u.tok_end - tok0));   // uniform in the key group

      // scores: partial dot products over this lane's chunk
      float part[V];
#pragma unroll
      for (int kk = 0; kk < KPG; ++kk) {
        const uint4 raw = *reinterpret_cast<const uint4*>(kst + (kb + kk) * C::ROW_BYTES + l * 16);
        float kf[CH];
        Elem<T>::unpack(raw, kf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < CH; ++e) s = fmaf(qf[h][e], kf[e], s);
          part[kk * G + h] = s;
        }
      }
      // transposed reduction across the LPK lanes: lane l ends with scores
      // v = R*l .. R*l+R-1 (v = key*G + head)
#pragma unroll
      for (int m = LPK / 2, n = V; m >= 1; m >>= 1, n >>= 1) {
        const bool upper = (l & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float keep = upper ? part[i + n / 2] : part[i];
          const float send = upper ? part[i] : part[i + n / 2];
          part[i] = keep + __shfl_xor_sync(kFull, send, m);
        }
      }
      const bool key_ok = kk_l < nvalid;
      float mx[R];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        part[i] = key_ok ? part[i] : -INFINITY;
        mx[i] = part[i];
      }
#pragma unroll
      for (int m = G / R; m < LPK; m <<= 1)
#pragma unroll
        for (int i = 0; i < R; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(kFull, mx[i], m));
#pragma unroll
      for (int i = 0; i < R; ++i) {
        float m_new = m_run[i];
        if (mx[i] > m_run[i] + kLazyRescale || (m_run[i] == -INFINITY && mx[i] != -INFINITY))
          m_new = mx[i];
        const float alpha = (m_new == m_run[i]) ? 1.f : exp2f(m_run[i] - m_new);
        const float p = key_ok ? exp2f(part[i] - m_new) : 0.f;
        l_run[i] = l_run[i] * alpha + p;
        m_run[i] = m_new;
        my_p[R * l + i] = p;
        if (kk_l == 0) my_alpha[h0 + i] = alpha;
      }
      __syncwarp();
      float alpha[G];
#pragma unroll
      for (int h = 0; h < G; ++h) alpha[h] = my_alpha[h];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < CH; ++e) acc[h][e] *= alpha[h];
      // P.V over the valid keys of the group
#pragma unroll
      for (int kk = 0; kk < KPG; ++kk) {
        if (kk < nvalid) {
          const uint4 raw = *reinterpret_cast<const uint4*>(vst + (kb + kk) * C::ROW_BYTES + l * 16);
          float vf[CH];
          Elem<T>::unpack(raw, vf);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float p = my_p[kk * G + h];
#pragma unroll
            for (int e = 0; e < CH; ++e) acc[h][e] = fmaf(p, vf[e], acc[h][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);
    }

    // ---- merge the key groups of this unit
#pragma unroll
    for (int m = G / R; m < LPK; m <<= 1)
#pragma unroll
      for (int i = 0; i < R; ++i) l_run[i] += __shfl_xor_sync(kFull, l_run[i], m);
    if (kk_l == 0) {
#pragma unroll
      for (int i = 0; i < R; ++i) {
        comb_ml[(kg * G + h0 + i) * 2 + 0] = m_run[i];
        comb_ml[(kg * G + h0 + i) * 2 + 1] = l_run[i];
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < CH; ++e) comb[(kg * G + h) * D + l * CH + e] = acc[h][e];
    named_bar_sync(1, kConsumers);
    const bool direct = (u.ns == 1);
    for (int o = tid; o < G * D; o += kConsumers) {
      const int h = o / D, d = o - h * D;
      float M = -INFINITY;
#pragma unroll 4
      for (int k = 0; k < C::KG; ++k) M = fmaxf(M, comb_ml[(k * G + h) * 2]);
      float L = 0.f, O = 0.f;
#pragma unroll 4
      for (int k = 0; k < C::KG; ++k) {
        const float mk = comb_ml[(k * G + h) * 2];
        const float wk = (mk == -INFINITY) ? 0.f : exp2f(mk - M);
        L = fmaf(wk, comb_ml[(k * G + h) * 2 + 1], L);
        O = fmaf(wk, comb[(k * G + h) * D + d], O);
      }
      const int64_t row = (int64_t)u.b * a.num_q_heads + hq0 + h;
      if (direct) {
        Elem<T>::store(outp + row * D + d, O / L);
      } else {
        const int64_t pidx = row * a.max_splits + u.s;
        a.ws_acc[pidx * D + d] = O;
        if (d == 0) {
          a.ws_ml[pidx * 2 + 0] = M;
          a.ws_ml[pidx * 2 + 1] = L;
        }
      }
    }
    named_bar_sync(1, kConsumers);
  }
}

// Merge split partials: one warp per (sequence, query head).  Launched as the
// programmatic dependent of the main kernel (its launch overlaps that
// kernel's tail; its first instruction waits for that grid to complete).
// The partial rows are dead once merged: when the main kernel kept them in
// L2 (keep_partials) and they sit on whole 128-byte lines, each line is
// dropped from L2 after its last read, so they are never written back.
template <typename T, int D>
__global__ void __launch_bounds__(256)
decode_reduce_kernel(const DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_global >= a.num_seqs * a.num_q_heads) return;
  const int b = warp_global / a.num_q_heads;
  const int n = a.chunk_prior >= 0 ? a.chunk_prior + b + 1 : a.seq_lens[b];
  const int limit = min(a.max_seq_len, a.max_blocks_per_seq * kBlockSize);
  if (n < 1 || n > limit) return;  // reported by the main kernel
  const int h = warp_global - b * a.num_q_heads;
  const int ns = a.balanced
                     ? a.ws_np[b * a.num_kv_heads + h / (a.num_q_heads / a.num_kv_heads)]
                     : (n + a.split_tokens - 1) / a.split_tokens;
  if (ns <= 1) return;              // written directly by the main kernel
  const int64_t base = (int64_t)warp_global * a.max_splits;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, a.ws_ml[(base + s) * 2]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float L = 0.f;
  for (int s = lane; s < ns; s += 32) {
    const float ms = a.ws_ml[(base + s) * 2];
    L += (ms == -INFINITY ? 0.f : exp2f(ms - M)) * a.ws_ml[(base + s) * 2 + 1];
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
  const float inv = 1.f / L;
  T* outp = static_cast<T*>(a.out) + (int64_t)warp_global * D;
  if constexpr (D == 128) {
    if (a.partials_f16) {
      // partials stored as O / l in fp16: lane = 4 columns (8 bytes of the
      // 256-byte row); split s weighs 2^(m_s - M) l_s
      const uint2* acc2 =
          reinterpret_cast<const uint2*>(reinterpret_cast<const __half*>(a.ws_acc) + base * D) + lane;
      // lanes 0 and 16 drop the row's two 128-byte lines once read
      const bool drop = a.keep_partials && (reinterpret_cast<uintptr_t>(a.ws_acc) & 127u) == 0 &&
                        (lane & 15) == 0;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < ns; s0 += 32) {
        float wl = 0.f;
        if (s0 + lane < ns) {
          const float ms = a.ws_ml[(base + s0 + lane) * 2];
          wl = ms == -INFINITY ? 0.f : exp2f(ms - M) * a.ws_ml[(base + s0 + lane) * 2 + 1];
        }
        const int cnt = min(32, ns - s0);
        for (int k = 0; k < cnt; k += 8) {
          const int c8 = min(8, cnt - k);
          uint2 v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < c8) v[i] = acc2[(int64_t)(s0 + k + i) * (D / 4)];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i < c8) {
              const float wgt = __shfl_sync(kFull, wl, k + i);
              const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&v[i].x));
              const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&v[i].y));
              o.x = fmaf(wgt, lo.x, o.x);
              o.y = fmaf(wgt, lo.y, o.y);
              o.z = fmaf(wgt, hi.x, o.z);
              o.w = fmaf(wgt, hi.y, o.w);
            }
          }
          // every lane's read of these rows has returned (the FMAs used them)
          __syncwarp();
          if (drop) {
            for (int i = 0; i < c8; ++i) discard_l2_line(acc2 + (int64_t)(s0 + k + i) * (D / 4));
          }
        }
      }
      Elem<T>::store(outp + lane * 4 + 0, o.x * inv);
      Elem<T>::store(outp + lane * 4 + 1, o.y * inv);
      Elem<T>::store(outp + lane * 4 + 2, o.z * inv);
      Elem<T>::store(outp + lane * 4 + 3, o.w * inv);
      return;
    }
    // lane = 4-column group; split weights are computed once per lane (32
    // splits at a time) and broadcast, and 8 partial rows are loaded before
    // their FMAs so the L2 latency of the walk over splits overlaps
    const float4* acc4 = reinterpret_cast<const float4*>(a.ws_acc) + base * (D / 4) + lane;
    // lane 8i reads the first 16 bytes of line i of every 512-byte row
    const bool drop = a.keep_partials && (reinterpret_cast<uintptr_t>(a.ws_acc) & 127u) == 0 &&
                      (lane & 7) == 0;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += 32) {
      float wl = 0.f;
      if (s0 + lane < ns) {
        const float ms = a.ws_ml[(base + s0 + lane) * 2];
        wl = ms == -INFINITY ? 0.f : exp2f(ms - M);
      }
      const int cnt = min(32, ns - s0);
      int k = 0;
      for (; k + 8 <= cnt; k += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = acc4[(int64_t)(s0 + k + i) * (D / 4)];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float wgt = __shfl_sync(kFull, wl, k + i);
          o.x = fmaf(wgt, v[i].x, o.x);
          o.y = fmaf(wgt, v[i].y, o.y);
          o.z = fmaf(wgt, v[i].z, o.z);
          o.w = fmaf(wgt, v[i].w, o.w);
        }
        // every lane's read of these rows has returned (the FMAs used them)
        __syncwarp();
        if (drop) {
#pragma unroll
          for (int i = 0; i < 8; ++i) discard_l2_line(acc4 + (int64_t)(s0 + k + i) * (D / 4));
        }
      }
      for (; k < cnt; ++k) {
        const float wgt = __shfl_sync(kFull, wl, k);
        const float4 v = acc4[(int64_t)(s0 + k) * (D / 4)];
        o.x = fmaf(wgt, v.x, o.x);
        o.y = fmaf(wgt, v.y, o.y);
        o.z = fmaf(wgt, v.z, o.z);
        o.w = fmaf(wgt, v.w, o.w);
        __syncwarp();
        if (drop) discard_l2_line(acc4 + (int64_t)(s0 + k) * (D / 4));
      }
    }
    Elem<T>::store(outp + lane * 4 + 0, o.x * inv);
    Elem<T>::store(outp + lane * 4 + 1, o.y * inv);
    Elem<T>::store(outp + lane * 4 + 2, o.z * inv);
    Elem<T>::store(outp + lane * 4 + 3, o.w * inv);
  } else {
  for (int d4 = lane; d4 < D / 4; d4 += 32) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ns; ++s) {
      const float ms = a.ws_ml[(base + s) * 2];
      const float wgt = ms == -INFINITY ? 0.f : exp2f(ms - M);
      const float4 v = reinterpret_cast<const float4*>(a.ws_acc + (base + s) * D)[d4];
      o.x = fmaf(wgt, v.x, o.x);
      o.y = fmaf(wgt, v.y, o.y);
      o.z = fmaf(wgt, v.z, o.z);
      o.w = fmaf(wgt, v.w, o.w);
    }
    Elem<T>::store(outp + d4 * 4 + 0, o.x * inv);
    Elem<T>::store(outp + d4 * 4 + 1, o.y * inv);
    Elem<T>::store(outp + d4 * 4 + 2, o.z * inv);
    Elem<T>::store(outp + d4 * 4 + 3, o.w * inv);
  }
  }
}

template <typename T, int D>
cudaError_t launch_reduce_typed(const DecodeArgs& a, cudaStream_t stream) {
  const int warps = a.num_seqs * a.num_q_heads;
  if (warps == 0) return cudaSuccess;
  // programmatic dependent of the main kernel before it in the stream
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((warps + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_reduce_kernel<T, D>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D, int G>
cudaError_t launch_typed(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  using C = Cfg<T, D, G>;
  if (a.split_tokens % C::STAGE_TOK != 0) return cudaErrorInvalidValue;
  const size_t smem = C::FIXED_SMEM + sizeof(int) * (size_t)(a.num_seqs + 1);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = allow_dynamic_smem(decode_split_kernel<T, D, G>, (int)smem);
  if (e != cudaSuccess) return e;
  const int per_sm = smem <= 110 * 1024 ? 2 : 1;
  const int64_t upper = (int64_t)a.num_seqs * a.num_kv_heads * a.max_splits;
  const int grid = (int)(upper < (int64_t)num_sms * per_sm ? upper : (int64_t)num_sms * per_sm);
  decode_split_kernel<T, D, G><<<grid, kThreads, smem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  return launch_reduce_typed<T, D>(a, stream);
}

template <typename T, int D>
cudaError_t launch_group(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_typed<T, D, 1>(a, num_sms, stream);
    case 2: return launch_typed<T, D, 2>(a, num_sms, stream);
    case 4: return launch_typed<T, D, 4>(a, num_sms, stream);
    case 8: return launch_typed<T, D, 8>(a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_reduce_bf16_128(const DecodeArgs& a, cudaStream_t stream) {
  return launch_reduce_typed<__nv_bfloat16, 128>(a, stream);
}

bool decode_supported(int is_bf16, int head_dim, int group) {
  const bool g_ok = group == 1 || group == 2 || group == 4 || group == 8;
  return g_ok && !is_bf16 && (head_dim == 16 || head_dim == 128);
}

cudaError_t launch_paged_decode(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  if (a.is_bf16) return cudaErrorInvalidValue;  // bf16 runs on the tensor-core kernels
  if (a.head_dim == 16) return launch_group<float, 16>(a, num_sms, stream);
  if (a.head_dim == 128) return launch_group<float, 128>(a, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
