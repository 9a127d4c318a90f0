// Decode attention over a latent (MLA-style) KV cache on tcgen05 (sm_103a).
//
// What it computes.  "The KV cache and prefix caching", section "What prefill
// stores and decode reads", names multi-head latent attention (the DeepSeek
// line): per token the cache stores a low-rank latent c instead of keys and
// values, and query head h sees the key W_K[h] c and the value W_V[h] c.
// With the projections absorbed -- q~_h = W_K[h]^T q_h before this kernel and
// o_h = W_V[h] z_h after it -- the attention over the latent is
//   z_h = sum_j softmax_j(scale * q~_h . c_j) c_j,
// grouped-query decode with a single KV head whose key and value are both the
// latent, shared by all 32 query heads.  This kernel computes z (rank 128).
//
// Every latent byte feeds 32 heads x 2 products, eight times the multiply
// work per byte of the GQA decode, so the products go to the tensor core and
// the warps keep only the softmax.  Per 128-key tile of latents (32 KiB):
//   S^T  = C . Q~^T    M = 128 keys,  N = 32 heads,   K = 128 rank
//   O^T += C^T . P^T   M = 128 rank,  N = 32 heads,   K = 128 keys
// The tile C is read by both products from the same shared-memory copy: as a
// K-major A operand for the scores and as an MN-major A operand for P V.
// S^T and O^T live in TMEM (fp32); P^T goes through shared memory (bf16, the
// B operand), heads contiguous per key: two tiles' P^T share one buffer of
// 128-byte rows, a half each, which leaves room for a five-tile latent ring
// (the ring's depth sets how many bytes are in flight per SM).
//
// Layout of a tile.  Each 16-token block (4 KiB) arrives in one TMA box of a
// 4-D view of the pool (column, row of 8, half, 8-row group) and lands as
// [row group][half][8 rows][128 B] with the 128-byte swizzle: every 8 keys x
// 64 rank columns are one 1 KiB swizzle atom.  For the score product the
// atoms of one half follow each other every 2 KiB along the keys; for P V the
// two rank halves of an atom pair sit 1 KiB apart and the 8-key atoms 2 KiB
// apart.  One box per block halves the TMA issue count of two 2 KiB boxes,
// and eight lanes of the producer warp issue a tile's boxes side by side.
//
// Roles (224 threads, one CTA per SM):
//   warps 0-3  softmax.  Thread j owns key j of each tile (TMEM lane j of
//              S^T) and rank dimension j of O^T.  The running max per head
//              (log2 domain) only has to bound the scores to within 2^8: one
//              barrier reduction (bar.red.or) over the 128 threads decides
//              whether any score exceeds it, and only then is the exact max
//              over the tile's keys taken (warp reductions, then shared
//              memory) and O^T rescaled in TMEM.  Each thread keeps the sum of
//              its own keys' weights per head; they are added up once per
//              unit.  Rows of keys past a sequence's end are zeroed in the
//              tile, so stale pool bytes (even NaN) never meet p = 0 in P V.
//   warp 4     TMA producer: the unit's q~ (32 rows) into a two-buffer ring,
//              the latent blocks of each tile into a five-tile ring.
//   warp 5     TMEM allocator and issuer of the score products S^T (converged
//              warp, one elected lane per instruction), as soon as a tile's
//              latents are in: the scores of the next tiles are computed
//              while the softmax of this one runs.
//   warp 6     issuer of P V, as soon as a tile's softmax is done (its own
//              warp, so it never waits behind latents still on their way).
// Work: persistent CTAs take the balanced walk over 128-token stages (equal
// shares of all sequences' stages, cut where sequences change) when the
// batch gives every CTA at least 512 tokens, else 512-token splits; a piece
// that covers its whole sequence writes z, the others write (m, l, O)
// partials that the merge + up-projection kernel launched next combines.  O^T is double-buffered across
// pieces, so a piece's epilogue overlaps the next piece's products.
// Every wait is bounded; on time-out the kernel records an error, stops
// issuing work, lets its copies and products finish, frees its TMEM and
// returns.  After an abort the softmax warps still walk their loops
// (skipping the work), so every named barrier is reached by all of them.
#include <cuda.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "host_cache.h"
#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace pkv {
namespace {

constexpr int kTK = 128;                        // keys per tile
constexpr int kR = 128;                         // latent rank
constexpr int kNH = 32;                         // query heads
constexpr int kNPV = 32;                        // P^T / O^T columns: the 32 heads
constexpr int kBlkPerTile = kTK / kBlockSize;   // 8
constexpr int kBlockBytes = kBlockSize * kR * 2;   // 4 KiB
constexpr int kTileBytes = kTK * kR * 2;        // 32 KiB
constexpr int kNS = 5;                          // latent ring depth (tiles)
constexpr int kQBytes = kNH * kR * 2;           // 8 KiB: q~ of one sequence
constexpr int kQHalf = kQBytes / 2;             // one 64-column half, 32 rows
// P^T of two tiles in one buffer of 128 keys x 128-byte rows: tile parity b
// holds its 32 heads in bytes 64 b .. 64 b + 63 of each row
constexpr int kPBytes = kTK * 128;
constexpr int kThreadsT = 224;
constexpr int kSoft = 128;                      // softmax threads
constexpr int W_PROD = 4, W_MMA = 5, W_PV = 6;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t COL_S = 0;                   // S^T of tile parity b at 32 b
constexpr uint32_t COL_O = 64;                  // O^T of unit parity b at 64 + 32 b
constexpr float kLazyT = 8.0f;
constexpr unsigned kAllT = 0xffffffffu;
constexpr int kStageTokT = kTK;                 // the balanced walk's stage: one tile
constexpr int kMinStagesT = kSplitTokens / kStageTokT;   // shares of at least 4 stages
// Empty stages the balanced walk counts after every sequence: what one piece
// costs on top of its tiles (its queries, its epilogue, the first tile's
// exact maximum), in tiles.  CTAs whose shares start many short sequences
// then take fewer tiles.  Shares still hold at least kMinStagesT stages, so
// a sequence of n tokens still falls to at most ceil(n / 512) + 1 CTAs.
// Swept on the ragged 128-sequence batch (us per layer, call with append):
// 3: 50.7, 4: 50.3, 5: 50.6, 6: 51.2, 8: 51.8; on the 2,301-token batch 4
// is 2% behind 3.
constexpr int kPadT = 4;

// The producer walks the CTA's share and publishes each piece (sequence,
// piece index and count, token range) in a small ring; the other roles read
// it there instead of walking themselves.  Measured: the walk's code, run
// once per piece by the softmax warps, cost them about 1.5 us per piece
// boundary (it is too rarely run to stay in the instruction cache).
constexpr int kND = 4;
constexpr int OFF_RING = 0;
constexpr int OFF_Q = OFF_RING + kNS * kTileBytes;          // [2] q~
constexpr int OFF_P = OFF_Q + 2 * kQBytes;                  // P^T of both tile parities
constexpr int OFF_RED = OFF_P + kPBytes;                    // [2][32 heads][4 warps] fp32 (max)
constexpr int OFF_SUM = OFF_RED + 2 * kNH * 4 * 4;          // [2][32 heads][4 warps] fp32 (sums)
constexpr int OFF_BAR = OFF_SUM + 2 * kNH * 4 * 4;

enum {
  B_CF = 0,                 // [kNS] latent tile landed
  B_CE = B_CF + kNS,        // [kNS] latent tile consumed (both products done)
  B_QF = B_CE + kNS,        // [2]  q~ landed
  B_QE = B_QF + 2,          // [2]  q~ consumed (last S^T of its unit done)
  B_SF = B_QE + 2,          // [2]  S^T ready
  B_SE = B_SF + 2,          // [2]  S^T read out by the softmax
  B_PF = B_SE + 2,          // [2]  P^T written (and invalid rows of C zeroed)
  B_PE = B_PF + 2,          // [2]  P V of that tile done (P^T free, O^T settled)
  B_OF = B_PE + 2,          // [2]  O^T of a unit complete
  B_OE = B_OF + 2,          // [2]  O^T read out by the epilogue
  B_DRAIN = B_OE + 2,       // [2] each issuer's last products done
  B_DF = B_DRAIN + 2,       // [kND] a piece descriptor published
  B_DE = B_DF + kND,        // [kND] a piece descriptor read by every role
  B_COUNT = B_DE + kND
};
constexpr int OFF_PD = OFF_BAR + B_COUNT * 8;               // [kND] piece descriptors, 8 ints each
constexpr int OFF_SP = OFF_PD + kND * 32;                   // [2] the softmax warps' copy
constexpr int OFF_TSLOT = OFF_SP + 2 * 32;
constexpr int OFF_ABORT = OFF_TSLOT + 4;
constexpr int OFF_CU = OFF_TSLOT + 16;
static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzled operands need 1 KiB alignment");
static_assert(kSplitTokens % kTK == 0, "a split holds whole tiles");
static_assert(32 % kBlkPerTile == 0, "a tile never straddles two block-id windows");

// kind::f16 instruction descriptor with both operands MN-major (A = C^T).
__host__ __device__ constexpr uint32_t idesc_mn_mn(int m, int n) {
  return make_idesc(true, m, n) | (1u << 15);
}

__device__ __forceinline__ void tma4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int w,
                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %3, %3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(w), "l"(policy)
      : "memory");
}
// Bring one 4 KiB block of the pool into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma4d_prefetch_l2(const CUtensorMap* map, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %1, %1, %2}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(w)
               : "memory");
}
__device__ __forceinline__ void tma2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                      int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// OR of `pred` over the `count` threads of named barrier `id` (a barrier too)
__device__ __forceinline__ bool bar_red_or(bool pred, int id, int count) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Maximum of v over the warp (every lane gets it); -inf inputs are ordinary.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Lane l returns the sum over the warp's lanes of element l of v (v is
// consumed): a butterfly that halves the elements each lane carries at every
// step.
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      const float got = __shfl_xor_sync(kAllT, send, w);
      v[i] = keep + got;
    }
  }
  return v[0];
}

// Per-tile facts every role derives the same way from the walk.
struct TileInfo {
  int tok0;      // first token of the tile in its sequence
  int valid;     // keys of the tile inside the piece (1..128)
  bool first;    // first tile of its piece
  bool last;     // last tile of its piece
};

__global__ void __launch_bounds__(kThreadsT, 1)
decode_mla_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_c,
                  const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  int* abort_i = reinterpret_cast<int*>(smem + OFF_ABORT);
  volatile int* abort_flag = abort_i;
  int* cu = reinterpret_cast<int*>(smem + OFF_CU);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  if (sbase & 1023u) {  // swizzled operand tiles need a 1 KiB-aligned base
    if (threadIdx.x == 0) record_error(a.err, DEVERR_SMEM_LAYOUT);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(bar(B_CF + i), 1);
      mbar_init(bar(B_CE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_QF + i), 1);
      mbar_init(bar(B_QE + i), 1);
      mbar_init(bar(B_SF + i), 1);
      mbar_init(bar(B_SE + i), 4);    // one arrival per softmax warp
      mbar_init(bar(B_PF + i), 4);
      mbar_init(bar(B_PE + i), 1);
      mbar_init(bar(B_OF + i), 1);
      mbar_init(bar(B_OE + i), 4);
    }
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    for (int i = 0; i < kND; ++i) {
      mbar_init(bar(B_DF + i), 1);
      mbar_init(bar(B_DE + i), 3);   // the two issuers and the softmax warps' leader
    }
    *abort_i = 0;
    fence_mbar_init();
  }
  // P^T starts finite (every byte a product reads is written before it is read)
  for (int i = tid; i < kPBytes / 16; i += kThreadsT)
    reinterpret_cast<uint4*>(smem + OFF_P)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // balanced walk over 128-token stages when the batch gives every CTA at
  // least 512 tokens; otherwise 512-token splits
  // the sequence lengths after the prefix sums, when they fit (the launcher
  // sized shared memory for them if so)
  int* lens = a.lens_in_smem ? cu + a.num_seqs + 1 : nullptr;
  plan_units(a, cu, a.balanced ? kStageTokT : 0, kPadT, lens);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool balanced =
      a.balanced && (int64_t)cu[a.num_seqs] >= (int64_t)kMinStagesT * gridDim.x;
  if (a.balanced && !balanced) {
    __syncthreads();
    plan_units(a, cu, 0, 0, lens);
    __syncthreads();
  }
  const uint32_t tmem = *tmem_slot;
  int* pd = reinterpret_cast<int*>(smem + OFF_PD);
  // the merge + up-projection launched next may start now: it stages W_V
  // while this grid runs and waits for it to finish before reading results
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  auto tile_info = [&](const Unit& u, int i, int ntile) {
    TileInfo ti;
    ti.tok0 = u.tok_begin + i * kTK;
    ti.valid = min(kTK, u.tok_end - ti.tok0);
    ti.first = i == 0;
    ti.last = i == ntile - 1;
    return ti;
  };
  auto tiles_of = [&](const Unit& u) { return (u.tok_end - u.tok_begin + kTK - 1) / kTK; };

  if (warp == W_PROD) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_c)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    }
    const uint64_t policy = policy_evict_first();
    uint32_t t = 0, ui = 0;
    bool ok = true;
    // 32 block ids of piece v from its block `first` on, one per lane (the
    // range check comes at use, so a look-ahead request does not wait)
    auto load_ids = [&](const Unit& v, int first) {
      const int blk0 = v.tok_begin / kBlockSize;
      const int nblk = (v.tok_end - 1) / kBlockSize - blk0 + 1;
      return first + lane < nblk
                 ? __ldg(a.block_table + (int64_t)v.b * a.bt_stride + blk0 + first + lane)
                 : 0;
    };
    // The walk is looked at one piece ahead: the next piece's first block ids
    // are requested when this piece starts, so a switch between pieces does
    // not wait for a block-table read.
    Walk wk = walk_begin(a, cu, balanced, lens);
    Unit u, nu;
    bool have = walk_next(a, cu, kStageTokT, wk, u, kPadT);
    int ids = have ? load_ids(u, 0) : 0;
    // this piece's q~ (32 rows of the absorbed queries)
    auto load_q = [&](const Unit& v) {
      if (lane == 0) {
        if (ui >= 2) ok = wait_or_abort(bar(B_QE + (ui & 1)), ((ui >> 1) - 1) & 1, abort_flag, a.err);
        if (ok) {
          const uint32_t qb = sbase + OFF_Q + (ui & 1) * kQBytes;
          mbar_arrive_expect_tx(bar(B_QF + (ui & 1)), kQBytes);
          tma2d(qb, &tm_q, bar(B_QF + (ui & 1)), 0, v.b * kNH);
          tma2d(qb + kQHalf, &tm_q, bar(B_QF + (ui & 1)), 64, v.b * kNH);
        }
      }
      ok = __shfl_sync(kAllT, (int)ok, 0) != 0;
      if (ok) ++ui;
    };
    // publish piece v (or, with end set, the end of the walk) to the others
    uint32_t di = 0;
    auto publish = [&](const Unit& v, bool end) {
      if (lane == 0) {
        if (di >= (uint32_t)kND)
          ok = ok && wait_or_abort(bar(B_DE + di % kND), ((di / kND) - 1) & 1, abort_flag, a.err);
        if (ok) {
          int* d = pd + (di % kND) * 8;
          d[0] = end ? -1 : v.b;
          d[1] = v.s;
          d[2] = v.ns;
          d[3] = v.tok_begin;
          d[4] = v.tok_end;
          mbar_arrive(bar(B_DF + di % kND));   // release: the descriptor is visible to its readers
        }
      }
      ok = __shfl_sync(kAllT, (int)ok, 0) != 0;
      ++di;
    };
    // q~ comes from the kernel before this one in the stream (launched as its
    // programmatic dependent, this grid may start before that one has
    // finished), and so may the latent of each sequence's new token (the
    // query absorption can append it).  Nothing is requested into shared
    // memory before that grid is done: latent tiles requested earlier
    // competed in HBM with its loads and delayed it (measured: 53.6 -> 51.7
    // us per layer on the ragged batch, 26.7 -> 26.0 us on the 2,301-token
    // batch).  Only the first tile of the first piece is prefetched into L2
    // (32 KiB per CTA; a later copy reads L2, which also holds the appended
    // latent once that grid is done): 23.0 -> 22.6 us per layer on the
    // 2,301-token batch, the ragged batch unchanged; two tiles were no
    // faster.
    if (have) {
      const int nblk0 = (u.tok_end - 1) / kBlockSize - u.tok_begin / kBlockSize + 1;
      if (lane < min(nblk0, kBlkPerTile) && ids >= 0 && (int64_t)ids < a.num_blocks)
        tma4d_prefetch_l2(&tm_c, 2 * ids);
    }
    if (lane == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncwarp();
    while (ok && have) {
      publish(u, false);
      if (!ok) break;
      const bool have_next = walk_next(a, cu, kStageTokT, wk, nu, kPadT);
      const int next_ids = have_next ? load_ids(nu, 0) : 0;
      const int nblk = (u.tok_end - 1) / kBlockSize - u.tok_begin / kBlockSize + 1;
      const int ntile = tiles_of(u);
      load_q(u);
      if (!ok) break;
      for (int i = 0; i < ntile; ++i, ++t) {
        if (i > 0 && (i * kBlkPerTile) % 32 == 0) ids = load_ids(u, i * kBlkPerTile);
        const int slot = t % kNS;
        if (lane == 0 && t >= (uint32_t)kNS)
          ok = wait_or_abort(bar(B_CE + slot), ((t / kNS) - 1) & 1, abort_flag, a.err);
        ok = __shfl_sync(kAllT, (int)ok, 0) != 0;
        if (!ok) break;
        const int nb = min(kBlkPerTile, nblk - i * kBlkPerTile);
        int blk = __shfl_sync(kAllT, ids, (i * kBlkPerTile + (lane & 7)) & 31);
        if (lane < nb && (blk < 0 || (int64_t)blk >= a.num_blocks)) {
          record_error(a.err, DEVERR_BLOCK_RANGE);
          blk = 0;  // read a valid block instead; the error word reports it
        }
        const uint32_t fb = bar(B_CF + slot);
        if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(nb * kBlockBytes));
        __syncwarp();
        if (lane < nb)
          tma4d(sbase + OFF_RING + slot * kTileBytes + lane * kBlockBytes, &tm_c, fb, 2 * blk, policy);
      }
      u = nu;
      have = have_next;
      ids = next_ids;
    }
    if (ok) publish(u, true);
    if (!ok && lane == 0) {  // after an abort, let the copies already issued land
      const uint32_t first = t > (uint32_t)kNS ? t - kNS : 0;
      for (uint32_t i = first; i < t; ++i) mbar_wait(bar(B_CF + (i % kNS)), (i / kNS) & 1, nullptr);
      const uint32_t qfirst = ui > 2u ? ui - 2 : 0;
      for (uint32_t i = qfirst; i < ui; ++i) mbar_wait(bar(B_QF + (i & 1)), (i >> 1) & 1, nullptr);
    }
  } else if (warp == W_MMA || warp == W_PV) {
    // ------------------------------------------------------------- MMA issuers
    // Warp W_MMA issues S^T of every tile as soon as its latents, its q~ and
    // the S^T buffer are there; warp W_PV issues P V of every tile as soon as
    // its softmax is done.  Two issuers, each blocking on its own barriers,
    // keep P V from waiting behind the next tile's latents (one warp polling
    // both sets of barriers measured slower: each non-blocking probe of an
    // mbarrier costs on the order of a hundred cycles).
    constexpr uint32_t idesc_s = make_idesc(false, kTK, kNH);
    constexpr uint32_t idesc_o = idesc_mn_mn(kR, kNPV);
    const bool is_s = warp == W_MMA;
    bool ok = true;
    uint32_t t = 0, ui = 0;
    while (ok) {
      // the next piece, as the producer published it
      ok = __all_sync(kAllT, wait_or_abort(bar(B_DF + ui % kND), (ui / kND) & 1, abort_flag, a.err));
      if (!ok) break;
      Unit u;
      const int* d = pd + (ui % kND) * 8;
      u.b = d[0];
      u.s = d[1];
      u.ns = d[2];
      u.tok_begin = d[3];
      u.tok_end = d[4];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DE + ui % kND));
      if (u.b < 0) break;   // the end of the walk
      const int ntile = tiles_of(u);
      if (is_s) {
        ok = __all_sync(kAllT, wait_or_abort(bar(B_QF + (ui & 1)), (ui >> 1) & 1, abort_flag, a.err));
        if (!ok) break;
      }
      const uint32_t qb = sbase + OFF_Q + (ui & 1) * kQBytes;
      for (int i = 0; i < ntile && ok; ++i, ++t) {
        const uint32_t ct = sbase + OFF_RING + (t % kNS) * kTileBytes;
        if (is_s) {
          ok = __all_sync(kAllT, wait_fast(bar(B_CF + (t % kNS)), (t / kNS) & 1, abort_flag, a.err));
          if (ok && t >= 2)
            ok = __all_sync(kAllT, wait_fast(bar(B_SE + (t & 1)), ((t >> 1) - 1) & 1, abort_flag, a.err));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kR / 16; ++k) {
            // A = C (K-major): rank half k/4, 32 bytes per 16 columns; 8-key atoms 2 KiB apart
            const uint64_t ad = make_sw128_desc(ct + (k >> 2) * 1024 + (k & 3) * 32, 16, 2048);
            // B = Q~ (K-major): 8-head atoms 1 KiB apart, halves 4 KiB apart
            const uint64_t bd = make_sw128_desc(qb + (k >> 2) * kQHalf + (k & 3) * 32, 16, 1024);
            mma_ss_e(tmem + COL_S + (t & 1) * kNH, ad, bd, idesc_s, k > 0 ? 1u : 0u);
          }
          commit_e(bar(B_SF + (t & 1)));
          if (i == ntile - 1) commit_e(bar(B_QE + (ui & 1)));   // q~ buffer read
        } else {
          ok = __all_sync(kAllT, wait_fast(bar(B_PF + (t & 1)), (t >> 1) & 1, abort_flag, a.err));
          if (ok && i == 0 && ui >= 2)   // O^T of two pieces back has been read out
            ok = __all_sync(kAllT, wait_fast(bar(B_OE + (ui & 1)), ((ui >> 1) - 1) & 1, abort_flag, a.err));
          if (!ok) break;
          tc_fence_after();
          const uint32_t pt = sbase + OFF_P + (t & 1) * 64;
#pragma unroll
          for (int kk = 0; kk < kTK / 16; ++kk) {
            // A = C^T (MN-major): rank halves 1 KiB apart, 8-key atoms 2 KiB apart
            const uint64_t ad = make_sw128_desc(ct + kk * 2 * 2048, 1024, 2048);
            // B = P^T (MN-major, N = 32): this tile parity's half of the
            // 128-byte rows, 8-key atoms 1 KiB apart
            const uint64_t bd = make_sw128_desc(pt + kk * 16 * 128, 16, 1024);
            mma_ss_e(tmem + COL_O + (ui & 1) * kNPV, ad, bd, idesc_o, (i == 0 && kk == 0) ? 0u : 1u);
          }
          commit_e(bar(B_CE + (t % kNS)));
          commit_e(bar(B_PE + (t & 1)));
          if (i == ntile - 1) commit_e(bar(B_OF + (ui & 1)));
        }
      }
      ++ui;
    }
    // every product this warp issued completes before TMEM is freed
    const int drain = is_s ? B_DRAIN : B_DRAIN + 1;
    commit_e(bar(drain));
    mbar_wait(bar(drain), 0, nullptr);
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int wl = warp;                          // 0..3
    const int j = tid;                            // key of the tile / TMEM lane / rank dim
    const uint32_t lane_base = tmem + ((uint32_t)(wl * 32) << 16);
    const float sl2 = a.scale * 1.4426950408889634f;
    float* red = reinterpret_cast<float*>(smem + OFF_RED);   // [2][32][4]
    float* sum = reinterpret_cast<float*>(smem + OFF_SUM);   // [2][32][4]
    unsigned char* prow0 = smem + OFF_P + j * 128;            // P^T row of key j (buffer 0)
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
    // this key's place in a tile: 8-key group j/8 every 2 KiB, row j%8
    const uint32_t crow = (uint32_t)((j >> 3) * 2048 + (j & 7) * 128);
    float m[kNH], l[kNH];
    uint32_t t = 0, ui = 0;
    int* sp = reinterpret_cast<int*>(smem + OFF_SP);
    while (true) {
      // the next piece: the leader takes it from the producer's ring and
      // hands it to the four warps, which then agree on it even after an
      // abort (every named barrier must be reached by all of them)
      if (tid == 0) {
        int* dst = sp + (ui & 1) * 8;
        if (wait_or_abort(bar(B_DF + ui % kND), (ui / kND) & 1, abort_flag, a.err)) {
          const int* d = pd + (ui % kND) * 8;
#pragma unroll
          for (int k = 0; k < 5; ++k) dst[k] = d[k];
          mbar_arrive(bar(B_DE + ui % kND));
        } else {
          dst[0] = -1;
        }
      }
      named_bar_sync(1, kSoft);
      Unit u;
      {
        const int* d = sp + (ui & 1) * 8;
        u.b = d[0];
        u.s = d[1];
        u.ns = d[2];
        u.tok_begin = d[3];
        u.tok_end = d[4];
      }
      if (u.b < 0) break;   // the end of the walk (or an abort)
      // the merge reads how many partials this sequence left
      if (a.balanced && u.s == 0 && tid == 0) a.ws_np[u.b] = u.ns;
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      const int ntile = tiles_of(u);
      for (int i = 0; i < ntile; ++i, ++t) {
        const TileInfo ti = tile_info(u, i, ntile);
        wait_fast(bar(B_SF + (t & 1)), (t >> 1) & 1, abort_flag, a.err);
        __syncwarp();
        tc_fence_after();
        float x[kNH];
        tmem_ld32(lane_base + COL_S + (t & 1) * kNH, x);
        tmem_wait_ld();
        reg_fence(x);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SE + (t & 1)));
        const bool kval = j < ti.valid;
        // scores in the log2 domain; keys past the piece's end are -inf
        bool grow = false;
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          x[h] = kval ? x[h] * sl2 : -INFINITY;
          grow |= x[h] > m[h] + kLazyT;
        }
        if (bar_red_or(grow, 1, kSoft)) {
          // exact max per head over the tile's keys
          // per head, the maximum over this warp's 32 keys (one warp
          // reduction each); lane h keeps head h's
          float wm = -INFINITY;
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const float r = warp_max(x[h]);
            wm = lane == h ? r : wm;
          }
          float* rb = red + (t & 1) * kNH * 4;
          rb[lane * 4 + wl] = wm;
          named_bar_sync(1, kSoft);
          // lane h decides head h (the same on every warp), then the new
          // maxima and their rescale factors go to every lane.  Per-lane code
          // keeps this rarely run path short: unrolled over the 32 heads it
          // missed the instruction cache on every first tile of a piece.
          const float4 r4 = *reinterpret_cast<const float4*>(rb + lane * 4);
          const float mx = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
          float m_old = m[0];
#pragma unroll
          for (int h = 1; h < kNH; ++h) m_old = lane == h ? m[h] : m_old;
          float m_new = m_old;
          if (mx > m_new + kLazyT || m_new == -INFINITY) m_new = mx;
#pragma unroll
          for (int h = 0; h < kNH; ++h) m[h] = __shfl_sync(kAllT, m_new, h);
          // the first tile of a piece has no sums or O^T to rescale yet
          const float alpha_l = (ti.first || m_new == m_old) ? 1.f : fast_exp2(m_old - m_new);
          if (__any_sync(kAllT, alpha_l != 1.f)) {   // the same on every thread: m is uniform
            float alpha[kNH];
#pragma unroll
            for (int h = 0; h < kNH; ++h) alpha[h] = __shfl_sync(kAllT, alpha_l, h);
#pragma unroll
            for (int h = 0; h < kNH; ++h) l[h] *= alpha[h];
            {
              // O^T holds P V of this piece's earlier tiles: rescale it in
              // place once the last of those products has completed
              wait_fast(bar(B_PE + ((t - 1) & 1)), ((t - 1) >> 1) & 1, abort_flag, a.err);
              __syncwarp();
              tc_fence_after();
              float o[kNH];
              const uint32_t oc = lane_base + COL_O + (ui & 1) * kNPV;
              tmem_ld32(oc, o);
              tmem_wait_ld();
              reg_fence(o);
#pragma unroll
              for (int h = 0; h < kNH; ++h) o[h] *= alpha[h];
              tmem_st32(oc, o);
              tmem_wait_st();
            }
          }
        }
        // p = 2^(x - m) as bf16 (what P V multiplies; the sums use the same values)
        uint32_t pk[kNH / 2];
#pragma unroll
        for (int h = 0; h < kNH; h += 2) {
          const uint32_t pp = pack_bf16(fast_exp2(x[h] - m[h]), fast_exp2(x[h + 1] - m[h + 1]));
          l[h] += bf16lo(pp);
          l[h + 1] += bf16hi(pp);
          pk[h / 2] = pp;
        }
        // P^T of tile t - 2 has been read by its P V
        if (t >= 2) wait_fast(bar(B_PE + (t & 1)), ((t >> 1) - 1) & 1, abort_flag, a.err);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(prow0 + (((c + 4 * (t & 1)) ^ (j & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        if (!kval) {
          // zero this key's latent row (both halves): stale pool bytes must
          // not meet p = 0 in P V (0 x NaN)
          unsigned char* cr = smem + OFF_RING + (t % kNS) * kTileBytes + crow;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(cr + c * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(cr + 1024 + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PF + (t & 1)));
      }
      // ---- end of the piece: sums over all keys, then O^T / l or partials
      {
        float tmp[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) tmp[h] = l[h];
        const float ws = warp_transpose_sum(tmp, lane);   // head `lane`, this warp
        float* sb = sum + (ui & 1) * kNH * 4;
        sb[lane * 4 + wl] = ws;
        named_bar_sync(1, kSoft);
        // lane h: the sum over all 128 keys of head h, and its reciprocal
        // (one division per lane; per-lane code keeps this once-per-piece
        // path short enough to stay in the instruction cache)
        const float4 s4 = *reinterpret_cast<const float4*>(sb + lane * 4);
        const float L_l = (s4.x + s4.y) + (s4.z + s4.w);
        const float inv_l = 1.f / L_l;
        wait_fast(bar(B_OF + (ui & 1)), (ui >> 1) & 1, abort_flag, a.err);
        __syncwarp();
        tc_fence_after();
        float o[kNH];
        tmem_ld32(lane_base + COL_O + (ui & 1) * kNPV, o);
        tmem_wait_ld();
        reg_fence(o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_OE + (ui & 1)));
        if (u.ns == 1) {
          // the whole sequence: z = O / l
          __nv_bfloat16* orow = outp + (int64_t)u.b * a.num_q_heads * kR + j;
#pragma unroll
          for (int h = 0; h < kNH; ++h)
            orow[h * kR] = __float2bfloat16_rn(o[h] * __shfl_sync(kAllT, inv_l, h));
        } else {
          // a piece: partial (m, l, O) in slot u.s of each head's row
          const int64_t prow = (int64_t)u.b * a.num_q_heads * a.max_splits + u.s;
          float* acc = a.ws_acc + prow * kR + j;
#pragma unroll
          for (int h = 0; h < kNH; ++h) acc[(int64_t)h * a.max_splits * kR] = o[h];
          if (wl == 0) {
            float m_l = m[0];
#pragma unroll
            for (int h = 1; h < kNH; ++h) m_l = lane == h ? m[h] : m_l;
            float* ml = a.ws_ml + (prow + (int64_t)lane * a.max_splits) * 2;
            ml[0] = m_l;
            ml[1] = L_l;
          }
        }
      }
      ++ui;
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

}  // namespace

cudaError_t launch_decode_mla(const DecodeArgs& args, const void* w_v, void* out, int num_sms,
                              cudaStream_t stream) {
  DecodeArgs a = args;
  a.balanced = a.ws_np != nullptr && stage_plan_fits(a, kStageTokT, kPadT);
  if (a.chunk_prior >= 0 || a.split_tokens % kTK != 0 || a.num_kv_heads != 1 ||
      a.num_q_heads != kNH || a.head_dim != kR)
    return cudaErrorInvalidValue;
  CUtensorMap tm_c, tm_q;
  if (!encode_latent_block_map(&tm_c, a.k_cache, a.num_blocks)) return cudaErrorInvalidValue;
  if (!encode_rows32_map_bf16(&tm_q, a.q, (int64_t)a.num_seqs * kNH)) return cudaErrorInvalidValue;
  size_t smem = OFF_CU + sizeof(int) * (size_t)(a.num_seqs + 1);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  a.lens_in_smem = smem + sizeof(int) * (size_t)a.num_seqs <= 227 * 1024;
  if (a.lens_in_smem) smem += sizeof(int) * (size_t)a.num_seqs;
  cudaError_t e = allow_dynamic_smem(decode_mla_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t upper = (int64_t)a.num_seqs * a.max_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(upper < (int64_t)num_sms ? upper : (int64_t)num_sms));
  cfg.blockDim = dim3(kThreadsT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_mla_kernel, a, tm_c, tm_q);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge_project(a, w_v, out, stream);
}

}  // namespace pkv
