// Chunked-prefill attention on tcgen05 for two query heads of one GQA group
// per CTA (sm_103a).
//
// What it computes ("The KV cache is not your bottleneck", section "The fix
// that mattered": prompts are admitted in capped chunks; "KV cache and
// continuous batching: 1,000 people ask AI", section "What does a KV cache
// keep?": prefill is matrix-matrix work): chunk row i of one sequence, at
// absolute position prior + i, attends keys 0 .. prior + i of that sequence:
// out[i][h] = softmax(scale * q[i][h] . K^T) V, K and V of KV head h / G.
//
// Why this shape.
//  * K/V gathers.  A 16-token cache block is 16 rows; with the 128-byte
//    swizzle a TMA box then carries at most 2 KiB, and the SM's TMA unit
//    moves such boxes at only ~15-20 B/clk.  K/V are instead gathered through
//    the block table by two producer warps with 16-byte cp.async copies,
//    written straight into the 128B-swizzled K-major layout the MMAs read;
//    rows past the sequence end are zero-filled by the copy (source size 0),
//    so stale pool contents never enter.
//  * Shared-memory bandwidth.  Each CTA serves 128 query rows of two query
//    heads of the same KV head (every K/V tile feeds 256 rows), key tiles are
//    128 wide (Q K^T as M=128, N=128 instructions), and P never touches shared
//    memory: the softmax writes it as bf16 into the TMEM columns of its own S,
//    and P V reads its A operand from TMEM.
//  * TMEM: S_h (128 columns, P_h aliased over its first 64) and O_h
//    (128 columns) for the two heads = all 512 columns; one CTA per SM.  The
//    two heads take turns on the tensor core: while one head's softmax runs,
//    the other head's products execute.
// Roles (384 threads):
//   warps 0-3 / 4-7   softmax of head A / B: thread r owns query row r (TMEM
//                     lane r).  It loads its whole S row into registers (four
//                     TMEM loads in flight), takes the row max (causal mask on
//                     the diagonal tiles); the max is raised lazily, only when
//                     it grows by more than 2^8, and then O is rescaled in
//                     TMEM.  It forms p = 2^(s*scale*log2e - m) with one FMA and
//                     ex2 per score, sums it and stores it as bf16 into TMEM.
//                     P goes to the MMA issuer in two halves (one arrival per
//                     warp each): P V of the first 64 keys runs while the
//                     exponentials of the second 64 are formed.  Once a
//                     tile's S_B is complete, the head-B warps release its K
//                     stage (the S_B commit follows both heads' Q K^T).
//                     Epilogue O / l.
//   warps 8-9 / 11    K producers / V producer (cp.async; once their copies of
//                     a tile landed: proxy fence, mbarrier arrive).  K and V
//                     sit in separate two-stage rings with their own
//                     producers: a K stage is released once both heads' Q K^T
//                     have read it, a tile before its V stage, so the next K
//                     tile is in flight earlier.
//   warp 10           TMEM allocator and MMA issuer:
//                     S_h = Q_h K_j^T    (A, B from shared memory)
//                     O_h += P_h V_j     (A from TMEM, V as an MN-major B)
//                     The whole warp runs the issue loop and computes the
//                     (warp-uniform) descriptors; one elected lane issues each
//                     tcgen05 instruction.  Issuing from a lone lane inside a
//                     divergent branch starved the tensor core: the same
//                     instruction stream ran about 25% slower.
// Work items.  One item is 128 query rows x the two heads; by default each
// CTA runs one item (heaviest first).  In persistent mode a chosen number of
// CTAs each run a host-assigned list of items (longest first greedily, then
// improved by moves and swaps that lower the largest load), so the prefill
// holds exactly that many SMs: the decode of the same layer is then
// launched as a programmatic dependent and runs on the other SMs at the same
// time.  Rings, barrier phases and TMEM carry over from item to item: the
// next item's first Q K^T and P V follow the previous item's last products in
// issue order, and the softmax warps read the previous O out before they
// hand over the next item's first P.  Each item's Q is loaded once the
// previous item's Q K^T are done (the first by the MMA warp at once, the
// rest by the V producer).
// Every mbarrier wait is bounded; on time-out the kernel records an error,
// stops issuing work, lets its copies land, frees its TMEM and returns.
#include <cuda.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include <type_traits>

#include "common.cuh"
#include "host_cache.h"
#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace pkv {
namespace {

constexpr int BM = 128, BN = 128, HD = 128;
constexpr int QHALF = BM * 128;               // one 64-column half of a Q tile, 16 KiB
constexpr int Q_BYTES = 2 * QHALF;            // 32 KiB per head
constexpr int KHALF = BN * 128;               // one 64-column half of a K/V tile, 16 KiB
constexpr int KV_TILE = 2 * KHALF;            // 32 KiB
constexpr int NSK = 2, NSV = 2;               // K ring and V ring, released separately
constexpr int OFF_Q = 0;                      // [head][Q tile]
constexpr int OFF_K = 2 * Q_BYTES;            // [K stage]
constexpr int OFF_V = OFF_K + NSK * KV_TILE;  // [V stage]
constexpr int OFF_BAR = OFF_V + NSV * KV_TILE;
constexpr int SMEM_BYTES = OFF_BAR + 256;
constexpr int kSoftThreads = 256;
constexpr int kProdThreads = 64;
constexpr int W_MMA = 10, W_VPROD = 11;     // K producers: warps 8-9
constexpr int kThreadsPair = kSoftThreads + kProdThreads + 64;   // + MMA issuer + V producer
// registers per thread after the split (setmaxnreg), against the launch budget
constexpr int kRegsSoft = 200, kRegsRest = 96;
constexpr int kRegsLaunch = (65536 / kThreadsPair) & ~7;   // 168
static_assert(kRegsSoft * kSoftThreads + kRegsRest * (kThreadsPair - kSoftThreads) <=
                  kRegsLaunch * kThreadsPair,
              "the register split must fit in what the CTA was launched with");
constexpr uint32_t kTmemColsPair = 512;
constexpr uint32_t COL_S = 0;                 // S_h at 128*h (P_h in its first 64 columns)
constexpr uint32_t COL_O = 2 * BN;            // O_h at 256 + 128*h
constexpr float kLazyP = 8.0f;
static_assert(SMEM_BYTES <= 227 * 1024, "one CTA per SM");

// barrier slots
enum {
  PB_Q = 0,
  PB_KF = 1,                  // [NSK]
  PB_KE = PB_KF + NSK,        // [NSK]
  PB_VF = PB_KE + NSK,        // [NSV]
  PB_VE = PB_VF + NSV,        // [NSV]
  PB_SF = PB_VE + NSV,        // [head]
  PB_PF = PB_SF + 2,          // [head][half]
  PB_OD = PB_PF + 4,          // [head]
  PB_COUNT = PB_OD + 2
};
static_assert(PB_COUNT * 8 + 8 <= 256, "barrier area");

constexpr int kMaxItems = 512;      // persistent mode: work items in the parameter list
constexpr int kMaxCtas = 160;
struct PairParams {
  PrefillArgs a;
  int total_len;
  int kv_rows;
  int q_tiles;
  // The CTA's two streams ("heads" A and B below): two query heads of one KV
  // head over the same 128 query rows (rows_mode 0, the GQA group even), or
  // one head over two consecutive 128-row query tiles (rows_mode 1, any
  // group).  Either way every K/V tile feeds both.
  int rows_mode;
  // Persistent mode (n_list > 0): CTA c runs the work items
  // list[start[c]] .. list[start[c + 1] - 1] one after the other, item =
  // query tile * (heads / 2) + head pair, assigned by the host.  Otherwise
  // each CTA runs one item, head pair blockIdx.x, query tile from blockIdx.y.
  int n_list;
  uint16_t start[kMaxCtas + 1];
  uint16_t list[kMaxItems];
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async16_full(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}


__global__ void __launch_bounds__(kThreadsPair, 1)
prefill_pair_kernel(const __grid_constant__ PairParams p, const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + PB_COUNT);
  int* abort_i = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort_flag = abort_i;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const PrefillArgs& a = p.a;
  if (sbase & 1023u) {  // swizzled operand tiles need a 1 KiB-aligned base
    if (threadIdx.x == 0) record_error(a.err, DEVERR_SMEM_LAYOUT);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = a.num_q_heads / a.num_kv_heads;
  // items: x * ... + t with x the head pair (rows_mode 0) or the head
  // (rows_mode 1) and t the query tile or tile pair
  const int n_x = p.rows_mode ? a.num_q_heads : a.num_q_heads / 2;
  const int n_t = p.rows_mode ? (p.q_tiles + 1) / 2 : p.q_tiles;
  const int it_begin = p.n_list > 0 ? p.start[blockIdx.x] : 0;
  const int it_end = p.n_list > 0 ? p.start[blockIdx.x + 1] : 1;
  // work item it: stream hh covers head[hh], query rows qrow[hh] ..
  // qrow[hh] + 127; both read KV head g, key tiles 0 .. n_tiles - 1
  struct Item {
    int head[2], qrow[2], g, n_tiles;
  };
  auto item_at = [&](int it) {
    int x, tq;
    if (p.n_list > 0) {
      const int item = p.list[it];
      x = item % n_x;
      tq = item / n_x;
    } else {
      x = blockIdx.x;
      tq = n_t - 1 - (int)blockIdx.y;                     // heaviest tiles first
    }
    Item w;
    if (p.rows_mode) {
      w.head[0] = w.head[1] = x;
      w.qrow[0] = 2 * tq * BM;
      w.qrow[1] = w.qrow[0] + BM;
    } else {
      w.head[0] = 2 * x;
      w.head[1] = 2 * x + 1;
      w.qrow[0] = w.qrow[1] = tq * BM;
    }
    w.g = w.head[0] / group;
    w.n_tiles = (a.prior_len + min(a.chunk_len, w.qrow[1] + BM) - 1) / BN + 1;
    return w;
  };

  if (tid == 0) {
    span_mark(a.span, false);
    mbar_init(bar(PB_Q), 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(bar(PB_KF + s), kProdThreads);
      mbar_init(bar(PB_KE + s), 4);              // one arrival per head-B softmax warp
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(bar(PB_VF + s), 32);
      mbar_init(bar(PB_VE + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(PB_SF + i), 1);
      mbar_init(bar(PB_PF + 2 * i), 4);          // one arrival per softmax warp
      mbar_init(bar(PB_PF + 2 * i + 1), 4);
      mbar_init(bar(PB_OD + i), 1);
    }
    *abort_i = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemColsPair));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // persistent mode: this CTA holds its SM for the whole launch, so a kernel
  // launched next as a programmatic dependent may start on the other SMs
  if (p.n_list > 0 && tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp >= 8) {
    // Warpgroup 2 (producers and MMA issuer) hands registers to
    // the two softmax warpgroups (kRegsRest / kRegsSoft).  With the 168 of
    // the launch the softmax spilled; with 200 its whole S row, the running
    // sums and the packed P fit.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsRest));
    if (warp != W_MMA) {
      // ------------------------------------------------------------- K/V producers
      // warps 8-9 gather K, warp 11 gathers V, each pool on its own ring
      const bool is_v = warp == W_VPROD;
      const int nblk_seq = (p.total_len + kBlockSize - 1) / kBlockSize;
      // block ids of the sequence, 32 per window (one per lane), next window prefetched
      auto load_ids = [&](int win) {
        const int idx = win * 32 + lane;
        int blk = 0;
        if (idx < nblk_seq) {
          blk = __ldg(a.block_table_row + idx);
          if (blk < 0 || (int64_t)blk >= a.num_blocks) {
            record_error(a.err, DEVERR_BLOCK_RANGE);
            blk = 0;
          }
        }
        return blk;
      };
      constexpr int kBlkPerTile = BN / kBlockSize;   // 8
      constexpr int kTilesPerWin = 32 / kBlkPerTile;  // 4
      // NT threads copy a 128-key tile: 8 blocks of 16 rows; per block each
      // thread takes NT/16-row steps of one 16-byte chunk.  Rows past the
      // sequence end (last tile only) are zero-filled.
      auto produce = [&](auto nt_tag, const __nv_bfloat16* pool, uint32_t ring, int nst, int full_bar,
                         int empty_bar, int pt) {
        constexpr int NT = decltype(nt_tag)::value;
        constexpr int RS = NT / 16;                  // rows per step
        const int rsub = pt >> 4, cc = pt & 15;
        const int half = cc >> 3, ch = cc & 7;
        const uint32_t thr_dst = half * KHALF + rsub * 128;
        int jg = 0;                            // ring position over all items
        bool go = true, q_pending = false;
        uint32_t q_phase = 0;
        for (int it = it_begin; it < it_end && go; ++it) {
        const Item w = item_at(it);
        if (is_v) {
          // the item's Q (after the first), once the previous item's last
          // Q_B K^T has read the buffer
          const int ii = it - it_begin;
          if (ii > 0) go = wait_or_abort(bar(PB_SF + 1), (jg - 1) & 1, abort_flag, a.err);
          go = __all_sync(0xffffffffu, go && !*abort_flag);
          if (!go) break;
          if (lane == 0 && ii > 0) {
            mbar_arrive_expect_tx(bar(PB_Q), 2 * Q_BYTES);
            for (int hh = 0; hh < 2; ++hh) {
              tma_load_3d(sbase + OFF_Q + hh * Q_BYTES, &tm_q, bar(PB_Q), 0, w.head[hh], w.qrow[hh]);
              tma_load_3d(sbase + OFF_Q + hh * Q_BYTES + QHALF, &tm_q, bar(PB_Q), 64, w.head[hh], w.qrow[hh]);
            }
          }
          __syncwarp();
          if (ii > 0) {
            q_pending = true;
            q_phase = ii & 1;
          }
        }
        int cur_ids = load_ids(0), next_ids = load_ids(1);
        for (int j = 0; j < w.n_tiles; ++j, ++jg) {
          if (j > 0 && j % kTilesPerWin == 0) {
            cur_ids = next_ids;
            next_ids = load_ids(j / kTilesPerWin + 1);
          }
          if (jg >= nst) go = wait_or_abort(bar(empty_bar + jg % nst), ((jg / nst) - 1) & 1, abort_flag, a.err);
          go = __all_sync(0xffffffffu, go && !*abort_flag);
          if (!go) break;                      // leave the loop as a warp
          const uint32_t dst = ring + (jg % nst) * KV_TILE;
          const bool full = (j + 1) * BN <= p.total_len;
#pragma unroll 2
          for (int bi = 0; bi < kBlkPerTile; ++bi) {
            const int blk = __shfl_sync(0xffffffffu, cur_ids, ((j % kTilesPerWin) * kBlkPerTile + bi) & 31);
            const __nv_bfloat16* bsrc =
                pool + ((int64_t)blk * a.num_kv_heads + w.g) * (kBlockSize * HD) + rsub * HD + cc * 8;
            const uint32_t bdst = dst + thr_dst + bi * kBlockSize * 128;
            if (full) {
#pragma unroll
              for (int rq = 0; rq < kBlockSize / RS; ++rq)
                cp_async16_full(bdst + rq * RS * 128 + ((ch ^ ((rq * RS + rsub) & 7)) << 4),
                                bsrc + rq * RS * HD);
            } else {
#pragma unroll
              for (int rq = 0; rq < kBlockSize / RS; ++rq) {
                const int tok = j * BN + bi * kBlockSize + rq * RS + rsub;
                cp_async16(bdst + rq * RS * 128 + ((ch ^ ((rq * RS + rsub) & 7)) << 4), bsrc + rq * RS * HD,
                           tok < p.total_len ? 16u : 0u);
              }
            }
          }
          cp_async_commit();
          cp_async_wait<0>();
          fence_proxy_async_smem();             // make them visible to the tensor core
          mbar_arrive(bar(full_bar + jg % nst));
        }
        if (is_v && go) q_pending = false;   // its consumer waits for it before the item's products
        }
        // after an abort, let a Q load still in flight land
        if (is_v && q_pending) mbar_wait(bar(PB_Q), q_phase, nullptr);
        cp_async_wait<0>();
      };
      if (is_v)
        produce(std::integral_constant<int, 32>{}, static_cast<const __nv_bfloat16*>(a.v_cache),
                sbase + OFF_V, NSV, PB_VF, PB_VE, lane);
      else
        produce(std::integral_constant<int, 64>{}, static_cast<const __nv_bfloat16*>(a.k_cache),
                sbase + OFF_K, NSK, PB_KF, PB_KE, tid - kSoftThreads);
    } else if (warp == W_MMA) {
      // ------------------------------------------------------------- MMA issuer
      {
        // the first item's Q, at once (the V producer loads the later ones
        // as their buffer frees up); issuing it here, first thing, measured
        // 3% faster than from the V producer warp
        if (lane == 0) {
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
          const Item w0 = item_at(it_begin);
          mbar_arrive_expect_tx(bar(PB_Q), 2 * Q_BYTES);
          for (int hh = 0; hh < 2; ++hh) {
            tma_load_3d(sbase + OFF_Q + hh * Q_BYTES, &tm_q, bar(PB_Q), 0, w0.head[hh], w0.qrow[hh]);
            tma_load_3d(sbase + OFF_Q + hh * Q_BYTES + QHALF, &tm_q, bar(PB_Q), 64, w0.head[hh], w0.qrow[hh]);
          }
        }
        __syncwarp();
        constexpr uint32_t idesc_qk = make_idesc(false, BM, BN);
        constexpr uint32_t idesc_pv = make_idesc(true, BM, HD);
        // S_h = Q_h K^T of ring position jg into the TMEM columns of S_h
        auto issue_qk = [&](int hh, int jg) {
          const uint32_t kb = sbase + OFF_K + (jg % NSK) * KV_TILE;
          const uint32_t qa = sbase + OFF_Q + hh * Q_BYTES;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k) {
            const uint64_t ad = make_sw128_desc(qa + (k >> 2) * QHALF + (k & 3) * 32, 16, 1024);
            const uint64_t bd = make_sw128_desc(kb + (k >> 2) * KHALF + (k & 3) * 32, 16, 1024);
            mma_ss_e(tmem + COL_S + hh * BN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
          }
          commit_e(bar(PB_SF + hh));
        };
        // O_h += P_h V, P_h from TMEM (16 keys = 8 columns per step), for key
        // tile j of the item at ring position jg (half 0: keys 0-63, half 1:
        // keys 64-127; O_done is committed after the item's last tile only)
        auto issue_pv = [&](int hh, int jg, int j, int n_tiles, int half) {
          const uint32_t vb = sbase + OFF_V + (jg % NSV) * KV_TILE;
#pragma unroll
          for (int k = half * 4; k < half * 4 + 4; ++k) {
            const uint64_t bd = make_sw128_desc(vb + k * 16 * 128, KHALF, 1024);
            mma_ts_e(tmem + COL_O + hh * HD, tmem + COL_S + hh * BN + k * 8, bd, idesc_pv,
                     (j > 0 || k > 0) ? 1u : 0u);
          }
          if (half == 1 && j == n_tiles - 1) commit_e(bar(PB_OD + hh));
        };
        // The two heads alternate on the tensor core: while head A's softmax
        // turns S_A into P_A, the products of head B run, and the other way
        // round.  Q_h K_{j+1}^T rewrites S_h, which holds P_h, right behind
        // P_h V_j: tcgen05.mma operations issued by one thread execute in issue
        // order, so the earlier product has read P_h before the later one
        // writes there, and no wait for its completion is needed.  The same
        // holds across items, for the next item's first Q K^T and for its first
        // P V, which overwrites O_h after the softmax warps have read it out.
        // The tensor core queues only a few products ahead of the issuer, so
        // whatever the issuer does between products (waits, commits, fences)
        // can leave it idle.  The loop therefore commits only what a waiter
        // needs (S_h and V(j) per tile, O_h after an item's last tile; the
        // softmax warps release the K stages) and its waits take a fast path.
        int jg = 0;                        // ring position over all items
        bool ok = true, q0_landed = false;
        for (int it = it_begin; it < it_end && ok; ++it) {
          const Item w = item_at(it);
          const int ii = it - it_begin;
          // this item's Q
          ok = __all_sync(0xffffffffu, wait_or_abort(bar(PB_Q), ii & 1, abort_flag, a.err));
          if (!ok) break;
          q0_landed = true;
          ok = __all_sync(0xffffffffu, wait_fast(bar(PB_KF + jg % NSK), (jg / NSK) & 1, abort_flag, a.err));
          if (!ok) break;
          tc_fence_after();
          issue_qk(0, jg);
          issue_qk(1, jg);
          for (int j = 0; j < w.n_tiles && ok; ++j, ++jg) {
            const bool more = j + 1 < w.n_tiles;
            for (int hh = 0; hh < 2 && ok; ++hh) {
              ok = __all_sync(0xffffffffu, wait_fast(bar(PB_PF + 2 * hh), jg & 1, abort_flag, a.err));
              if (!ok) break;
              tc_fence_after();
              if (hh == 0) ok = __all_sync(0xffffffffu, wait_fast(bar(PB_VF + jg % NSV), (jg / NSV) & 1, abort_flag, a.err));
              if (!ok) break;
              issue_pv(hh, jg, j, w.n_tiles, 0);
              ok = __all_sync(0xffffffffu, wait_fast(bar(PB_PF + 2 * hh + 1), jg & 1, abort_flag, a.err));
              if (!ok) break;
              tc_fence_after();
              issue_pv(hh, jg, j, w.n_tiles, 1);
              if (hh == 1) commit_e(bar(PB_VE + jg % NSV));   // V no longer needed
              if (more) {
                if (hh == 0) ok = __all_sync(0xffffffffu, wait_fast(bar(PB_KF + (jg + 1) % NSK), ((jg + 1) / NSK) & 1, abort_flag, a.err));
                if (!ok) break;
                issue_qk(hh, jg + 1);
              }
            }
          }
        }
        // after an abort, let the first item's Q load (issued above) land
        if (!q0_landed) mbar_wait(bar(PB_Q), 0, nullptr);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoft));
    // ------------------------------------------------------------- softmax (head hh)
    const int hh = warp >> 2;               // 0: warps 0-3, 1: warps 4-7
    const int r = tid & 127;                // query row in the tile, TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t col_s = COL_S + hh * BN, col_o = COL_O + hh * HD;
    const float sl2 = a.scale * 1.4426950408889634f;
    int jg = 0;                             // tile position over all items
    for (int it = it_begin; it < it_end; ++it) {
    const Item w = item_at(it);
    const int q0 = w.qrow[hh], head = w.head[hh];
    const int row_pos = a.prior_len + q0 + r;
    float m_run = -INFINITY, l_run = 0.f;   // running max in scaled log2 units
    for (int j = 0; j < w.n_tiles; ++j, ++jg) {
      wait_fast(bar(PB_SF + hh), jg & 1, abort_flag, a.err);
      __syncwarp();
      tc_fence_after();
      // the S_B commit follows both heads' Q K^T: this K stage can be refilled
      if (hh == 1 && lane == 0) mbar_arrive(bar(PB_KE + jg % NSK));
      const int k0 = j * BN;
      const bool diag = k0 + BN - 1 > a.prior_len + q0;   // causal mask needed
      // the whole S row into registers: four loads in flight, one wait
      float t[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(lane_base + col_s + c * 32, t[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) reg_fence(t[c]);
      if (diag) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (k0 + c * 32 + i > row_pos) t[c][i] = -INFINITY;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          mx4[0] = fmax3(mx4[0], t[c][i], t[c][i + 4]);
          mx4[1] = fmax3(mx4[1], t[c][i + 1], t[c][i + 5]);
          mx4[2] = fmax3(mx4[2], t[c][i + 2], t[c][i + 6]);
          mx4[3] = fmax3(mx4[3], t[c][i + 3], t[c][i + 7]);
        }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
      float m_new = m_run;
      if (mx > m_run + kLazyP || m_run == -INFINITY) m_new = mx;
      const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds P V of the tiles before; the S_h commit of this tile was
        // issued behind their last product, so that product is complete and
        // O can be rescaled in place
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float o[32];
          tmem_ld32(lane_base + col_o + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(lane_base + col_o + c * 32, o);
        }
        tmem_wait_st();
      }
      // p = 2^(s*scale*log2e - m), written as bf16 pairs over the first 64
      // columns of S
      float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
      const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m_new, -m_new);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = ffma2(make_float2(t[c][i], t[c][i + 1]), sl2x2, negm);
          const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          sum2[(i >> 1) & 3] = fadd2(sum2[(i >> 1) & 3], pp);
          pk[i / 2] = pack_bf16(pp.x, pp.y);
        }
        tmem_st16(lane_base + col_s + c * 16, pk);
        if (c & 1) {                        // a half of P is in TMEM
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(PB_PF + 2 * hh + (c >> 1)));
        }
      }
      const float2 s01 = fadd2(sum2[0], sum2[1]), s23 = fadd2(sum2[2], sum2[3]);
      const float sum0 = s01.x + s23.x, sum1 = s01.y + s23.y;
      l_run = l_run * alpha + (sum0 + sum1);
      m_run = m_new;
    }
    wait_or_abort(bar(PB_OD + hh), (it - it_begin) & 1, abort_flag, a.err);
    __syncwarp();
    tc_fence_after();
    const float inv = 1.f / l_run;
    const bool row_ok = (q0 + r) < a.chunk_len;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                          ((int64_t)(q0 + r) * a.num_q_heads + head) * HD;
#pragma unroll 1
    for (int c = 0; c < HD / 32; ++c) {
      float o[32];
      tmem_ld32(lane_base + col_o + c * 32, o);
      tmem_wait_ld();
      reg_fence(o);
      if (row_ok) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 v = make_uint4(pack_bf16(o[i] * inv, o[i + 1] * inv),
                               pack_bf16(o[i + 2] * inv, o[i + 3] * inv),
                               pack_bf16(o[i + 4] * inv, o[i + 5] * inv),
                               pack_bf16(o[i + 6] * inv, o[i + 7] * inv));
          *reinterpret_cast<uint4*>(orow + c * 32 + i) = v;
        }
      }
    }
    }                                       // items
    tc_fence_before();
  }
  __syncthreads();
  if (tid == 0) span_mark(a.span, true);
  if (warp == W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemColsPair));
  }
}

}  // namespace

namespace {
// rows mode (two query tiles of one head per CTA) unless the group is even
bool rows_mode_for(const PrefillArgs& a) { return (a.num_q_heads / a.num_kv_heads) % 2 != 0; }
int items_for(const PrefillArgs& a) {
  const int q_tiles = (a.chunk_len + BM - 1) / BM;
  return rows_mode_for(a) ? a.num_q_heads * ((q_tiles + 1) / 2) : a.num_q_heads / 2 * q_tiles;
}
}  // namespace

// Items -> P persistent CTAs.  Item costs are their key tiles plus one for
// the fixed part (its queries, its epilogue).  Greedy longest-first leaves the
// largest load up to 12% above the mean at some CTA counts (42 CTAs for the
// 2,048-token chunk over 4,096 cached tokens: 276 against 247 tiles); then,
// while it lowers the largest load, one item moves from the most loaded CTA
// to another, or two items are swapped, with both new loads below the old
// maximum.  That reaches the mean to within 0.5% at every count from 36 to 47
// CTAs.  The result depends only on the costs and P, so it is kept per shape.
static std::vector<std::vector<int>> assign_items(const std::vector<int>& cost, int P) {
  std::vector<std::vector<int>> per(P);
  std::vector<long> load(P, 0);
  {
    std::vector<int> order(cost.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
    // longest first; among equals the given order (heaviest query tile first)
    std::stable_sort(order.begin(), order.end(),
                     [&](int x, int y) { return cost[x] > cost[y]; });
    std::priority_queue<std::pair<long, int>, std::vector<std::pair<long, int>>, std::greater<>>
        heap;
    for (int c = 0; c < P; ++c) heap.push({0, c});
    for (int it : order) {
      auto top = heap.top();
      heap.pop();
      per[top.second].push_back(it);
      load[top.second] += cost[it];
      heap.push({load[top.second], top.second});
    }
  }
  for (int iter = 0; iter < 20000; ++iter) {
    const int a = (int)(std::max_element(load.begin(), load.end()) - load.begin());
    const long M = load[a];
    long best = M;
    int bj = -1, bx = -1, by = -1;   // by < 0: a move
    for (int j = 0; j < P; ++j) {
      if (j == a) continue;
      for (int xi = 0; xi < (int)per[a].size(); ++xi) {
        const int x = cost[per[a][xi]];
        if (load[j] + x < M && load[a] - x < M && std::max(load[j] + x, load[a] - x) < best) {
          best = std::max(load[j] + x, load[a] - x);
          bj = j, bx = xi, by = -1;
        }
        for (int yi = 0; yi < (int)per[j].size(); ++yi) {
          const int d = x - cost[per[j][yi]];
          if (d <= 0) continue;
          if (load[j] + d < M && load[a] - d < M && std::max(load[j] + d, load[a] - d) < best) {
            best = std::max(load[j] + d, load[a] - d);
            bj = j, bx = xi, by = yi;
          }
        }
      }
    }
    if (bj < 0) break;
    const int x = per[a][bx];
    per[a].erase(per[a].begin() + bx);
    per[bj].push_back(x);
    load[a] -= cost[x];
    load[bj] += cost[x];
    if (by >= 0) {
      const int y = per[bj][by];
      per[bj].erase(per[bj].begin() + by);
      per[a].push_back(y);
      load[bj] -= cost[y];
      load[a] += cost[y];
    }
  }
  for (auto& v : per)   // each CTA runs its items longest first
    std::stable_sort(v.begin(), v.end(), [&](int x, int y) { return cost[x] > cost[y]; });
  return per;
}

bool prefill_pair_persistent_ok(const PrefillArgs& a, int ctas) {
  return items_for(a) <= kMaxItems && ctas >= 1 && ctas <= kMaxCtas;
}

cudaError_t launch_prefill_pair(const PrefillArgs& a, cudaStream_t stream, int persistent_ctas) {
  PairParams p;
  p.a = a;
  p.total_len = a.prior_len + a.chunk_len;
  const int64_t kv_rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  if (kv_rows >= (1ll << 31) - 1) return cudaErrorInvalidValue;
  p.kv_rows = (int)kv_rows;
  p.q_tiles = (a.chunk_len + BM - 1) / BM;
  if (p.q_tiles == 0) return cudaSuccess;
  CUtensorMap tm_q;
  if (!encode_rows_map_bf16(&tm_q, a.q, a.chunk_len, a.num_q_heads)) return cudaErrorInvalidValue;
  cudaError_t e = allow_dynamic_smem(prefill_pair_kernel, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  p.rows_mode = rows_mode_for(a) ? 1 : 0;
  const int n_x = p.rows_mode ? a.num_q_heads : a.num_q_heads / 2;
  const int n_t = p.rows_mode ? (p.q_tiles + 1) / 2 : p.q_tiles;
  const int n_items = items_for(a);
  const int P = persistent_ctas < n_items ? persistent_ctas : n_items;
  p.n_list = 0;
  if (persistent_ctas > 0 && n_items <= kMaxItems && P <= kMaxCtas) {
    // the items' assignment to the P persistent CTAs, kept per shape
    using Key = std::tuple<int, int, int, int, int>;
    static std::mutex mu;
    static std::map<Key, std::vector<std::vector<int>>> cache;
    const Key key{a.prior_len, a.chunk_len, n_x, (int)p.rows_mode, P};
    std::vector<std::vector<int>> per;
    {
      std::lock_guard<std::mutex> lock(mu);
      auto f = cache.find(key);
      if (f != cache.end()) {
        per = f->second;
      } else {
        // item tq * n_x + x: query tile (pair) tq of head (pair) x
        std::vector<int> cost(n_items);
        for (int tq = 0; tq < n_t; ++tq) {
          const int last_row = p.rows_mode ? (2 * tq + 2) * BM : (tq + 1) * BM;
          const int n_tiles = (a.prior_len + std::min(a.chunk_len, last_row) - 1) / BN + 1;
          for (int x = 0; x < n_x; ++x) cost[tq * n_x + x] = n_tiles + 1;
        }
        per = assign_items(cost, P);
        if (cache.size() >= 256) cache.clear();
        cache.emplace(key, per);
      }
    }
    int k = 0;
    for (int c = 0; c < P; ++c) {
      p.start[c] = (uint16_t)k;
      for (int item : per[c]) p.list[k++] = (uint16_t)item;
    }
    p.start[P] = (uint16_t)k;
    p.n_list = n_items;
    prefill_pair_kernel<<<P, kThreadsPair, SMEM_BYTES, stream>>>(p, tm_q);
    return cudaGetLastError();
  }
  dim3 grid(n_x, n_t);
  prefill_pair_kernel<<<grid, kThreadsPair, SMEM_BYTES, stream>>>(p, tm_q);
  return cudaGetLastError();
}

}  // namespace pkv
