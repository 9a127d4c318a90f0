// Paged grouped-query decode attention on warp-level bf16 tensor-core tiles
// (mma.sync m16n8k16, fp32 accumulate) for sm_103a.
//
// What it computes ("KV cache and continuous batching: 1,000 people ask AI",
// section "What does a KV cache keep?"; "The KV cache and prefix caching",
// section "What prefill stores and decode reads"): for each sequence b and
// query head h, out[b][h] = softmax(scale * q[b][h] . K_b^T) V_b over every
// key and value the sequence has stored, with K_b, V_b those of KV head
// h / G, read through the sequence's block table.
//
// The work is HBM-bound: every cached byte is read once and used for 2*G
// multiply-adds.  For a GQA group the score and value products are small
// dense contractions, done per 16-token block on warp-level m16n8k16 tiles
// with the keys as the M side and the G query heads as the N side (8 columns,
// or 16 for G = 16):
//   S^T = K . Q^T   (A = K, 16 keys x 16 dims; B = Q^T)
//   O^T = V^T . P^T (A = V^T, 16 dims x 16 keys; B = P^T)
// which is 8 + 8 products per block for G <= 8.
//
// Structure (per CTA: one TMA producer warp + four consumer warps, persistent
// over streams; run alone on a large enough batch, or beside a prefill with
// grouped stages (below), each CTA takes an equal share of all streams'
// stages and a stream cut between CTAs leaves one partial per piece;
// otherwise units of 512-token splits go round-robin to the CTAs):
//  * Grouped stages, when the KV heads form groups of four: a stream is
//    (sequence, group of four KV heads) and a stage is one 16-token block of
//    all four heads (16 KiB of K and 16 KiB of V, contiguous in the pool), so
//    consumer warp w follows KV head w of the group through every block of a
//    unit and writes its result itself.  Otherwise a stream is (sequence, KV
//    head) and a stage is four consecutive blocks of that head; warp w takes
//    block w, and the four warps merge at the end of a unit.  The grouped
//    layout measured faster: 435 -> 432 us per layer alone on the ragged
//    batch, 95.0 -> 94.0-94.5 us on the 2,301-token batch, and 490 -> 483 us
//    per layer beside the prefill (at that split's best SM count).
//  * The producer streams each (block, head) tile's K and V with 2-D TMA
//    tensor copies (two 64-column halves each, 128-byte swizzle) into a
//    2-stage ring of four tiles per stage, completing on mbarriers.  It runs
//    ahead across unit boundaries.  With 128 registers per thread and 75 KB of
//    shared memory, three CTAs (12 consumer warps) share an SM for G <= 4.
//  * Consumer warp w takes tile w of every stage.  Each lane loads its share
//    of K straight into A fragments with 16-byte shared loads: the order of
//    the contraction over head dims is permuted per lane (q is loaded with
//    the same permutation) so that the loads are contiguous and free of bank
//    conflicts.  The V pairs of the transposed A fragment are assembled from
//    two key rows with byte permutes, the output dims being permuted to match.
//    P moves from the S^T accumulator layout to the B layout with movmatrix.
//  * Online softmax per head: the running max (log2 domain) only has to bound
//    the scores to within 2^8, so a warp vote decides whether any score
//    exceeds it; only then is the exact max reduced over the block's keys.
//  * Each warp keeps its own (m, l, O) for its tiles; with per-head stages the
//    four warps merge through shared memory at the end of a unit.  A unit
//    that covers its whole sequence writes the output; otherwise it writes
//    (m, l, O) partials that the reduce kernel merges.
//  * Keys past the end of a sequence are masked before the softmax, and the
//    matching V values are zeroed in registers, so stale pool contents (even
//    NaN) never reach the output.
#include <cuda.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "host_cache.h"
#include "launch.h"
#include "tmap.h"

namespace pkv {
namespace {

constexpr int kCW = 4;                           // consumer warps
constexpr int kConsumersM = kCW * 32;
constexpr int kThreadsM = kConsumersM + 32;
constexpr int kBPS = kCW;                        // blocks per stage: one per consumer warp
constexpr int kStageTok = kBPS * kBlockSize;     // 64 tokens
constexpr int kHalfB = kBlockSize * 128;         // 16 rows x 128 B: one 64-column half
constexpr int kTileB = 2 * kHalfB;               // one block of K (or V), 4 KiB
constexpr int kStageB = 2 * kBPS * kTileB;       // K and V of a stage, 32 KiB
constexpr int kNST = 2;
constexpr int kRingB = kNST * kStageB;
constexpr int kHD = 128;
constexpr int kCombRowM = kHD + 4;               // padded row of the merge buffer
constexpr float kLazyM = 8.0f;
constexpr unsigned kAllM = 0xffffffffu;

static_assert(kSplitTokens % kStageTok == 0, "a split holds whole stages");
static_assert(32 % kBPS == 0, "a stage never straddles two block-id windows");

template <int G>
struct MCfg {
  static constexpr int NT = (G + 7) / 8;                      // head tiles of 8
  static constexpr int COMB_B = kCW * G * kCombRowM * 4;      // merged O per warp
  static constexpr int ML_B = kCW * G * 2 * 4;
  static constexpr int OFF_COMB = kRingB;
  static constexpr int OFF_ML = OFF_COMB + COMB_B;
  static constexpr int OFF_BAR = OFF_ML + ML_B;
  static constexpr int OFF_CU = OFF_BAR + 2 * kNST * 8 + 16;
  static_assert(G >= 1 && G <= 16 && (G & (G - 1)) == 0, "group of 1..16 heads");
};

// transpose of an 8x8 16-bit tile held as one m8n8 fragment per lane
__device__ __forceinline__ uint32_t movm_t16(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}
__device__ __forceinline__ uint32_t prmt16(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// 2^x by the MUFU approximation (subnormal results flush to zero)
__device__ __forceinline__ float ex2m(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint4 lds128m(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// D (16x8 fp32) += A (16x16 bf16, row) . B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void tma2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                           int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// byte offset of (row, 16-byte chunk c of 16) inside one 128B-swizzled tile
__device__ __forceinline__ uint32_t sw_off(int row, int c) {
  return (uint32_t)((c >> 3) * kHalfB + row * 128 + (((c & 7) ^ (row & 7)) << 4));
}

// Two fp16 values to global memory in one 4-byte store with an L2 policy.
__device__ __forceinline__ void st_global_hint_f16x2(__half* dst, float lo, float hi,
                                                     uint64_t policy) {
  const __half2 v = __floats2half2_rn(lo, hi);
  asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(dst),
               "r"(*reinterpret_cast<const uint32_t*>(&v)), "l"(policy)
               : "memory");
}

// G: query heads per KV head.  FUSE: each sequence's new key and value are
// appended in the same launch.  HS (grouped stages): a stage is one block of
// a group of kBPS KV heads, warp w following head w; otherwise kBPS blocks of
// one KV head, merged across the warps at each unit's end.
template <int G, bool FUSE, bool HS>
__global__ void __launch_bounds__(kThreadsM, G <= 8 ? 3 : 2)
decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v) {
  using C = MCfg<G>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  float* comb = reinterpret_cast<float*>(smem + C::OFF_COMB);   // [kCW][G][128]
  float* comb_ml = reinterpret_cast<float*>(smem + C::OFF_ML);  // [kCW][G][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  int* abort_flag = reinterpret_cast<int*>(bars + 2 * kNST);
  int* cu = reinterpret_cast<int*>(smem + C::OFF_CU);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kNST);

  if (tid == 0) {
    span_mark(a.span, false);
    for (int i = 0; i < kNST; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kCW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // The walk's streams: (sequence, group of kBPS KV heads) with one
  // 16-token block per stage (HS), or (sequence, KV head) with kBPS blocks
  // per stage.  Balanced walk when the batch gives every CTA at least 512
  // tokens of stages; otherwise 512-token splits.
  DecodeArgs aw = a;
  if (HS) aw.num_kv_heads = a.num_kv_heads / kBPS;
  constexpr int kWalkTok = HS ? kBlockSize : kStageTok;
  // the sequence lengths after the prefix sums, when the launcher made room
  int* lens = a.lens_in_smem ? cu + a.num_seqs + 1 : nullptr;
  plan_units(aw, cu, a.balanced ? kWalkTok : 0, 0, lens);
  __syncthreads();
  const bool balanced =
      a.balanced && (int64_t)cu[a.num_seqs] >= (int64_t)(kSplitTokens / kWalkTok) * gridDim.x;
  if (a.balanced && !balanced) {
    __syncthreads();
    plan_units(aw, cu, 0, 0, lens);
    __syncthreads();
  }
  volatile int* vabort = abort_flag;

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
#ifdef PKV_TEST_WAIT_TIMEOUT
    // Test build only: the producer withholds every stage before issuing any
    // copy.  The consumers' first waits then run out with nothing in flight;
    // they record PKV_DEVERR_TIMEOUT, skip every later wait, and the kernel
    // returns.
    return;
#endif
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
    }
    const uint64_t policy = policy_evict_first();
    uint32_t issued = 0;
    bool ok = true;
    Walk wk = walk_begin(aw, cu, balanced, lens);
    Unit u;
    while (ok && walk_next(aw, cu, kWalkTok, wk, u)) {
      const int blk0 = u.tok_begin / kBlockSize;
      const int nblk = (u.tok_end - 1) / kBlockSize - blk0 + 1;
      const int32_t* bt_row = a.block_table + (int64_t)u.b * a.bt_stride + blk0;
      int my_blk = 0;
      const int nst = HS ? nblk : (nblk + kBPS - 1) / kBPS;
      for (int st = 0; st < nst; ++st, ++issued) {
        const int bps = HS ? 1 : kBPS;   // blocks per stage
        if ((st * bps) % 32 == 0) {  // next window of 32 block ids, one per lane
          const int idx = st * bps + lane;
          my_blk = 0;
          if (idx < nblk) {
            my_blk = __ldg(bt_row + idx);
            if (my_blk < 0 || (int64_t)my_blk >= a.num_blocks) {
              record_error(a.err, DEVERR_BLOCK_RANGE);
              my_blk = 0;  // read a valid block instead; the error word reports it
            }
          }
        }
        const int buf = issued % kNST;
        const uint32_t phase = (issued / kNST) & 1;
        if (lane == 0 && issued >= (uint32_t)kNST && !*vabort) {
          if (!mbar_wait(empty0 + 8 * buf, phase ^ 1, a.err)) *vabort = 1;
        }
        __syncwarp();
        if (*vabort) { ok = false; break; }
        // tile i of the stage: HS, head u.g * kBPS + i of the stage's block;
        // otherwise block st * kBPS + i of head u.g
        const int nb = HS ? kBPS : min(kBPS, nblk - st * kBPS);
        int rows[kBPS];
#pragma unroll
        for (int i = 0; i < kBPS; ++i)
          rows[i] = HS ? (__shfl_sync(kAllM, my_blk, st & 31) * a.num_kv_heads + u.g * kBPS + i) *
                             kBlockSize
                       : (__shfl_sync(kAllM, my_blk, (st * kBPS + i) & 31) * a.num_kv_heads + u.g) *
                             kBlockSize;
        if (lane == 0) {
          const uint32_t fb = full0 + 8 * buf;
          mbar_arrive_expect_tx(fb, (uint32_t)(nb * 2 * kTileB));
          const uint32_t kdst = sbase + buf * kStageB, vdst = kdst + kBPS * kTileB;
#pragma unroll
          for (int i = 0; i < kBPS; ++i) {
            if (i < nb) {
              tma2d_hint(kdst + i * kTileB, &tm_k, fb, 0, rows[i], policy);
              tma2d_hint(kdst + i * kTileB + kHalfB, &tm_k, fb, 64, rows[i], policy);
              tma2d_hint(vdst + i * kTileB, &tm_v, fb, 0, rows[i], policy);
              tma2d_hint(vdst + i * kTileB + kHalfB, &tm_v, fb, 64, rows[i], policy);
            }
          }
        }
      }
    }
    if (!ok && lane == 0) {  // on abort, let the copies already issued land
      const uint32_t first = issued > (uint32_t)kNST ? issued - kNST : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait(full0 + 8 * (i % kNST), (i / kNST) & 1, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  constexpr int NT = C::NT;
  const int g = lane >> 2, t = lane & 3;
  const float sl2 = a.scale * 1.4426950408889634f;
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
  // this lane's K / q pieces: load step i takes the 16-byte chunk kc(i) of
  // the 64-column half (t >> 1); dims 64 * (t >> 1) + 8 * kc(i) + 0..7 feed
  // the k-steps 2i and 2i + 1
  const int khalf = t >> 1;
  const int kc0 = 4 * (t & 1), kx = (t >> 1) << 1;
  // V pieces: half g >> 2, chunk 2 * (g & 3) + (j ^ (g & 1)), i.e. dims
  // 16g + 8 * (j ^ (g & 1)) + 0..7 of the key rows 2t, 2t+1, 2t+8, 2t+9
  const int vhalf = g >> 2;
  uint32_t consumed = 0;

  Walk wk = walk_begin(aw, cu, balanced, lens);
  Unit u;
  while (walk_next(aw, cu, kWalkTok, wk, u)) {
    const int head = HS ? u.g * kBPS + warp : u.g;   // this warp's KV head
    const int hq0 = head * G;
    // the merge reads how many partials this (sequence, KV head) left
    if (a.balanced && u.s == 0 && (HS ? lane == 0 : tid == 0))
      a.ws_np[u.b * a.num_kv_heads + head] = u.ns;
    // Q^T as B fragments of head 8nt + g, in the lane's K order
    uint4 qf[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hh = 8 * nt + g;
      const __nv_bfloat16* qrow =
          static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)u.b * a.num_q_heads + hq0 + hh) * kHD;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qf[nt][i] = hh < G ? __ldg(reinterpret_cast<const uint4*>(qrow + 64 * khalf + 8 * (kc0 + (i ^ kx))))
                           : make_uint4(0, 0, 0, 0);
    }
    // O^T accumulators: o[nt][mt] holds dims d(mt), d(mt) + 1 (c0/c1, c2/c3)
    // with d(mt) = 16g + 8 * ((mt >> 2) ^ (g & 1)) + 2 * (mt & 3), for heads
    // 8nt + 2t (c0, c2) and 8nt + 2t + 1 (c1, c3)
    float o[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
    float m_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
    }

    const int nblk = (u.tok_end - 1) / kBlockSize - u.tok_begin / kBlockSize + 1;
    const int nst = HS ? nblk : (nblk + kBPS - 1) / kBPS;
    for (int st = 0; st < nst; ++st, ++consumed) {
      const int buf = consumed % kNST;
      const uint32_t phase = (consumed / kNST) & 1;
      if (!*vabort) {
        if (!mbar_wait(full0 + 8 * buf, phase, a.err)) *vabort = 1;
      }
      const int tok0 = u.tok_begin + (HS ? st : st * kBPS + warp) * kBlockSize;
      const int valid = min(kBlockSize, u.tok_end - tok0);   // keys of this warp's block
      if (valid <= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * buf);
        continue;
      }
      const uint32_t kt = sbase + buf * kStageB + warp * kTileB;
      const uint32_t vt = kt + kBPS * kTileB;
      if (FUSE && u.s == u.ns - 1 && tok0 + valid == u.tok_end) {
        // this block holds the sequence's new token (position tok_end - 1):
        // the staged tile still has the pool's old row there, so put the new
        // key and value into shared memory and into the pool.  Lanes 0-15
        // move the 16-byte chunks of K, lanes 16-31 those of V.
        const int r = valid - 1;
        const int c = lane & 15;
        const bool is_v = lane >= 16;
        const int64_t src = (((int64_t)u.b * a.num_kv_heads + head) * kHD) + c * 8;
        const uint4 val = __ldg(reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(is_v ? a.v_new : a.k_new) + src));
        unsigned char* tile = smem + buf * kStageB + (is_v ? kBPS * kTileB : 0) + warp * kTileB;
        *reinterpret_cast<uint4*>(tile + sw_off(r, c)) = val;
        const int blk = __ldg(a.block_table + (int64_t)u.b * a.bt_stride + (tok0 / kBlockSize));
        if (blk >= 0 && (int64_t)blk < a.num_blocks) {
          __nv_bfloat16* pool = const_cast<__nv_bfloat16*>(
              static_cast<const __nv_bfloat16*>(is_v ? a.v_cache : a.k_cache));
          const int64_t dst = (((int64_t)blk * a.num_kv_heads + head) * kBlockSize + r) * kHD + c * 8;
          *reinterpret_cast<uint4*>(pool + dst) = val;
        }
        // order these generic-proxy writes before the TMA refill of this slot
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      // ---- K of keys g and g + 8, straight into A fragments
      uint4 kg[4], kh[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = kc0 + (i ^ kx);
        kg[i] = lds128m(kt + khalf * kHalfB + g * 128 + ((c ^ g) << 4));
        kh[i] = lds128m(kt + khalf * kHalfB + (g + 8) * 128 + ((c ^ g) << 4));
      }
      // ---- S^T = K . Q^T: two dependent chains of four products
      float s[NT][4], s2[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = s2[nt][i] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816(s[nt], kg[i].x, kh[i].x, kg[i].y, kh[i].y, qf[nt][i].x, qf[nt][i].y);
          mma16816(s2[nt], kg[i].z, kh[i].z, kg[i].w, kh[i].w, qf[nt][i].z, qf[nt][i].w);
        }
      // ---- V of keys 2t, 2t+1, 2t+8, 2t+9; then the slot is free
      uint4 va[2], vb[2], vc[2], vd[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = 2 * (g & 3) + (j ^ (g & 1));
        const uint32_t base = vt + vhalf * kHalfB;
        va[j] = lds128m(base + (2 * t) * 128 + ((c ^ (2 * t)) << 4));
        vb[j] = lds128m(base + (2 * t + 1) * 128 + ((c ^ (2 * t + 1)) << 4));
        vc[j] = lds128m(base + (2 * t + 8) * 128 + ((c ^ (2 * t)) << 4));
        vd[j] = lds128m(base + (2 * t + 9) * 128 + ((c ^ (2 * t + 1)) << 4));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] += s2[nt][i];

      // ---- online softmax per head; this lane holds keys g, g+8 of heads 2t, 2t+1
      const bool k0ok = g < valid, k1ok = g + 8 < valid;
      float v[NT][4];
      bool grow = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[nt][i] = (i < 2 ? k0ok : k1ok) ? s[nt][i] * sl2 : -INFINITY;
          grow |= v[nt][i] > m_run[nt][i & 1] + kLazyM;
        }
      if (__any_sync(kAllM, grow)) {
        bool rescale = false;
        float alpha[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(v[nt][j], v[nt][j + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(kAllM, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kAllM, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kAllM, mx, 16));
            float m_new = m_run[nt][j];
            if (mx > m_new + kLazyM || m_new == -INFINITY) m_new = mx;
            alpha[nt][j] = (m_new == m_run[nt][j]) ? 1.f : ex2m(m_run[nt][j] - m_new);
            rescale |= alpha[nt][j] != 1.f;
            m_run[nt][j] = m_new;
          }
        if (__any_sync(kAllM, rescale)) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            l_run[nt][0] *= alpha[nt][0];
            l_run[nt][1] *= alpha[nt][1];
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o[nt][mt][0] *= alpha[nt][0];
              o[nt][mt][1] *= alpha[nt][1];
              o[nt][mt][2] *= alpha[nt][0];
              o[nt][mt][3] *= alpha[nt][1];
            }
          }
        }
      }
      uint32_t pb0[NT], pb1[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // bf16 weights (what P.V multiplies; the sum uses the same values)
        const uint32_t x0 = pack2_bf16(ex2m(v[nt][0] - m_run[nt][0]), ex2m(v[nt][1] - m_run[nt][1]));
        const uint32_t x1 = pack2_bf16(ex2m(v[nt][2] - m_run[nt][0]), ex2m(v[nt][3] - m_run[nt][1]));
        l_run[nt][0] += bf16lo(x0) + bf16lo(x1);
        l_run[nt][1] += bf16hi(x0) + bf16hi(x1);
        pb0[nt] = movm_t16(x0);   // head g: keys 2t, 2t+1
        pb1[nt] = movm_t16(x1);   // head g: keys 2t+8, 2t+9
      }

      // ---- O^T += V^T . P^T; V of keys past the end becomes +0
      if (valid < kBlockSize) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (2 * t >= valid) va[j] = make_uint4(0, 0, 0, 0);
          if (2 * t + 1 >= valid) vb[j] = make_uint4(0, 0, 0, 0);
          if (2 * t + 8 >= valid) vc[j] = make_uint4(0, 0, 0, 0);
          if (2 * t + 9 >= valid) vd[j] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t aw[4] = {va[j].x, va[j].y, va[j].z, va[j].w};
        const uint32_t bw[4] = {vb[j].x, vb[j].y, vb[j].z, vb[j].w};
        const uint32_t cw[4] = {vc[j].x, vc[j].y, vc[j].z, vc[j].w};
        const uint32_t dw[4] = {vd[j].x, vd[j].y, vd[j].z, vd[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t a0 = prmt16(aw[e], bw[e], 0x5410u);   // keys 2t, 2t+1 at dim d
          const uint32_t a1 = prmt16(aw[e], bw[e], 0x7632u);   // ... at dim d + 1
          const uint32_t a2 = prmt16(cw[e], dw[e], 0x5410u);   // keys 2t+8, 2t+9 at dim d
          const uint32_t a3 = prmt16(cw[e], dw[e], 0x7632u);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(o[nt][4 * j + e], a0, a1, a2, a3, pb0[nt], pb1[nt]);
        }
      }
    }

    // ---- l summed over the lanes of each head
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        l_run[nt][j] += __shfl_xor_sync(kAllM, l_run[nt][j], 4);
        l_run[nt][j] += __shfl_xor_sync(kAllM, l_run[nt][j], 8);
        l_run[nt][j] += __shfl_xor_sync(kAllM, l_run[nt][j], 16);
      }
    const bool direct = (u.ns == 1);
    // keep_partials: partials stay in L2 (evict-last) until the merge reads
    // and drops them
    const uint64_t keep = a.keep_partials ? policy_evict_last() : policy_evict_normal();
    if constexpr (HS) {
      // this warp saw every key of the unit for its own heads: O / l goes out
      // straight from the accumulators (dims d, d + 1 per lane and tile)
      __half* ws_half = reinterpret_cast<__half*>(a.ws_acc);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int hh = 8 * nt + 2 * t + j;
          if (hh < G) {
            const float rl = 1.f / l_run[nt][j];
            const int64_t row = (int64_t)u.b * a.num_q_heads + hq0 + hh;
            const int64_t pidx = row * a.max_splits + u.s;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const int d = 16 * g + 8 * ((mt >> 2) ^ (g & 1)) + 2 * (mt & 3);
              const float x0 = o[nt][mt][j] * rl, x1 = o[nt][mt][j + 2] * rl;
              if (direct)
                *reinterpret_cast<__nv_bfloat162*>(outp + row * kHD + d) = __floats2bfloat162_rn(x0, x1);
              else   // O / l in fp16: half the bytes of the partial's trip through memory
                st_global_hint_f16x2(ws_half + pidx * kHD + d, x0, x1, keep);
            }
            if (!direct && g == 0) {
              a.ws_ml[pidx * 2 + 0] = m_run[nt][j];
              a.ws_ml[pidx * 2 + 1] = l_run[nt][j];
            }
          }
        }
    } else {
      // ---- otherwise merge the four warps of this unit (each saw a quarter
      // of its blocks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int hh = 8 * nt + 2 * t + j;
          if (hh < G) {
            if (g == 0) {
              comb_ml[(warp * G + hh) * 2 + 0] = m_run[nt][j];
              comb_ml[(warp * G + hh) * 2 + 1] = l_run[nt][j];
            }
            float* crow = comb + (warp * G + hh) * kCombRowM + 16 * g;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
              *reinterpret_cast<float2*>(crow + 8 * ((mt >> 2) ^ (g & 1)) + 2 * (mt & 3)) =
                  make_float2(o[nt][mt][j], o[nt][mt][j + 2]);
          }
        }
      named_bar_sync(1, kConsumersM);
      // warp w merges heads w, w + 4, ...: the combine weights once per head,
      // then 4 dims per lane
      for (int h = warp; h < G; h += kCW) {
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kCW; ++k) M = fmaxf(M, comb_ml[(k * G + h) * 2]);
        float wk[kCW], L = 0.f;
#pragma unroll
        for (int k = 0; k < kCW; ++k) {
          const float mk = comb_ml[(k * G + h) * 2];
          wk[k] = (mk == -INFINITY) ? 0.f : ex2m(mk - M);
          L = fmaf(wk[k], comb_ml[(k * G + h) * 2 + 1], L);
        }
        const float rl = 1.f / L;
        const int64_t row = (int64_t)u.b * a.num_q_heads + hq0 + h;
        const int64_t pidx = row * a.max_splits + u.s;
#pragma unroll
        for (int i = 0; i < kHD / 32; ++i) {
          const int d = lane + 32 * i;
          float O = 0.f;
#pragma unroll
          for (int k = 0; k < kCW; ++k) O = fmaf(wk[k], comb[(k * G + h) * kCombRowM + d], O);
          if (direct)
            outp[row * kHD + d] = __float2bfloat16_rn(O * rl);
          else   // O / l in fp16: half the bytes of the partial's trip through memory
            st_global_hint_f16(reinterpret_cast<__half*>(a.ws_acc) + pidx * kHD + d,
                               __float2half_rn(O * rl), keep);
        }
        if (!direct && lane == 0) {
          a.ws_ml[pidx * 2 + 0] = M;
          a.ws_ml[pidx * 2 + 1] = L;
        }
      }
      named_bar_sync(1, kConsumersM);
    }
  }
  // This CTA's work is done: the split merge launched next (a programmatic
  // dependent that waits for this grid to complete before it reads) may be
  // scheduled as SMs free up, instead of after the last CTA has exited.
  if (tid == 0) span_mark(a.span, true);
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched as the programmatic dependent of a persistent prefill on the
  // other SMs, this grid finishes only after that one, so the launches that
  // follow in the stream see both.  Without such a launch it returns at once.
  if (tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int G, bool FUSE, bool HS>
cudaError_t launch_g(const DecodeArgs& args, int num_sms, cudaStream_t stream, bool dependent) {
  using C = MCfg<G>;
  DecodeArgs a = args;
  // Partials kept in L2 (evict-last, dropped by the merge once read), except
  // for per-head stages beside a prefill: their 512-token splits leave some
  // 12 MB of partials a layer, which crowded the prefill's L2-resident K/V
  // (pair 490 -> 498 us).  The balanced walk's few partials do not (pair
  // 470.6-471.3 -> 468.9-470.1 us at 43-44 prefill SMs).
  a.keep_partials = (dependent && !HS) ? 0 : 1;
  a.partials_f16 = 1;
  // The balanced walk, except for the per-head stages beside a prefill,
  // where 512-token splits measured faster.  With a group of kBPS heads per
  // stage a split is four times the bytes, too coarse to share out evenly,
  // and the balanced walk is faster there as well.
  DecodeArgs aw = a;
  if (HS) aw.num_kv_heads = a.num_kv_heads / kBPS;
  a.balanced = a.ws_np != nullptr && (HS || !dependent) &&
               stage_plan_fits(aw, HS ? kBlockSize : kStageTok);
  CUtensorMap tm_k, tm_v;
  const int64_t rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  if (!encode_pool_map_bf16(&tm_k, a.k_cache, rows) || !encode_pool_map_bf16(&tm_v, a.v_cache, rows))
    return cudaErrorInvalidValue;
  size_t smem = C::OFF_CU + sizeof(int) * (size_t)(a.num_seqs + 1) + 1024;
  // the sequence lengths go to shared memory too unless that costs a CTA per SM
  {
    const size_t with = smem + sizeof(int) * (size_t)a.num_seqs;
    a.lens_in_smem = with <= 227 * 1024 &&
                     (228 * 1024) / (with + 1024) >= (228 * 1024) / (smem + 1024);
    if (a.lens_in_smem) smem = with;
  }
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = allow_dynamic_smem(decode_mma_kernel<G, FUSE, HS>, (int)smem);
  if (e != cudaSuccess) return e;
  const int by_smem = (int)((228 * 1024) / (smem + 1024));
  const int per_sm = by_smem < 1 ? 1 : (by_smem > (G <= 8 ? 3 : 2) ? (G <= 8 ? 3 : 2) : by_smem);
  const int64_t upper = (int64_t)a.num_seqs * a.num_kv_heads * a.max_splits;
  const int grid = (int)(upper < (int64_t)num_sms * per_sm ? upper : (int64_t)num_sms * per_sm);
  if (dependent) {
    // programmatic dependent launch: may start while the previous kernel in
    // the stream (a persistent prefill holding its own SMs) still runs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsM);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_mma_kernel<G, FUSE, HS>, a, tm_k, tm_v);
    if (e != cudaSuccess) return e;
  } else {
    decode_mma_kernel<G, FUSE, HS><<<grid, kThreadsM, smem, stream>>>(a, tm_k, tm_v);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  return launch_decode_reduce_bf16_128(a, stream);
}

}  // namespace

bool decode_mma_supported(int is_bf16, int head_dim, int group) {
  return is_bf16 && head_dim == 128 &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_paged_decode_mma(const DecodeArgs& a, int num_sms, cudaStream_t stream,
                                    bool dependent) {
  if (a.chunk_prior >= 0 || a.split_tokens % kStageTok != 0) return cudaErrorInvalidValue;
  const bool fuse = a.k_new != nullptr;
  // one block of kBPS KV heads per stage when the heads form such groups
  const bool hs = a.num_kv_heads % kBPS == 0;
  const int d = dependent;
#define PKV_LAUNCH_G(GG)                                                            \
  return hs ? (fuse ? launch_g<GG, true, true>(a, num_sms, stream, d)               \
                    : launch_g<GG, false, true>(a, num_sms, stream, d))             \
            : (fuse ? launch_g<GG, true, false>(a, num_sms, stream, d)              \
                    : launch_g<GG, false, false>(a, num_sms, stream, d))
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: PKV_LAUNCH_G(1);
    case 2: PKV_LAUNCH_G(2);
    case 4: PKV_LAUNCH_G(4);
    case 8: PKV_LAUNCH_G(8);
    case 16: PKV_LAUNCH_G(16);
#undef PKV_LAUNCH_G
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
