// Paged grouped-query decode attention over an fp8 (E4M3) KV cache with
// per-KV-head scales, on warp-level f16 tensor-core tiles (sm_103a).
//
// What it computes: the decode attention of decode_mma.cu ("KV cache and
// continuous batching: 1,000 people ask AI", section "What does a KV cache
// keep?"), with every cached key and value stored as an E4M3 code c and read
// as c * scale[kv_head] -- the cache quantisation "The KV cache is not your
// bottleneck" mentions (section "What the profile said"; the pages give no
// format).  The cache is half the bytes of bf16, and decode is HBM-bound.
//
// Same unit structure as the bf16 kernel -- persistent CTAs walking streams
// in equal per-CTA shares of stages, or in 512-token splits for small
// batches; a stage is one 16-token block of a group of four KV heads when the
// heads form such groups (each consumer warp following one head through the
// unit and writing its own result), otherwise four blocks of one KV head
// (merged across the warps at each unit's end); one producer warp streams
// each (block, head) tile of K and V with 2-D TMA (one 16-row x 128-byte box
// each, 128-byte swizzle) into a 4-stage ring, four consumer warps taking one
// tile per stage -- but the products are turned around: keys are the M side
// of the m16n8k16 tile and the G query heads its N side (8 columns, or 16 for
// G = 16), so one block costs 8 + 8 products instead of 16 + 16 with heads
// padded to 16 rows.
//   S^T = K . Q^T   A = K (16 keys x 16 dims), B = Q^T
//   O^T = V^T . P^T A = V^T (16 dims x 16 keys), B = P^T
// Each lane reads its share of the fp8 codes straight from the ring into
// registers and widens them there (E4M3 -> f16 is exact): the contraction
// order over head dimensions and the output order are permuted so that every
// lane's codes are contiguous 16-byte pieces of a key row (dims
// 32t + 4ks + 0..3 of key g for the k-step ks; dims 16g + 2mt, +1 of keys 2t,
// 2t+1, 2t+8, 2t+9 for the M tile mt); the transposed V pairs are assembled
// with byte permutes, and P moves from the S^T accumulator layout to the B
// layout with movmatrix.  The K scale folds into the softmax scale and the V
// scale into the output, so the products see the raw codes.  Keys past a
// sequence's end are masked, and their V codes are zeroed in registers.
#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "host_cache.h"
#include "launch.h"
#include "tmap.h"

namespace pkv {
namespace {

constexpr int kCW = 4;                           // consumer warps
constexpr int kConsumers8 = kCW * 32;
constexpr int kThreads8 = kConsumers8 + 32;
constexpr int kBPS = kCW;                        // blocks per stage: one per consumer warp
constexpr int kStageTok = kBPS * kBlockSize;     // 64 tokens
constexpr int kTile8 = kBlockSize * 128;         // one fp8 (block, head) tile: 16 rows x 128 B
constexpr int kStage8 = 2 * kBPS * kTile8;       // K and V of a stage, 16 KiB
constexpr int kNST8 = 4;
constexpr int kRing8 = kNST8 * kStage8;
constexpr int kHD = 128;
constexpr int kCombRow = kHD + 4;                // padded row of the merge buffer
constexpr float kLazy8 = 8.0f;
constexpr unsigned kAll8 = 0xffffffffu;

static_assert(kSplitTokens % kStageTok == 0, "a split holds whole stages");
static_assert(32 % kBPS == 0, "a stage never straddles two block-id windows");

template <int G>
struct F8Cfg {
  static constexpr int NT = (G + 7) / 8;         // head tiles of 8
  static constexpr int OFF_COMB = kRing8;
  static constexpr int COMB_B = kCW * G * kCombRow * 4;
  static constexpr int OFF_ML = OFF_COMB + COMB_B;
  static constexpr int OFF_BAR = OFF_ML + kCW * G * 2 * 4;
  static constexpr int OFF_CU = OFF_BAR + 2 * kNST8 * 8 + 16;
};

// D (16x8 fp32) += A (16x16 f16, row) . B (16x8 f16, col)
__device__ __forceinline__ void mma16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  return pack2_f16(bf16lo(u), bf16hi(u));
}

__device__ __forceinline__ void tma2d_u8(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                         int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw8(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t lo16_to_f16x2(uint32_t w) {
  return e4m3x2_to_f16x2((uint16_t)(w & 0xffffu));
}
__device__ __forceinline__ uint32_t hi16_to_f16x2(uint32_t w) {
  return e4m3x2_to_f16x2((uint16_t)(w >> 16));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// transpose of an 8x8 f16 tile held as one m8n8 fragment per lane
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}
// 2^x by the MUFU approximation (flushes subnormal results to zero); x is
// never above the lazy-rescale threshold here
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint4 lds128(const unsigned char* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// G: query heads per KV head.  HS (grouped stages): a stage is one block of a
// group of kBPS KV heads, warp w following head w with that head's scales;
// otherwise kBPS blocks of one KV head, merged across the warps at each
// unit's end.
template <int G, bool HS>
__global__ void __launch_bounds__(kThreads8, G <= 8 ? 3 : 2)
decode_fp8_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v) {
  using C = F8Cfg<G>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  float* comb = reinterpret_cast<float*>(smem + C::OFF_COMB);
  float* comb_ml = reinterpret_cast<float*>(smem + C::OFF_ML);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  int* abort_flag = reinterpret_cast<int*>(bars + 2 * kNST8);
  int* cu = reinterpret_cast<int*>(smem + C::OFF_CU);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kNST8);

  if (tid == 0) {
    for (int i = 0; i < kNST8; ++i) {
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
              my_blk = 0;
            }
          }
        }
        const int buf = issued % kNST8;
        const uint32_t phase = (issued / kNST8) & 1;
        if (lane == 0 && issued >= (uint32_t)kNST8 && !*vabort) {
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
          rows[i] = HS ? (__shfl_sync(kAll8, my_blk, st & 31) * a.num_kv_heads + u.g * kBPS + i) *
                             kBlockSize
                       : (__shfl_sync(kAll8, my_blk, (st * kBPS + i) & 31) * a.num_kv_heads + u.g) *
                             kBlockSize;
        if (lane == 0) {
          const uint32_t fb = full0 + 8 * buf;
          mbar_arrive_expect_tx(fb, (uint32_t)(nb * 2 * kTile8));
          const uint32_t kdst = sbase + buf * kStage8, vdst = kdst + kBPS * kTile8;
#pragma unroll
          for (int i = 0; i < kBPS; ++i) {
            if (i < nb) {
              tma2d_u8(kdst + i * kTile8, &tm_k, fb, 0, rows[i], policy);
              tma2d_u8(vdst + i * kTile8, &tm_v, fb, 0, rows[i], policy);
            }
          }
        }
      }
    }
    if (!ok && lane == 0) {
      const uint32_t first = issued > (uint32_t)kNST8 ? issued - kNST8 : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait(full0 + 8 * (i % kNST8), (i / kNST8) & 1, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  constexpr int NT = C::NT;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
  uint32_t consumed = 0;

  Walk wk = walk_begin(aw, cu, balanced, lens);
  Unit u;
  while (walk_next(aw, cu, kWalkTok, wk, u)) {
    const int head = HS ? u.g * kBPS + warp : u.g;   // this warp's KV head
    const int hq0 = head * G;
    // the merge reads how many partials this (sequence, KV head) left
    if (a.balanced && u.s == 0 && (HS ? lane == 0 : tid == 0))
      a.ws_np[u.b * a.num_kv_heads + head] = u.ns;
    const float sl2 = a.scale * __ldg(a.k_scale + head) * 1.4426950408889634f;
    const float vscale = __ldg(a.v_scale + head);
    // Q^T fragments: head 8nt + g, dims 32t + 4ks + {0,1} (b0) and {2,3} (b1)
    uint32_t qf[NT][8][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hh = 8 * nt + g;
      if (hh < G) {
        const uint4* qrow = reinterpret_cast<const uint4*>(
            q32 + ((int64_t)u.b * a.num_q_heads + hq0 + hh) * (kHD / 2) + 16 * t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = __ldg(qrow + i);
          qf[nt][2 * i][0] = bf16x2_to_f16x2(v.x);
          qf[nt][2 * i][1] = bf16x2_to_f16x2(v.y);
          qf[nt][2 * i + 1][0] = bf16x2_to_f16x2(v.z);
          qf[nt][2 * i + 1][1] = bf16x2_to_f16x2(v.w);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) qf[nt][ks][0] = qf[nt][ks][1] = 0u;
      }
    }
    // O^T accumulators: o[nt][mt] = dims 16g + 2mt (+1 in c2, c3), heads 8nt + 2t (+1 in c1, c3)
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
      const int buf = consumed % kNST8;
      const uint32_t phase = (consumed / kNST8) & 1;
      if (!*vabort) {
        if (!mbar_wait(full0 + 8 * buf, phase, a.err)) *vabort = 1;
      }
      const int tok0 = u.tok_begin + (HS ? st : st * kBPS + warp) * kBlockSize;
      const int valid = min(kBlockSize, u.tok_end - tok0);
      uint4 kg0, kg1, kh0, kh1, va, vb, vc, vd;
      if (valid > 0) {
        const unsigned char* k8 = smem + buf * kStage8 + warp * kTile8;
        kg0 = lds128(k8 + sw8(g, 2 * t));
        kg1 = lds128(k8 + sw8(g, 2 * t + 1));
        kh0 = lds128(k8 + sw8(g + 8, 2 * t));
        kh1 = lds128(k8 + sw8(g + 8, 2 * t + 1));
      }
      if (valid <= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * buf);
        continue;
      }

      // ---- S^T = K . Q^T over 8 k-steps of 16 (permuted) head dimensions
      float s[NT][4], s2[NT][4];   // even and odd k-steps: two short dependency chains
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = s2[nt][i] = 0.f;
      const uint32_t kgw[8] = {kg0.x, kg0.y, kg0.z, kg0.w, kg1.x, kg1.y, kg1.z, kg1.w};
      const uint32_t khw[8] = {kh0.x, kh0.y, kh0.z, kh0.w, kh1.x, kh1.y, kh1.z, kh1.w};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t a0 = lo16_to_f16x2(kgw[ks]), a2 = hi16_to_f16x2(kgw[ks]);
        const uint32_t a1 = lo16_to_f16x2(khw[ks]), a3 = hi16_to_f16x2(khw[ks]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma16816_f16((ks & 1) ? s2[nt] : s[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] += s2[nt][i];

      {
        const unsigned char* v8 = smem + buf * kStage8 + warp * kTile8 + kBPS * kTile8;
        va = lds128(v8 + sw8(2 * t, g));
        vb = lds128(v8 + sw8(2 * t + 1, g));
        vc = lds128(v8 + sw8(2 * t + 8, g));
        vd = lds128(v8 + sw8(2 * t + 9, g));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);   // codes are in registers: free the slot
      // ---- online softmax per head (column); this lane holds keys g, g+8.
      // The running max m only has to bound the scores to within the lazy
      // threshold (p = 2^(s - m) <= 2^8 stays in f16), so a warp vote decides
      // whether any score exceeds it; only then is the exact max reduced over
      // the block's keys (every unit's first block, and rarely later).
      const bool k0ok = g < valid, k1ok = g + 8 < valid;
      float v[NT][4];
      bool grow = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[nt][i] = (i < 2 ? k0ok : k1ok) ? s[nt][i] * sl2 : -INFINITY;
          grow |= v[nt][i] > m_run[nt][i & 1] + kLazy8;
        }
      if (__any_sync(kAll8, grow)) {
        bool rescale = false;
        float alpha[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(v[nt][j], v[nt][j + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(kAll8, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kAll8, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kAll8, mx, 16));
            float m_new = m_run[nt][j];
            if (mx > m_new + kLazy8 || m_new == -INFINITY) m_new = mx;
            alpha[nt][j] = (m_new == m_run[nt][j]) ? 1.f : ex2(m_run[nt][j] - m_new);
            rescale |= alpha[nt][j] != 1.f;
            m_run[nt][j] = m_new;
          }
        if (__any_sync(kAll8, rescale)) {
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
        const uint32_t x0 = pack2_f16(ex2(v[nt][0] - m_run[nt][0]), ex2(v[nt][1] - m_run[nt][1]));
        const uint32_t x1 = pack2_f16(ex2(v[nt][2] - m_run[nt][0]), ex2(v[nt][3] - m_run[nt][1]));
        const __half2 h0 = *reinterpret_cast<const __half2*>(&x0);   // key g,     heads 2t, 2t+1
        const __half2 h1 = *reinterpret_cast<const __half2*>(&x1);   // key g + 8, heads 2t, 2t+1
        l_run[nt][0] += __low2float(h0) + __low2float(h1);
        l_run[nt][1] += __high2float(h0) + __high2float(h1);
        pb0[nt] = movm_t(x0);                          // head g: keys 2t, 2t+1
        pb1[nt] = movm_t(x1);                          // head g: keys 2t+8, 2t+9
      }

      // ---- O^T += V^T . P^T; V codes of keys past the end become +0
      uint32_t vaw[4] = {va.x, va.y, va.z, va.w}, vbw[4] = {vb.x, vb.y, vb.z, vb.w};
      uint32_t vcw[4] = {vc.x, vc.y, vc.z, vc.w}, vdw[4] = {vd.x, vd.y, vd.z, vd.w};
      if (valid < kBlockSize) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (2 * t >= valid) vaw[j] = 0u;
          if (2 * t + 1 >= valid) vbw[j] = 0u;
          if (2 * t + 8 >= valid) vcw[j] = 0u;
          if (2 * t + 9 >= valid) vdw[j] = 0u;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int j = mt >> 1;
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;   // byte pairs (2e, 2e+1) of two keys
        const uint32_t ab = prmt(vaw[j], vbw[j], sel);        // keys 2t, 2t+1 at dims d, d+1
        const uint32_t cd = prmt(vcw[j], vdw[j], sel);        // keys 2t+8, 2t+9
        const uint32_t a0 = lo16_to_f16x2(ab), a1 = hi16_to_f16x2(ab);
        const uint32_t a2 = lo16_to_f16x2(cd), a3 = hi16_to_f16x2(cd);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816_f16(o[nt][mt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
      }
    }

    // ---- l summed over the lanes of each head
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        l_run[nt][j] += __shfl_xor_sync(kAll8, l_run[nt][j], 4);
        l_run[nt][j] += __shfl_xor_sync(kAll8, l_run[nt][j], 8);
        l_run[nt][j] += __shfl_xor_sync(kAll8, l_run[nt][j], 16);
      }
    const bool direct = (u.ns == 1);
    if constexpr (HS) {
      // this warp saw every key of the unit for its own heads: O / l (V's
      // scale applied) goes out straight from the accumulators, dims
      // 16g + 2mt and the next one per lane and tile
      __half* ws_half = reinterpret_cast<__half*>(a.ws_acc);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int hh = 8 * nt + 2 * t + j;
          if (hh < G) {
            const float rl = vscale / l_run[nt][j];
            const int64_t row = (int64_t)u.b * a.num_q_heads + hq0 + hh;
            const int64_t pidx = row * a.max_splits + u.s;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const int d = 16 * g + 2 * mt;
              const float x0 = o[nt][mt][j] * rl, x1 = o[nt][mt][j + 2] * rl;
              if (direct)
                *reinterpret_cast<__nv_bfloat162*>(outp + row * kHD + d) = __floats2bfloat162_rn(x0, x1);
              else
                *reinterpret_cast<__half2*>(ws_half + pidx * kHD + d) = __floats2half2_rn(x0, x1);
            }
            if (!direct && g == 0) {
              a.ws_ml[pidx * 2 + 0] = m_run[nt][j];
              a.ws_ml[pidx * 2 + 1] = l_run[nt][j];
            }
          }
        }
    } else {
      // ---- otherwise merge the four warps of this unit (each saw a quarter
      // of its blocks); V's scale applies here
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
            float* crow = comb + (warp * G + hh) * kCombRow + 16 * g;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)   // pair slot mt stored at mt ^ g: no bank conflicts
              *reinterpret_cast<float2*>(crow + 2 * (mt ^ g)) =
                  make_float2(o[nt][mt][j], o[nt][mt][j + 2]);
          }
        }
      named_bar_sync(1, kConsumers8);
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
          wk[k] = (mk == -INFINITY) ? 0.f : ex2(mk - M);
          L = fmaf(wk[k], comb_ml[(k * G + h) * 2 + 1], L);
        }
        const float rl = vscale / L;
        const int64_t row = (int64_t)u.b * a.num_q_heads + hq0 + h;
        const int64_t pidx = row * a.max_splits + u.s;
#pragma unroll
        for (int i = 0; i < kHD / 32; ++i) {
          const int d = lane + 32 * i;
          const int dp = (d & ~15) | ((((d & 15) >> 1) ^ (d >> 4)) << 1) | (d & 1);
          float O = 0.f;
#pragma unroll
          for (int k = 0; k < kCW; ++k) O = fmaf(wk[k], comb[(k * G + h) * kCombRow + dp], O);
          if (direct)
            outp[row * kHD + d] = __float2bfloat16_rn(O * rl);
          else
            reinterpret_cast<__half*>(a.ws_acc)[pidx * kHD + d] = __float2half_rn(O * rl);
        }
        if (!direct && lane == 0) {
          a.ws_ml[pidx * 2 + 0] = M;
          a.ws_ml[pidx * 2 + 1] = L;
        }
      }
      named_bar_sync(1, kConsumers8);
    }
  }
}

template <int G, bool HS>
cudaError_t launch_fp8_g(const DecodeArgs& args, int num_sms, cudaStream_t stream) {
  using C = F8Cfg<G>;
  DecodeArgs a = args;
  DecodeArgs aw = a;
  if (HS) aw.num_kv_heads = a.num_kv_heads / kBPS;
  a.balanced = a.ws_np != nullptr && stage_plan_fits(aw, HS ? kBlockSize : kStageTok);
  a.partials_f16 = 1;
  CUtensorMap tm_k, tm_v;
  const int64_t rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  if (!encode_pool_map_u8(&tm_k, a.k_cache, rows) || !encode_pool_map_u8(&tm_v, a.v_cache, rows))
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
  cudaError_t e = allow_dynamic_smem(decode_fp8_kernel<G, HS>, (int)smem);
  if (e != cudaSuccess) return e;
  const int by_smem = (int)((228 * 1024) / (smem + 1024));
  const int per_sm = by_smem < 1 ? 1 : (by_smem > (G <= 8 ? 3 : 2) ? (G <= 8 ? 3 : 2) : by_smem);
  const int64_t upper = (int64_t)a.num_seqs * a.num_kv_heads * a.max_splits;
  const int grid = (int)(upper < (int64_t)num_sms * per_sm ? upper : (int64_t)num_sms * per_sm);
  decode_fp8_kernel<G, HS><<<grid, kThreads8, smem, stream>>>(a, tm_k, tm_v);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  return launch_decode_reduce_bf16_128(a, stream);
}

}  // namespace

cudaError_t launch_paged_decode_fp8(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  if (a.chunk_prior >= 0 || a.split_tokens % kStageTok != 0 || !a.k_scale || !a.v_scale)
    return cudaErrorInvalidValue;
  // one block of kBPS KV heads per stage when the heads form such groups
  const bool hs = a.num_kv_heads % kBPS == 0;
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return hs ? launch_fp8_g<1, true>(a, num_sms, stream) : launch_fp8_g<1, false>(a, num_sms, stream);
    case 2: return hs ? launch_fp8_g<2, true>(a, num_sms, stream) : launch_fp8_g<2, false>(a, num_sms, stream);
    case 4: return hs ? launch_fp8_g<4, true>(a, num_sms, stream) : launch_fp8_g<4, false>(a, num_sms, stream);
    case 8: return hs ? launch_fp8_g<8, true>(a, num_sms, stream) : launch_fp8_g<8, false>(a, num_sms, stream);
    case 16: return hs ? launch_fp8_g<16, true>(a, num_sms, stream) : launch_fp8_g<16, false>(a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
