// Decode attention over a latent (MLA-style) KV cache, on warp-level bf16
// tensor-core tiles (mma.sync m16n8k16, fp32 accumulate) for sm_103a.
//
// What it computes.  "The KV cache and prefix caching", section "What prefill
// stores and decode reads", names multi-head latent attention (the DeepSeek
// line): per token the cache stores a low-rank latent c instead of keys and
// values, and query head h sees the key W_K[h] c and the value W_V[h] c.
// With the projections absorbed -- q~_h = W_K[h]^T q_h before this kernel and
// o_h = W_V[h] z_h after it -- the attention over the latent is
//   z_h = sum_j softmax_j(scale * q~_h . c_j) c_j,
// i.e. grouped-query decode with a single KV head whose key and value are both
// the latent, shared by all Hq query heads.  This kernel computes z (rank 128,
// 32 query heads).
//
// Structure: the bf16 decode kernel's (persistent CTAs walking the sequences
// in equal per-CTA shares of 64-token stages, or 512-token splits for small
// batches; one TMA producer warp; keys on the M side of the
// tile and heads on N; the running max gated by a warp vote; split partials
// merged by the reduce kernel), with two changes for the 32 heads that share
// each latent block:
//  * a block is loaded once (16 rows x 256 B) and serves as both the K and the
//    V operand;
//  * eight consumer warps: warp w takes block w % 4 of each stage for the
//    query heads 16 * (w / 4) .. + 15, so each staged block feeds two warps;
//  * a register split (setmaxnreg): the producer warp and three idle warps
//    completing its warpgroup drop to 40 registers so the consumers can take
//    232; at the 168 of the launch the consumers spilled.
#include <cuda.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "host_cache.h"
#include "launch.h"
#include "tmap.h"

namespace pkv {
namespace {

constexpr int kHeads = 32;                       // query heads sharing the latent
constexpr int kHalfHeads = 16;                   // heads per consumer warp
constexpr int kNTL = kHalfHeads / 8;             // head tiles of 8 per warp
constexpr int kBPSL = 4;                         // blocks per stage
constexpr int kCWL = 2 * kBPSL;                  // consumer warps
constexpr int kConsumersL = kCWL * 32;
constexpr int kThreadsL = kConsumersL + 128;     // producer warp + three idle warps (warpgroup 2)
constexpr int kRegsConsL = 232, kRegsRestL = 40;
static_assert(kRegsConsL * kConsumersL + kRegsRestL * 128 <= ((65536 / kThreadsL) & ~7) * kThreadsL,
              "register split within the launch budget");
constexpr int kStageTokL = kBPSL * kBlockSize;   // 64 tokens
constexpr int kHalfL = kBlockSize * 128;         // 16 rows x 128 B: one 64-column half
constexpr int kTileL = 2 * kHalfL;               // one latent block, 4 KiB
constexpr int kStageL = kBPSL * kTileL;          // 16 KiB
constexpr int kNSTL = 4;
constexpr int kRingL = kNSTL * kStageL;
constexpr int kR = 128;                          // latent rank
constexpr int kCombRowL = kR + 4;
constexpr float kLazyL = 8.0f;
constexpr unsigned kAllL = 0xffffffffu;

constexpr int OFF_COMB_L = kRingL;                               // [warp][16 heads][132] fp32
constexpr int OFF_ML_L = OFF_COMB_L + kCWL * kHalfHeads * kCombRowL * 4;
constexpr int OFF_BAR_L = OFF_ML_L + kCWL * kHalfHeads * 2 * 4;
constexpr int OFF_CU_L = OFF_BAR_L + 2 * kNSTL * 8 + 16;

static_assert(kSplitTokens % kStageTokL == 0, "a split holds whole stages");
static_assert(32 % kBPSL == 0, "a stage never straddles two block-id windows");

__device__ __forceinline__ void mma16816l(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2_bf16l(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t movm_tl(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}
__device__ __forceinline__ uint32_t prmtl(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ float ex2l(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint4 lds128l(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void tma2d_l(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                        int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__global__ void __launch_bounds__(kThreadsL, 1)
decode_mla_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_c) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  float* comb = reinterpret_cast<float*>(smem + OFF_COMB_L);
  float* comb_ml = reinterpret_cast<float*>(smem + OFF_ML_L);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR_L);
  int* abort_flag = reinterpret_cast<int*>(bars + 2 * kNSTL);
  int* cu = reinterpret_cast<int*>(smem + OFF_CU_L);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kNSTL);

  if (tid == 0) {
    for (int i = 0; i < kNSTL; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kCWL);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // balanced walk over 64-token stages when the batch gives every CTA at
  // least kMinStagesPerCta of them; otherwise 512-token splits
  plan_units(a, cu, a.balanced ? kStageTokL : 0);
  __syncthreads();
  const bool balanced =
      a.balanced && (int64_t)cu[a.num_seqs] >= (int64_t)kMinStagesPerCta * gridDim.x;
  if (a.balanced && !balanced) {
    __syncthreads();
    plan_units(a, cu);
    __syncthreads();
  }
  volatile int* vabort = abort_flag;

  if (warp >= kCWL) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsRestL));
  if (warp > kCWL) return;   // idle warps of warpgroup 2
  if (warp == kCWL) {
    // ------------------------------------------------------------ producer
    if (lane == 0)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_c)) : "memory");
    const uint64_t policy = policy_evict_first();
    uint32_t issued = 0;
    bool ok = true;
    Walk wk = walk_begin(a, cu, balanced);
    Unit u;
    while (ok && walk_next(a, cu, kStageTokL, wk, u)) {
      const int blk0 = u.tok_begin / kBlockSize;
      const int nblk = (u.tok_end - 1) / kBlockSize - blk0 + 1;
      const int32_t* bt_row = a.block_table + (int64_t)u.b * a.bt_stride + blk0;
      int my_blk = 0;
      const int nst = (nblk + kBPSL - 1) / kBPSL;
      for (int st = 0; st < nst; ++st, ++issued) {
        if ((st * kBPSL) % 32 == 0) {  // next window of 32 block ids, one per lane
          const int idx = st * kBPSL + lane;
          my_blk = 0;
          if (idx < nblk) {
            my_blk = __ldg(bt_row + idx);
            if (my_blk < 0 || (int64_t)my_blk >= a.num_blocks) {
              record_error(a.err, DEVERR_BLOCK_RANGE);
              my_blk = 0;  // read a valid block instead; the error word reports it
            }
          }
        }
        const int buf = issued % kNSTL;
        const uint32_t phase = (issued / kNSTL) & 1;
        if (lane == 0 && issued >= (uint32_t)kNSTL && !*vabort) {
          if (!mbar_wait(empty0 + 8 * buf, phase ^ 1, a.err)) *vabort = 1;
        }
        __syncwarp();
        if (*vabort) { ok = false; break; }
        const int nb = min(kBPSL, nblk - st * kBPSL);
        int rows[kBPSL];
#pragma unroll
        for (int i = 0; i < kBPSL; ++i)
          rows[i] = __shfl_sync(kAllL, my_blk, (st * kBPSL + i) & 31) * kBlockSize;
        if (lane == 0) {
          const uint32_t fb = full0 + 8 * buf;
          mbar_arrive_expect_tx(fb, (uint32_t)(nb * kTileL));
          const uint32_t dst = sbase + buf * kStageL;
#pragma unroll
          for (int i = 0; i < kBPSL; ++i) {
            if (i < nb) {
              tma2d_l(dst + i * kTileL, &tm_c, fb, 0, rows[i], policy);
              tma2d_l(dst + i * kTileL + kHalfL, &tm_c, fb, 64, rows[i], policy);
            }
          }
        }
      }
    }
    if (!ok && lane == 0) {  // on abort, let the copies already issued land
      const uint32_t first = issued > (uint32_t)kNSTL ? issued - kNSTL : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait(full0 + 8 * (i % kNSTL), (i / kNSTL) & 1, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsConsL));
  const int g = lane >> 2, t = lane & 3;
  const int bw = warp & (kBPSL - 1);              // block of the stage this warp takes
  const int hbase = (warp / kBPSL) * kHalfHeads;   // its 16 query heads
  const float sl2 = a.scale * 1.4426950408889634f;
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
  // latent pieces of this lane, as in the bf16 decode kernel: load step i
  // takes chunk kc(i) of the 64-column half (t >> 1) for the score products;
  // rows 2t, 2t+1, 2t+8, 2t+9 at dims 16g + 8 * (j ^ (g & 1)) for P.V
  const int khalf = t >> 1;
  const int kc0 = 4 * (t & 1), kx = (t >> 1) << 1;
  const int vhalf = g >> 2;
  uint32_t consumed = 0;

  Walk wk = walk_begin(a, cu, balanced);
  Unit u;
  while (walk_next(a, cu, kStageTokL, wk, u)) {
    // the merge reads how many partials this sequence left
    if (a.balanced && u.s == 0 && tid == 0) a.ws_np[u.b] = u.ns;
    // q~ of heads hbase + 8nt + g as B fragments, in the lane's K order
    uint4 qf[kNTL][4];
#pragma unroll
    for (int nt = 0; nt < kNTL; ++nt) {
      const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) +
                                  ((int64_t)u.b * a.num_q_heads + hbase + 8 * nt + g) * kR;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qf[nt][i] = __ldg(reinterpret_cast<const uint4*>(qrow + 64 * khalf + 8 * (kc0 + (i ^ kx))));
    }
    float o[kNTL][8][4];
#pragma unroll
    for (int nt = 0; nt < kNTL; ++nt)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
    float m_run[kNTL][2], l_run[kNTL][2];
#pragma unroll
    for (int nt = 0; nt < kNTL; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
    }

    const int nblk = (u.tok_end - 1) / kBlockSize - u.tok_begin / kBlockSize + 1;
    const int nst = (nblk + kBPSL - 1) / kBPSL;
    for (int st = 0; st < nst; ++st, ++consumed) {
      const int buf = consumed % kNSTL;
      const uint32_t phase = (consumed / kNSTL) & 1;
      if (!*vabort) {
        if (!mbar_wait(full0 + 8 * buf, phase, a.err)) *vabort = 1;
      }
      const int tok0 = u.tok_begin + (st * kBPSL + bw) * kBlockSize;
      const int valid = min(kBlockSize, u.tok_end - tok0);
      if (valid <= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * buf);
        continue;
      }
      const uint32_t ct = sbase + buf * kStageL + bw * kTileL;
      // ---- the latent as the K operand: keys g and g + 8
      uint4 kg[4], kh[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = kc0 + (i ^ kx);
        kg[i] = lds128l(ct + khalf * kHalfL + g * 128 + ((c ^ g) << 4));
        kh[i] = lds128l(ct + khalf * kHalfL + (g + 8) * 128 + ((c ^ g) << 4));
      }
      float s[kNTL][4], s2[kNTL][4];
#pragma unroll
      for (int nt = 0; nt < kNTL; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = s2[nt][i] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int nt = 0; nt < kNTL; ++nt) {
          mma16816l(s[nt], kg[i].x, kh[i].x, kg[i].y, kh[i].y, qf[nt][i].x, qf[nt][i].y);
          mma16816l(s2[nt], kg[i].z, kh[i].z, kg[i].w, kh[i].w, qf[nt][i].z, qf[nt][i].w);
        }
      // ---- the same latent rows as the V operand
      uint4 va[2], vb[2], vc[2], vd[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = 2 * (g & 3) + (j ^ (g & 1));
        const uint32_t base = ct + vhalf * kHalfL;
        va[j] = lds128l(base + (2 * t) * 128 + ((c ^ (2 * t)) << 4));
        vb[j] = lds128l(base + (2 * t + 1) * 128 + ((c ^ (2 * t + 1)) << 4));
        vc[j] = lds128l(base + (2 * t + 8) * 128 + ((c ^ (2 * t)) << 4));
        vd[j] = lds128l(base + (2 * t + 9) * 128 + ((c ^ (2 * t + 1)) << 4));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);
#pragma unroll
      for (int nt = 0; nt < kNTL; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] += s2[nt][i];

      // ---- online softmax per head; this lane holds keys g, g+8
      const bool k0ok = g < valid, k1ok = g + 8 < valid;
      float v[kNTL][4];
      bool grow = false;
#pragma unroll
      for (int nt = 0; nt < kNTL; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[nt][i] = (i < 2 ? k0ok : k1ok) ? s[nt][i] * sl2 : -INFINITY;
          grow |= v[nt][i] > m_run[nt][i & 1] + kLazyL;
        }
      if (__any_sync(kAllL, grow)) {
        bool rescale = false;
        float alpha[kNTL][2];
#pragma unroll
        for (int nt = 0; nt < kNTL; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(v[nt][j], v[nt][j + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(kAllL, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kAllL, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kAllL, mx, 16));
            float m_new = m_run[nt][j];
            if (mx > m_new + kLazyL || m_new == -INFINITY) m_new = mx;
            alpha[nt][j] = (m_new == m_run[nt][j]) ? 1.f : ex2l(m_run[nt][j] - m_new);
            rescale |= alpha[nt][j] != 1.f;
            m_run[nt][j] = m_new;
          }
        if (__any_sync(kAllL, rescale)) {
#pragma unroll
          for (int nt = 0; nt < kNTL; ++nt) {
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
      uint32_t pb0[kNTL], pb1[kNTL];
#pragma unroll
      for (int nt = 0; nt < kNTL; ++nt) {
        const uint32_t x0 = pack2_bf16l(ex2l(v[nt][0] - m_run[nt][0]), ex2l(v[nt][1] - m_run[nt][1]));
        const uint32_t x1 = pack2_bf16l(ex2l(v[nt][2] - m_run[nt][0]), ex2l(v[nt][3] - m_run[nt][1]));
        l_run[nt][0] += bf16lo(x0) + bf16lo(x1);
        l_run[nt][1] += bf16hi(x0) + bf16hi(x1);
        pb0[nt] = movm_tl(x0);
        pb1[nt] = movm_tl(x1);
      }
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
        const uint32_t bw4[4] = {vb[j].x, vb[j].y, vb[j].z, vb[j].w};
        const uint32_t cw[4] = {vc[j].x, vc[j].y, vc[j].z, vc[j].w};
        const uint32_t dw[4] = {vd[j].x, vd[j].y, vd[j].z, vd[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t a0 = prmtl(aw[e], bw4[e], 0x5410u);
          const uint32_t a1 = prmtl(aw[e], bw4[e], 0x7632u);
          const uint32_t a2 = prmtl(cw[e], dw[e], 0x5410u);
          const uint32_t a3 = prmtl(cw[e], dw[e], 0x7632u);
#pragma unroll
          for (int nt = 0; nt < kNTL; ++nt) mma16816l(o[nt][4 * j + e], a0, a1, a2, a3, pb0[nt], pb1[nt]);
        }
      }
    }

    // ---- merge: the four warps of each head half
#pragma unroll
    for (int nt = 0; nt < kNTL; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        l_run[nt][j] += __shfl_xor_sync(kAllL, l_run[nt][j], 4);
        l_run[nt][j] += __shfl_xor_sync(kAllL, l_run[nt][j], 8);
        l_run[nt][j] += __shfl_xor_sync(kAllL, l_run[nt][j], 16);
      }
#pragma unroll
    for (int nt = 0; nt < kNTL; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int hl = 8 * nt + 2 * t + j;          // head within this warp's half
        if (g == 0) {
          comb_ml[(warp * kHalfHeads + hl) * 2 + 0] = m_run[nt][j];
          comb_ml[(warp * kHalfHeads + hl) * 2 + 1] = l_run[nt][j];
        }
        float* crow = comb + (warp * kHalfHeads + hl) * kCombRowL + 16 * g;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          *reinterpret_cast<float2*>(crow + 8 * ((mt >> 2) ^ (g & 1)) + 2 * (mt & 3)) =
              make_float2(o[nt][mt][j], o[nt][mt][j + 2]);
      }
    named_bar_sync(1, kConsumersL);
    const bool direct = (u.ns == 1);
    for (int h = warp; h < kHeads; h += kCWL) {
      const int half = h / kHalfHeads, hl = h % kHalfHeads;
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < kBPSL; ++k)
        M = fmaxf(M, comb_ml[((half * kBPSL + k) * kHalfHeads + hl) * 2]);
      float wk[kBPSL], L = 0.f;
#pragma unroll
      for (int k = 0; k < kBPSL; ++k) {
        const float mk = comb_ml[((half * kBPSL + k) * kHalfHeads + hl) * 2];
        wk[k] = (mk == -INFINITY) ? 0.f : ex2l(mk - M);
        L = fmaf(wk[k], comb_ml[((half * kBPSL + k) * kHalfHeads + hl) * 2 + 1], L);
      }
      const float rl = 1.f / L;
      const int64_t row = (int64_t)u.b * a.num_q_heads + h;
      const int64_t pidx = row * a.max_splits + u.s;
#pragma unroll
      for (int i = 0; i < kR / 32; ++i) {
        const int d = lane + 32 * i;
        float O = 0.f;
#pragma unroll
        for (int k = 0; k < kBPSL; ++k)
          O = fmaf(wk[k], comb[((half * kBPSL + k) * kHalfHeads + hl) * kCombRowL + d], O);
        if (direct)
          outp[row * kR + d] = __float2bfloat16_rn(O * rl);
        else
          a.ws_acc[pidx * kR + d] = O;
      }
      if (!direct && lane == 0) {
        a.ws_ml[pidx * 2 + 0] = M;
        a.ws_ml[pidx * 2 + 1] = L;
      }
    }
    named_bar_sync(1, kConsumersL);
  }
}

}  // namespace

cudaError_t launch_decode_mla(const DecodeArgs& args, int num_sms, cudaStream_t stream) {
  DecodeArgs a = args;
  a.balanced = a.ws_np != nullptr && stage_plan_fits(a, kStageTokL);
  if (a.chunk_prior >= 0 || a.split_tokens % kStageTokL != 0 || a.num_kv_heads != 1 ||
      a.num_q_heads != kHeads || a.head_dim != kR)
    return cudaErrorInvalidValue;
  CUtensorMap tm_c;
  const int64_t rows = a.num_blocks * kBlockSize;
  if (!encode_pool_map_bf16(&tm_c, a.k_cache, rows)) return cudaErrorInvalidValue;
  const size_t smem = OFF_CU_L + sizeof(int) * (size_t)(a.num_seqs + 1) + 1024;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = allow_dynamic_smem(decode_mla_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t upper = (int64_t)a.num_seqs * a.max_splits;
  const int grid = (int)(upper < (int64_t)num_sms ? upper : (int64_t)num_sms);
  decode_mla_kernel<<<grid, kThreadsL, smem, stream>>>(a, tm_c);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  return launch_decode_reduce_bf16_128(a, stream);
}

}  // namespace pkv
