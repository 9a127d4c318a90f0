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
// The work is HBM-bound: every cached byte is read once and used for
// 2*G multiply-adds.  For a GQA group the score and value products are small
// dense contractions -- [G x 128] . [128 x 16 keys] and [G x 16] . [16 x 128]
// per 16-token block -- so one warp does each block with 32 m16n8k16 tiles
// (the G query heads are the M rows, zero-padded to 16).  That leaves the
// warps far below their issue limit, so the kernel is free to run at the
// speed of the memory system; doing the same products on CUDA cores needs
// about eight times as many instructions (shuffle reductions, unpacking).
//
// Structure (per CTA: one TMA producer warp + four consumer warps, two CTAs
// per SM, persistent over a flat list of (sequence, KV head, 512-token
// split) units):
//  * The producer streams, for each 16-token block, its K and V tiles with
//    2-D TMA tensor copies (two 64-column halves each, 128-byte swizzle) into
//    a 3-stage ring of 4 blocks per stage, completing on mbarriers.  It runs
//    ahead across unit boundaries.
//  * Consumer warp w takes block w of every stage: ldmatrix (non-transposed
//    for K, transposed for V; the swizzle makes both conflict-free), 16 MMAs
//    for S = Q K^T, an online softmax on the S fragments in registers (running
//    max in the log2 domain, raised lazily only when it grows by more than 8;
//    max over the 4 lanes of a row by two shuffles), the S accumulators
//    repacked as bf16 A fragments, then 16 MMAs for O += P V.
//  * Each warp keeps its own (m, l, O) for its blocks; at the end of a unit
//    the four warps merge through shared memory.  A unit that covers its
//    whole sequence writes the output; otherwise it writes (m, l, O) partials
//    that the reduce kernel merges.
//  * Keys past the end of a sequence are masked before the softmax, and the
//    matching V rows of the last (partial) block are zeroed in shared memory
//    before P.V, so stale pool contents (even NaN) never reach the output.
#include <cuda.h>

#include "common.cuh"
#include "decode_common.cuh"
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
constexpr int kNST = 3;
constexpr int kRingB = kNST * kStageB;
constexpr int kHD = 128;
constexpr float kLazyM = 8.0f;
constexpr unsigned kAllM = 0xffffffffu;

static_assert(kSplitTokens % kStageTok == 0, "a split holds whole stages");
static_assert(32 % kBPS == 0, "a stage never straddles two block-id windows");

template <int G>
struct MCfg {
  static constexpr int COMB_B = kCW * G * kHD * 4;            // merged O per warp
  static constexpr int ML_B = kCW * G * 2 * 4;
  static constexpr int OFF_COMB = kRingB;
  static constexpr int OFF_ML = OFF_COMB + COMB_B;
  static constexpr int OFF_BAR = OFF_ML + ML_B;
  static constexpr int OFF_CU = OFF_BAR + 2 * kNST * 8 + 16;
  static_assert(G >= 1 && G <= 16 && (G & (G - 1)) == 0, "group of 1..16 heads");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
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

template <int G, bool FUSE>
__global__ void __launch_bounds__(kThreadsM, 2)
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
    for (int i = 0; i < kNST; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kCW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  plan_units(a, cu);
  __syncthreads();
  const int total = cu[a.num_seqs];
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
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Unit u = find_unit(a, cu, w);
      const int blk0 = u.tok_begin / kBlockSize;
      const int nblk = (u.tok_end - 1) / kBlockSize - blk0 + 1;
      const int32_t* bt_row = a.block_table + (int64_t)u.b * a.bt_stride + blk0;
      int my_blk = 0;
      const int nst = (nblk + kBPS - 1) / kBPS;
      for (int st = 0; st < nst; ++st, ++issued) {
        if ((st * kBPS) % 32 == 0) {  // next window of 32 block ids, one per lane
          const int idx = st * kBPS + lane;
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
        const int nb = min(kBPS, nblk - st * kBPS);
        int rows[kBPS];
#pragma unroll
        for (int i = 0; i < kBPS; ++i)
          rows[i] = (__shfl_sync(kAllM, my_blk, (st * kBPS + i) & 31) * a.num_kv_heads + u.g) *
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
  const int g = lane >> 2, t = lane & 3;
  const bool row_real = g < G;                  // row g of the M tile is a real head
  const float sl2 = a.scale * 1.4426950408889634f;
  const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
  // ldmatrix lane roles: matrix mi = lane >> 3, row-in-matrix rr = lane & 7
  const int mi = lane >> 3, rr = lane & 7;
  uint32_t consumed = 0;

  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const Unit u = find_unit(a, cu, w);
    const int hq0 = u.g * G;
    // Q as A fragments: a0 = (row g, d 16ks+2t..+1), a2 = (row g, d 16ks+8+2t..+1);
    // rows g+8 (a1, a3) are real only when G == 16.
    uint32_t qa[8][2], qb[8][2];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = qa[ks][1] = qb[ks][0] = qb[ks][1] = 0u;
    }
    if (row_real) {
      const uint32_t* qrow = q32 + ((int64_t)u.b * a.num_q_heads + hq0 + g) * (kHD / 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = __ldg(qrow + ks * 8 + t);
        qa[ks][1] = __ldg(qrow + ks * 8 + 4 + t);
      }
    }
    if (G == 16) {
      const uint32_t* qrow = q32 + ((int64_t)u.b * a.num_q_heads + hq0 + g + 8) * (kHD / 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qb[ks][0] = __ldg(qrow + ks * 8 + t);
        qb[ks][1] = __ldg(qrow + ks * 8 + 4 + t);
      }
    }
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    const int nblk = (u.tok_end - 1) / kBlockSize - u.tok_begin / kBlockSize + 1;
    const int nst = (nblk + kBPS - 1) / kBPS;
    for (int st = 0; st < nst; ++st, ++consumed) {
      const int buf = consumed % kNST;
      const uint32_t phase = (consumed / kNST) & 1;
      if (!*vabort) {
        if (!mbar_wait(full0 + 8 * buf, phase, a.err)) *vabort = 1;
      }
      const int tok0 = u.tok_begin + (st * kBPS + warp) * kBlockSize;
      const int valid = min(kBlockSize, u.tok_end - tok0);   // keys of this warp's block
      if (valid > 0) {
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
          const int64_t src = (((int64_t)u.b * a.num_kv_heads + u.g) * kHD) + c * 8;
          const uint4 val = __ldg(reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(is_v ? a.v_new : a.k_new) + src));
          unsigned char* tile = smem + buf * kStageB + (is_v ? kBPS * kTileB : 0) + warp * kTileB;
          *reinterpret_cast<uint4*>(tile + sw_off(r, c)) = val;
          const int blk = __ldg(a.block_table + (int64_t)u.b * a.bt_stride + (tok0 / kBlockSize));
          if (blk >= 0 && (int64_t)blk < a.num_blocks) {
            __nv_bfloat16* pool = const_cast<__nv_bfloat16*>(
                static_cast<const __nv_bfloat16*>(is_v ? a.v_cache : a.k_cache));
            const int64_t dst = (((int64_t)blk * a.num_kv_heads + u.g) * kBlockSize + r) * kHD + c * 8;
            *reinterpret_cast<uint4*>(pool + dst) = val;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        if (valid < kBlockSize) {
          // zero the V rows past the sequence end (whole rows, so the swizzle does not matter)
          unsigned char* vrow = smem + buf * kStageB + kBPS * kTileB + warp * kTileB;
          for (int i = lane; i < (kBlockSize - valid) * 16; i += 32) {
            const int row = valid + (i >> 4), c = i & 15;
            *reinterpret_cast<uint4*>(vrow + (c >> 3) * kHalfB + row * 128 + (c & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          // order these generic-proxy writes before the TMA refill of this slot
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        // ---- S = Q K^T : two n-tiles of 8 keys
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = ((mi >> 1) << 3) + rr;   // key row this lane addresses
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t kb[4];
          ldsm_x4(kt + sw_off(krow, 2 * ks + (mi & 1)), kb);
          mma16816(s[0], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], kb[0], kb[1]);
          mma16816(s[1], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], kb[2], kb[3]);
        }
        // ---- online softmax on the fragments: row g holds keys 8nt+2t, +1 (c0, c1),
        // row g+8 the same keys (c2, c3)
        float p[2][4];
        float alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float v[4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int key = nt * 8 + 2 * t + j;
              v[nt * 2 + j] = key < valid ? s[nt][2 * r + j] * sl2 : -INFINITY;
            }
          float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
          mx = fmaxf(mx, __shfl_xor_sync(kAllM, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(kAllM, mx, 2));
          float m_new = m_run[r];
          if (mx > m_run[r] + kLazyM || m_run[r] == -INFINITY) m_new = mx;
          alpha[r] = (m_new == m_run[r]) ? 1.f : exp2f(m_run[r] - m_new);
          m_run[r] = m_new;
          float sum = 0.f;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float e = exp2f(v[nt * 2 + j] - m_new);
              p[nt][2 * r + j] = e;
            }
          // the sum uses the bf16-rounded weights that P.V multiplies
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t pk = pack2_bf16(p[nt][2 * r], p[nt][2 * r + 1]);
            sum += bf16lo(pk) + bf16hi(pk);
          }
          l_run[r] = l_run[r] * alpha[r] + sum;
        }
        if (__any_sync(kAllM, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[0];
            o[n][2] *= alpha[1];
            o[n][3] *= alpha[1];
          }
        }
        // S accumulators -> A fragments of P (keys 0-7 from n-tile 0, 8-15 from n-tile 1)
        const uint32_t pa0 = pack2_bf16(p[0][0], p[0][1]);
        const uint32_t pa1 = pack2_bf16(p[0][2], p[0][3]);
        const uint32_t pa2 = pack2_bf16(p[1][0], p[1][1]);
        const uint32_t pa3 = pack2_bf16(p[1][2], p[1][3]);
        // ---- O += P V : 16 n-tiles of 8 columns, V through transposed ldmatrix
        const int vrow = ((mi & 1) << 3) + rr;
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t vb[4];
          ldsm_x4_t(vt + sw_off(vrow, 2 * np + (mi >> 1)), vb);
          mma16816(o[2 * np], pa0, pa1, pa2, pa3, vb[0], vb[1]);
          mma16816(o[2 * np + 1], pa0, pa1, pa2, pa3, vb[2], vb[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);
    }

    // ---- merge the four warps of this unit
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(kAllM, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(kAllM, l_run[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = g + 8 * r;
      if (row < G) {
        if (t == 0) {
          comb_ml[(warp * G + row) * 2 + 0] = m_run[r];
          comb_ml[(warp * G + row) * 2 + 1] = l_run[r];
        }
#pragma unroll
        for (int n = 0; n < 16; ++n)
          *reinterpret_cast<float2*>(comb + (warp * G + row) * kHD + n * 8 + 2 * t) =
              make_float2(o[n][2 * r], o[n][2 * r + 1]);
      }
    }
    named_bar_sync(1, kConsumersM);
    const bool direct = (u.ns == 1);
    for (int oi = tid; oi < G * kHD; oi += kConsumersM) {
      const int h = oi / kHD, d = oi - h * kHD;
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < kCW; ++k) M = fmaxf(M, comb_ml[(k * G + h) * 2]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int k = 0; k < kCW; ++k) {
        const float mk = comb_ml[(k * G + h) * 2];
        const float wk = (mk == -INFINITY) ? 0.f : exp2f(mk - M);
        L = fmaf(wk, comb_ml[(k * G + h) * 2 + 1], L);
        O = fmaf(wk, comb[(k * G + h) * kHD + d], O);
      }
      const int64_t row = (int64_t)u.b * a.num_q_heads + hq0 + h;
      if (direct) {
        outp[row * kHD + d] = __float2bfloat16_rn(O / L);
      } else {
        const int64_t pidx = row * a.max_splits + u.s;
        a.ws_acc[pidx * kHD + d] = O;
        if (d == 0) {
          a.ws_ml[pidx * 2 + 0] = M;
          a.ws_ml[pidx * 2 + 1] = L;
        }
      }
    }
    named_bar_sync(1, kConsumersM);
  }
}

template <int G, bool FUSE>
cudaError_t launch_g(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  using C = MCfg<G>;
  CUtensorMap tm_k, tm_v;
  const int64_t rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  if (!encode_pool_map_bf16(&tm_k, a.k_cache, rows) || !encode_pool_map_bf16(&tm_v, a.v_cache, rows))
    return cudaErrorInvalidValue;
  const size_t smem = C::OFF_CU + sizeof(int) * (size_t)(a.num_seqs + 1) + 1024;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<G, FUSE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int per_sm = smem <= 113 * 1024 ? 2 : 1;
  const int64_t upper = (int64_t)a.num_seqs * a.num_kv_heads * a.max_splits;
  const int grid = (int)(upper < (int64_t)num_sms * per_sm ? upper : (int64_t)num_sms * per_sm);
  decode_mma_kernel<G, FUSE><<<grid, kThreadsM, smem, stream>>>(a, tm_k, tm_v);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  return launch_decode_reduce_bf16_128(a, stream);
}

}  // namespace

bool decode_mma_supported(int is_bf16, int head_dim, int group) {
  return is_bf16 && head_dim == 128 &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_paged_decode_mma(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  if (a.chunk_prior >= 0 || a.split_tokens % kStageTok != 0) return cudaErrorInvalidValue;
  const bool fuse = a.k_new != nullptr;
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return fuse ? launch_g<1, true>(a, num_sms, stream) : launch_g<1, false>(a, num_sms, stream);
    case 2: return fuse ? launch_g<2, true>(a, num_sms, stream) : launch_g<2, false>(a, num_sms, stream);
    case 4: return fuse ? launch_g<4, true>(a, num_sms, stream) : launch_g<4, false>(a, num_sms, stream);
    case 8: return fuse ? launch_g<8, true>(a, num_sms, stream) : launch_g<8, false>(a, num_sms, stream);
    case 16: return fuse ? launch_g<16, true>(a, num_sms, stream) : launch_g<16, false>(a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
