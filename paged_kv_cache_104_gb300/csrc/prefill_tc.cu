// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05).
//
// What it computes ("The KV cache is not your bottleneck", section "The fix
// that mattered": prompts are admitted in capped chunks; "KV cache and
// continuous batching: 1,000 people ask AI", section "What does a KV cache
// keep?": prefill is matrix-matrix work): a chunk of C prompt tokens of one
// sequence, at absolute positions prior .. prior+C-1, whose keys and values
// were already appended to the paged pools, attends causally over the
// sequence: row i sees keys 0 .. prior+i.  out[i][h] = softmax(scale *
// q[i][h] . K[:, h/G]) V[:, h/G] over those keys.
//
// CTA = 128 query rows of one query head; keys stream in tiles of 64 (four
// 16-token blocks gathered through the block table by 2-D TMA with 128-byte
// swizzle, which is the canonical K-major operand layout).  A CTA needs
// 112 KiB of shared memory and 256 TMEM columns, so two CTAs share an SM and
// their softmax warpgroups take turns with one tensor core.
//   warp 4      TMA producer: Q once, then K/V tiles into a 2-stage ring;
//               blocks past the end of the sequence are fetched at an
//               out-of-range coordinate, which the TMA unit fills with zeros
//   warp 5      TMEM allocator and single-thread MMA issuer:
//               S[j%2] = Q K_j^T  (M=128, N=64, K=128, bf16 -> fp32 in TMEM)
//               O     += P_j V_j  (M=128, N=128, K=64; P from shared memory,
//                                  V as an MN-major operand)
//   warps 0-3   softmax: thread r owns query row r = TMEM lane r; reads its S
//               row with tcgen05.ld, applies the causal mask on diagonal
//               tiles, keeps a running max (raised lazily, only when it grows
//               by more than 2^8) and sum, forms p = 2^(s*scale*log2e - m) with
//               one FMA and ex2 per score, writes P (bf16) into the swizzled
//               A-operand tile, and rescales its O row in TMEM when the max
//               moved.  Epilogue: O / l.
// S is double-buffered in TMEM so Q K_{j+1}^T runs while the softmax of tile
// j does; fully masked key tiles are never visited.
// Every mbarrier wait is bounded; on time-out the kernel records an error,
// stops issuing work, lets its copies land, frees its TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace pkv {
namespace {

constexpr int BM = 128, BN = 64, HD = 128;
constexpr int QHALF = BM * 128;           // Q: one 64-column half of 128 rows, 16 KiB
constexpr int Q_BYTES = 2 * QHALF;        // 32 KiB
constexpr int KHALF = BN * 128;           // K or V: one 64-column half of 64 keys, 8 KiB
constexpr int KV_TILE = 2 * KHALF;        // 16 KiB
constexpr int NSTAGE = 2;
constexpr int P_BYTES = BM * 128;         // P: 128 rows x 64 keys bf16, 16 KiB
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + Q_BYTES;
constexpr int OFF_V = OFF_K + NSTAGE * KV_TILE;
constexpr int OFF_P = OFF_V + NSTAGE * KV_TILE;
constexpr int OFF_BAR = OFF_P + P_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 128;  // 112 KiB + barriers: two CTAs per SM
constexpr int kThreadsTC = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t COL_S0 = 0, COL_O = 2 * BN;
constexpr float kLazy = 8.0f;

// barrier slots (8 bytes each) inside OFF_BAR
enum { B_Q = 0, B_KV_FULL = 1, B_KV_EMPTY = 3, B_S_FULL = 5, B_S_FREE = 7, B_P_FULL = 9,
       B_O_DONE = 10, B_COUNT = 11 };

struct TcParams {
  PrefillArgs a;
  int total_len;     // prior + chunk
  int kv_rows;       // num_blocks * Hkv * 16 (rows of the 2-D pool view)
  int q_tiles;
};

__global__ void __launch_bounds__(kThreadsTC, 2)
prefill_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  int* abort_i = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort_flag = abort_i;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const PrefillArgs& a = p.a;
  // The swizzled operand tiles need a 1 KiB-aligned base; there is no room
  // for slack at two CTAs per SM, so refuse (and report) rather than misread.
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_error(a.err, DEVERR_SMEM_LAYOUT);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;                              // query head
  const int qt = p.q_tiles - 1 - (int)blockIdx.y;        // heaviest tiles first
  const int q0 = qt * BM;
  const int g = h / (a.num_q_heads / a.num_kv_heads);    // KV head of the group
  const int last_row_pos = a.prior_len + min(a.chunk_len, q0 + BM) - 1;
  const int n_tiles = last_row_pos / BN + 1;             // key tiles with any visible key

  if (tid == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_KV_EMPTY + s), 1);
      mbar_init(bar(B_S_FULL + s), 1);
      mbar_init(bar(B_S_FREE + s), 128);
    }
    mbar_init(bar(B_P_FULL), 128);
    mbar_init(bar(B_O_DONE), 1);
    *abort_i = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      mbar_arrive_expect_tx(bar(B_Q), Q_BYTES);
      tma_load_3d(sbase + OFF_Q, &tm_q, bar(B_Q), 0, h, q0);
      tma_load_3d(sbase + OFF_Q + QHALF, &tm_q, bar(B_Q), 64, h, q0);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        if (j >= 2 && !wait_or_abort(bar(B_KV_EMPTY + st), ((j >> 1) - 1) & 1, abort_flag, a.err))
          break;
        if (*abort_flag) break;
        mbar_arrive_expect_tx(bar(B_KV_FULL + st), 2 * KV_TILE);
        const uint32_t kd = sbase + OFF_K + st * KV_TILE, vd = sbase + OFF_V + st * KV_TILE;
#pragma unroll
        for (int i = 0; i < BN / kBlockSize; ++i) {
          const int tok = j * BN + i * kBlockSize;
          int y = p.kv_rows;  // past the end: zero fill
          if (tok < p.total_len) {
            int blk = __ldg(a.block_table_row + tok / kBlockSize);
            if (blk < 0 || (int64_t)blk >= a.num_blocks) {
              record_error(a.err, DEVERR_BLOCK_RANGE);
              blk = 0;
            }
            y = (blk * a.num_kv_heads + g) * kBlockSize;
          }
          const uint32_t off = i * kBlockSize * 128;  // 16 rows x 128 B
          tma_load_2d(kd + off, &tm_k, bar(B_KV_FULL + st), 0, y);
          tma_load_2d(kd + KHALF + off, &tm_k, bar(B_KV_FULL + st), 64, y);
          tma_load_2d(vd + off, &tm_v, bar(B_KV_FULL + st), 0, y);
          tma_load_2d(vd + KHALF + off, &tm_v, bar(B_KV_FULL + st), 64, y);
        }
        issued = j + 1;
      }
      if (*abort_flag) {  // let the loads already issued land
        mbar_wait(bar(B_Q), 0, nullptr);
        for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j)
          mbar_wait(bar(B_KV_FULL + (j & 1)), (j >> 1) & 1, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(false, BM, BN);
      constexpr uint32_t idesc_pv = make_idesc(true, BM, HD);
      bool ok = wait_or_abort(bar(B_Q), 0, abort_flag, a.err);
      tc_fence_after();
      auto issue_pv = [&](int jj) {
        const int st = jj & 1;
        if (!wait_or_abort(bar(B_P_FULL), jj & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t pa = sbase + OFF_P, vb = sbase + OFF_V + st * KV_TILE;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t ad = make_sw128_desc(pa + k * 32, 16, 1024);
          const uint64_t bd = make_sw128_desc(vb + k * 16 * 128, KHALF, 1024);
          mma_bf16(tmem + COL_O, ad, bd, idesc_pv, (jj > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(B_O_DONE));
        mma_commit(bar(B_KV_EMPTY + st));
        return true;
      };
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int st = j & 1, sb = j & 1;
        ok = wait_or_abort(bar(B_KV_FULL + st), (j >> 1) & 1, abort_flag, a.err);
        if (ok && j >= 2) ok = wait_or_abort(bar(B_S_FREE + sb), ((j >> 1) - 1) & 1, abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qa = sbase + OFF_Q, kb = sbase + OFF_K + st * KV_TILE;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint64_t ad = make_sw128_desc(qa + (k >> 2) * QHALF + (k & 3) * 32, 16, 1024);
          const uint64_t bd = make_sw128_desc(kb + (k >> 2) * KHALF + (k & 3) * 32, 16, 1024);
          mma_bf16(tmem + COL_S0 + sb * BN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(B_S_FULL + sb));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n_tiles - 1);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int r = tid;                      // query row in the tile, TMEM lane
    const int row_pos = a.prior_len + q0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = a.scale * 1.4426950408889634f;
    float m_run = -INFINITY, l_run = 0.f;   // running max in scaled log2 units
    unsigned char* prow = smem + OFF_P + r * 128;
    const int sw = r & 7;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      wait_or_abort(bar(B_S_FULL + sb), (j >> 1) & 1, abort_flag, a.err);
      __syncwarp();
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        float t[32];
        tmem_ld32(lane_base + COL_S0 + sb * BN + c * 32, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = t[i];
      }
      tmem_wait_ld();
      reg_fence(s);
      tc_fence_before();
      mbar_arrive(bar(B_S_FREE + sb));
      // causal mask: key k visible iff k <= row_pos (only tiles that reach past
      // the first row of this query tile need it)
      const int k0 = j * BN;
      const bool masked = k0 + BN - 1 > a.prior_len + q0;
      if (masked) {
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = (k0 + c <= row_pos) ? s[c] : -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1];
#pragma unroll
      for (int c = 2; c < BN; c += 2) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
      }
      const float mx = fmaxf(mx0, mx1) * sl2;   // scale > 0 commutes with max
      float m_new = m_run;
      if (mx > m_run + kLazy || m_run == -INFINITY) m_new = mx;
      const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t packed[BN / 2];
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float p0 = fast_exp2(fmaf(s[c], sl2, -m_new));       // exp2(-inf) = 0
        const float p1 = fast_exp2(fmaf(s[c + 1], sl2, -m_new));
        sum0 += p0;
        sum1 += p1;
        packed[c / 2] = pack_bf16(p0, p1);
      }
      // P_{j-1} . V must be finished before P is overwritten or O rescaled
      if (j >= 1) {
        wait_or_abort(bar(B_O_DONE), (j - 1) & 1, abort_flag, a.err);
        __syncwarp();
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            float o[32];
            tmem_ld32(lane_base + COL_O + c * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(lane_base + COL_O + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      l_run = l_run * alpha + (sum0 + sum1);
      m_run = m_new;
      // the last tile may hold stale rows past the sequence end: zero their V
      if (j == n_tiles - 1 && k0 + BN > p.total_len) {
        wait_or_abort(bar(B_KV_FULL + (j & 1)), (j >> 1) & 1, abort_flag, a.err);
        if (r < BN && k0 + r >= p.total_len) {
          unsigned char* vrow = smem + OFF_V + (j & 1) * KV_TILE + r * 128;
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = z;
            *reinterpret_cast<uint4*>(vrow + KHALF + c * 16) = z;
          }
        }
      }
      // write P row r into the 128B-swizzled K-major tile
#pragma unroll
      for (int cc = 0; cc < BN / 8; ++cc) {
        uint4 v = make_uint4(packed[cc * 4 + 0], packed[cc * 4 + 1], packed[cc * 4 + 2],
                             packed[cc * 4 + 3]);
        *reinterpret_cast<uint4*>(prow + ((cc ^ sw) << 4)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL));
    }
    // epilogue: O / l
    wait_or_abort(bar(B_O_DONE), (n_tiles - 1) & 1, abort_flag, a.err);
    __syncwarp();
    tc_fence_after();
    const float inv = 1.f / l_run;
    const bool row_ok = (q0 + r) < a.chunk_len;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                          ((int64_t)(q0 + r) * a.num_q_heads + h) * HD;
#pragma unroll 1
    for (int c = 0; c < HD / 32; ++c) {
      float o[32];
      tmem_ld32(lane_base + COL_O + c * 32, o);
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
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  TcParams p;
  p.a = a;
  p.total_len = a.prior_len + a.chunk_len;
  const int64_t kv_rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  if (kv_rows >= (1ll << 31) - 1) return cudaErrorInvalidValue;
  p.kv_rows = (int)kv_rows;
  p.q_tiles = (a.chunk_len + BM - 1) / BM;
  if (p.q_tiles == 0) return cudaSuccess;
  CUtensorMap tm_q, tm_k, tm_v;
  if (!encode_rows_map_bf16(&tm_q, a.q, a.chunk_len, a.num_q_heads) ||
      !encode_pool_map_bf16(&tm_k, a.k_cache, kv_rows) ||
      !encode_pool_map_bf16(&tm_v, a.v_cache, kv_rows))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_q_heads, p.q_tiles);
  prefill_tc_kernel<<<grid, kThreadsTC, SMEM_BYTES, stream>>>(p, tm_q, tm_k, tm_v);
  return cudaGetLastError();
}

}  // namespace pkv
