// Per-head projections for the latent (MLA-style) cache, on warp-level bf16
// tensor-core tiles (mma.sync m16n8k16, fp32 accumulate).
//   * The query absorption q~_h = W_K[h]^T q_h: Y[b][h][:] = X[b][h][:] . W[h]
//     for every row b and head h, with W[h] = W_K[h] stored [D][r] = [K][N].
//   * The merge of the latent attention's split partials fused with the
//     output up-projection o_h = W_V[h] z_h (W_V[h] stored [D][r] = [N][K]);
//     see merge_project_kernel.
// The absorption's launch can also place each decode sequence's new latent
// in the pool (the CTAs of the first column quarter, a few rows each).
// Absorption: one CTA of 4 warps covers one head, 64 rows and a quarter (32 columns) of
// the output, so that a decode batch of 64-128 rows still spreads over 256-512
// CTAs.  The CTA's 32 columns of W[h] are staged in shared memory with rows
// padded to 16 bytes beyond their length, so the transposing ldmatrix reads of
// the B fragments are free of bank conflicts; a warp computes
// a 16 x 32 tile with 32 m16n8k16 products.  bf16 out, fp32 accumulation.
#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kGD = 128;            // K = N = 128
constexpr int kGRow = kGD + 8;      // padded smem row (elements)

__device__ __forceinline__ void mma16816g(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__global__ void __launch_bounds__(128) gemm_heads_kernel(__nv_bfloat16* __restrict__ y,
                                                         const __nv_bfloat16* __restrict__ x,
                                                         const __nv_bfloat16* __restrict__ wts,
                                                         int rows, int heads,
                                                         const LatentAppend app) {
  // a kernel launched next as a programmatic dependent (the latent
  // attention) may start now; it waits for this grid before reading y or
  // the pool
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kQ = 32;                 // output columns per CTA
  // 128 k-rows x this CTA's 32 columns (rows of 40 elements)
  __shared__ __align__(16) __nv_bfloat16 ws[kGD * (kQ + 8)];
  const int h = blockIdx.y, n0 = blockIdx.z * kQ;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (app.c_new && blockIdx.z == 0) {
    // the new latents of this CTA's 64-row block, spread over its heads'
    // CTAs (2 rows each for 32 heads): one 16-byte chunk per thread, copied
    // to position seq_lens[r] - 1 (bit-exact; bad lengths or block ids are
    // skipped, and block ids reported).  The chunk is requested first, so
    // it arrives while the length and the block id are looked up.
    const int per = (64 + heads - 1) / heads;
    const int row_end = min(rows, blockIdx.x * 64 + 64);
    for (int i = tid; i < per * 16; i += 128) {
      const int r = blockIdx.x * 64 + blockIdx.y * per + (i >> 4), c = i & 15;
      if (r >= row_end) break;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                          static_cast<const __nv_bfloat16*>(app.c_new) + (int64_t)r * kGD) + c);
      const int n = __ldg(app.seq_lens + r);
      if (n < 1 || n > app.max_len) continue;
      const int blk = __ldg(app.block_table + (int64_t)r * app.bt_stride + (n - 1) / kBlockSize);
      if (blk < 0 || (int64_t)blk >= app.num_blocks) {
        record_error(app.err, DEVERR_BLOCK_RANGE);
        continue;
      }
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(app.c_cache) +
                               ((int64_t)blk * kBlockSize + (n - 1) % kBlockSize) * kGD)[c] = v;
    }
  }
  const int g = lane >> 2, t = lane & 3;
  const __nv_bfloat16* wh = wts + (int64_t)h * kGD * kGD;
  // this warp's 16 rows of x first: their loads overlap the staging of W
  const int r0 = blockIdx.x * 64 + warp * 16;
  uint32_t af[8][4];
  const int ra = r0 + g, rb = r0 + g + 8;
  const uint32_t* xa = reinterpret_cast<const uint32_t*>(x + ((int64_t)ra * heads + h) * kGD);
  const uint32_t* xb = reinterpret_cast<const uint32_t*>(x + ((int64_t)rb * heads + h) * kGD);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    af[ks][0] = ra < rows ? __ldg(xa + ks * 8 + t) : 0u;
    af[ks][1] = rb < rows ? __ldg(xb + ks * 8 + t) : 0u;
    af[ks][2] = ra < rows ? __ldg(xa + ks * 8 + 4 + t) : 0u;
    af[ks][3] = rb < rows ? __ldg(xb + ks * 8 + 4 + t) : 0u;
  }
  // columns n0 .. n0+31 of every row of W[k][n], 4 chunks each (a thread's
  // four pieces requested before any is stored)
  {
    uint4 wv[kGD * 4 / 128];
#pragma unroll
    for (int j = 0; j < kGD * 4 / 128; ++j) {
      const int i = tid + j * 128, r = i >> 2, c = i & 3;
      wv[j] = __ldg(reinterpret_cast<const uint4*>(wh + (int64_t)r * kGD + n0) + c);
    }
#pragma unroll
    for (int j = 0; j < kGD * 4 / 128; ++j) {
      const int i = tid + j * 128, r = i >> 2, c = i & 3;
      *reinterpret_cast<uint4*>(ws + r * (kQ + 8) + c * 8) = wv[j];
    }
  }
  __syncthreads();
  if (r0 >= rows) return;
  const uint32_t wbase = smem_u32(ws);
  const int mi = lane >> 3, rr = lane & 7;
  float acc[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
    for (int np = 0; np < 2; ++np) {      // pairs of 8-column n-tiles within the 32
      uint32_t b[4];
      const int k = ks * 16 + ((mi & 1) << 3) + rr;
      const int n = np * 16 + ((mi >> 1) << 3);
      ldsm4_t(wbase + (uint32_t)(k * (kQ + 8) + n) * 2, b);
      mma16816g(acc[2 * np], af[ks][0], af[ks][1], af[ks][2], af[ks][3], b[0], b[1]);
      mma16816g(acc[2 * np + 1], af[ks][0], af[ks][1], af[ks][2], af[ks][3], b[2], b[3]);
    }
  }
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const int col = n0 + n * 8 + 2 * t;
    if (ra < rows)
      *reinterpret_cast<__nv_bfloat162*>(y + ((int64_t)ra * heads + h) * kGD + col) =
          __floats2bfloat162_rn(acc[n][0], acc[n][1]);
    if (rb < rows)
      *reinterpret_cast<__nv_bfloat162*>(y + ((int64_t)rb * heads + h) * kGD + col) =
          __floats2bfloat162_rn(acc[n][2], acc[n][3]);
  }
}

// Merge of the latent attention's split partials fused with the output
// up-projection: for 16 sequences and one head h per CTA,
//   z[b][h] = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s   (M = max_s m_s)
// (or the z row the attention wrote itself, for a sequence it covered in one
// piece), rounded to bf16, then o[b][h] = W_V[h] z[b][h] on m16n8k16 tiles
// with W_V[h] ([D][r] = [N][K]) staged in padded shared memory.  Eight warps:
// warp w merges rows 2w and 2w + 1 (lane = 4 of the 128 columns; the split
// weights are formed one split per lane), then computes output columns
// 16w .. 16w + 15.  W_V[h] is loaded before the grid waits for
// the attention kernel it depends on (programmatic dependent launch), so that
// load overlaps the attention's tail.
constexpr int kMRows = 16;
constexpr int kMThreads = 256;

// z of rows b[0], b[1] (lane = 4 of the 128 columns).  Every load a row may
// need -- its length, its partial count, its z row, the (m, l) pair of split
// `lane` and the first eight partial rows -- is issued before any is used
// (all lie inside the row's slots, so the ones the row turns out not to need
// are harmless), so the two rows cost about one memory latency, not three
// each.
__device__ __forceinline__ void merge_rows2(const DecodeArgs& a, const __nv_bfloat16* z,
                                            const int (&b)[2], int h, int lane, int limit,
                                            float4 (&o)[2]) {
  constexpr int kPre = 8;
  int n[2], np[2];
  int64_t base[2];
  uint2 zr[2];
  float ms[2], ls[2];
  float4 v[2][kPre];
  const float4* acc4 = reinterpret_cast<const float4*>(a.ws_acc);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const bool in = b[r] < a.num_seqs;
    const int64_t row = (int64_t)(in ? b[r] : 0) * a.num_q_heads + h;
    base[r] = row * a.max_splits;
    n[r] = in ? a.seq_lens[b[r]] : 0;
    np[r] = in && a.balanced ? a.ws_np[b[r]] : 0;
    zr[r] = *reinterpret_cast<const uint2*>(z + row * kGD + 4 * lane);
    ms[r] = -INFINITY;
    ls[r] = 0.f;
    if (a.max_splits > 1 && lane < a.max_splits) {
      ms[r] = a.ws_ml[(base[r] + lane) * 2];
      ls[r] = a.ws_ml[(base[r] + lane) * 2 + 1];
    }
#pragma unroll
    for (int i = 0; i < kPre; ++i)
      v[r][i] = (a.max_splits > 1 && i < a.max_splits) ? acc4[(base[r] + i) * (kGD / 4) + lane]
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    o[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (n[r] < 1 || n[r] > limit) continue;   // reported by the attention kernel
    const int ns = a.balanced ? np[r] : (n[r] + a.split_tokens - 1) / a.split_tokens;
    if (ns <= 1) {
      o[r] = make_float4(bf16lo(zr[r].x), bf16hi(zr[r].x), bf16lo(zr[r].y), bf16hi(zr[r].y));
      continue;
    }
    float M = lane < ns ? ms[r] : -INFINITY;
    for (int s = lane + 32; s < ns; s += 32) M = fmaxf(M, a.ws_ml[(base[r] + s) * 2]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += 32) {
      float wl = 0.f;
      if (s0 + lane < ns) {
        const float m_s = s0 == 0 ? ms[r] : a.ws_ml[(base[r] + s0 + lane) * 2];
        const float l_s = s0 == 0 ? ls[r] : a.ws_ml[(base[r] + s0 + lane) * 2 + 1];
        wl = m_s == -INFINITY ? 0.f : exp2f(m_s - M);
        L = fmaf(wl, l_s, L);
      }
      const int cnt = min(32, ns - s0);
      for (int k = 0; k < cnt; k += kPre) {
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
          if (k + i >= cnt) break;
          const float4 x = (s0 == 0 && k == 0) ? v[r][i]
                                               : acc4[(base[r] + s0 + k + i) * (kGD / 4) + lane];
          const float wgt = __shfl_sync(0xffffffffu, wl, (k + i) & 31);
          acc.x = fmaf(wgt, x.x, acc.x);
          acc.y = fmaf(wgt, x.y, acc.y);
          acc.z = fmaf(wgt, x.z, acc.z);
          acc.w = fmaf(wgt, x.w, acc.w);
        }
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float inv = 1.f / L;
    o[r] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
}

__global__ void __launch_bounds__(kMThreads) merge_project_kernel(const DecodeArgs a,
                                                                  const __nv_bfloat16* __restrict__ wts,
                                                                  __nv_bfloat16* __restrict__ y) {
  __shared__ __align__(16) __nv_bfloat16 ws[kGD * kGRow];
  __shared__ __align__(16) __nv_bfloat16 zs[kMRows * kGRow];
  const int h = blockIdx.y, b0 = blockIdx.x * kMRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const __nv_bfloat16* wh = wts + (int64_t)h * kGD * kGD;
  {
    // all eight of a thread's 16-byte pieces are requested before any is
    // stored: a CTA that starts only when the attention's last CTAs leave
    // its SM stages W_V in one memory latency, not eight
    constexpr int kPer = kGD * 16 / kMThreads;
    uint4 wv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid + j * kMThreads, r = i >> 4, c = i & 15;
      wv[j] = __ldg(reinterpret_cast<const uint4*>(wh + (int64_t)r * kGD) + c);
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid + j * kMThreads, r = i >> 4, c = i & 15;
      *reinterpret_cast<uint4*>(ws + r * kGRow + c * 8) = wv[j];
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // ---- z rows 2w, 2w + 1
  const int limit = min(a.max_seq_len, a.max_blocks_per_seq * kBlockSize);
  const __nv_bfloat16* z = static_cast<const __nv_bfloat16*>(a.out);
  {
    const int rows[2] = {b0 + 2 * warp, b0 + 2 * warp + 1};
    float4 o[2];
    merge_rows2(a, z, rows, h, lane, limit, o);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      __nv_bfloat162* zr = reinterpret_cast<__nv_bfloat162*>(zs + (2 * warp + rr) * kGRow + 4 * lane);
      zr[0] = __floats2bfloat162_rn(o[rr].x, o[rr].y);
      zr[1] = __floats2bfloat162_rn(o[rr].z, o[rr].w);
    }
  }
  __syncthreads();
  // ---- o = z W_V[h]^T for the 16 rows: this warp's 16 columns
  const int g = lane >> 2, t = lane & 3;
  const uint32_t wbase = smem_u32(ws), zbase = smem_u32(zs);
  const int mi = lane >> 3, rr8 = lane & 7;
  const int n0 = warp * 16;
  float acc[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t af[4], b[4];
    ldsm4(zbase + (uint32_t)((rr8 + ((mi & 1) << 3)) * kGRow + ks * 16 + ((mi >> 1) << 3)) * 2, af);
    const int n = n0 + ((mi >> 1) << 3) + rr8;
    const int k = ks * 16 + ((mi & 1) << 3);
    ldsm4(wbase + (uint32_t)(n * kGRow + k) * 2, b);
    mma16816g(acc[0], af[0], af[1], af[2], af[3], b[0], b[1]);
    mma16816g(acc[1], af[0], af[1], af[2], af[3], b[2], b[3]);
  }
  const int ra = b0 + g, rb = b0 + g + 8;
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const int col = n0 + n * 8 + 2 * t;
    if (ra < a.num_seqs)
      *reinterpret_cast<__nv_bfloat162*>(y + ((int64_t)ra * a.num_q_heads + h) * kGD + col) =
          __floats2bfloat162_rn(acc[n][0], acc[n][1]);
    if (rb < a.num_seqs)
      *reinterpret_cast<__nv_bfloat162*>(y + ((int64_t)rb * a.num_q_heads + h) * kGD + col) =
          __floats2bfloat162_rn(acc[n][2], acc[n][3]);
  }
}

}  // namespace

cudaError_t launch_merge_project(const DecodeArgs& a, const void* w_v, void* out,
                                 cudaStream_t stream) {
  if (a.num_seqs <= 0) return cudaSuccess;
  if (a.head_dim != kGD || a.num_kv_heads != 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.num_seqs + kMRows - 1) / kMRows, a.num_q_heads);
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, merge_project_kernel, a,
                                           static_cast<const __nv_bfloat16*>(w_v),
                                           static_cast<__nv_bfloat16*>(out));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm_heads(void* y, const void* x, const void* w, int rows, int heads,
                              cudaStream_t stream, const LatentAppend* app) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((rows + 63) / 64, heads, kGD / 32);
  const LatentAppend none{};
  gemm_heads_kernel<<<grid, 128, 0, stream>>>(static_cast<__nv_bfloat16*>(y),
                                              static_cast<const __nv_bfloat16*>(x),
                                              static_cast<const __nv_bfloat16*>(w), rows, heads,
                                              app ? *app : none);
  return cudaGetLastError();
}

}  // namespace pkv
