// Per-head projections for the latent (MLA-style) cache, on warp-level bf16
// tensor-core tiles: Y[b][h][:] = X[b][h][:] . W[h] for every row b and head
// h, with W[h] a 128 x 128 matrix.
//   * the query absorption q~_h = W_K[h]^T q_h takes W_K[h] stored [D][r]
//     as [K][N] (W_IS_NK = false);
//   * the output up-projection o_h = W_V[h] z_h takes W_V[h] stored [D][r]
//     as [N][K] (W_IS_NK = true).
// One CTA of 4 warps covers one head, 64 rows and a quarter (32 columns) of
// the output, so that a decode batch of 64-128 rows still spreads over 256-512
// CTAs.  The CTA's 32 columns of W[h] are staged in shared memory with rows
// padded to 16 bytes beyond their length, so the ldmatrix reads of the B
// fragments (transposed for [K][N]) are free of bank conflicts; a warp computes
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

template <bool W_IS_NK>
__global__ void __launch_bounds__(128) gemm_heads_kernel(__nv_bfloat16* __restrict__ y,
                                                         const __nv_bfloat16* __restrict__ x,
                                                         const __nv_bfloat16* __restrict__ wts,
                                                         int rows, int heads) {
  constexpr int kQ = 32;                 // output columns per CTA
  // [K][N]: 128 k-rows x 32 columns (row 40 elements); [N][K]: 32 n-rows x 128 k
  __shared__ __align__(16) __nv_bfloat16 ws[W_IS_NK ? kQ * kGRow : kGD * (kQ + 8)];
  const int h = blockIdx.y, n0 = blockIdx.z * kQ;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const __nv_bfloat16* wh = wts + (int64_t)h * kGD * kGD;
  if (W_IS_NK) {   // rows n0 .. n0+31 of W[n][k], 16 chunks each
    for (int i = tid; i < kQ * 16; i += 128) {
      const int r = i >> 4, c = i & 15;
      *reinterpret_cast<uint4*>(ws + r * kGRow + c * 8) =
          __ldg(reinterpret_cast<const uint4*>(wh + (int64_t)(n0 + r) * kGD) + c);
    }
  } else {         // columns n0 .. n0+31 of every row of W[k][n], 4 chunks each
    for (int i = tid; i < kGD * 4; i += 128) {
      const int r = i >> 2, c = i & 3;
      *reinterpret_cast<uint4*>(ws + r * (kQ + 8) + c * 8) =
          __ldg(reinterpret_cast<const uint4*>(wh + (int64_t)r * kGD + n0) + c);
    }
  }
  __syncthreads();
  const int r0 = blockIdx.x * 64 + warp * 16;
  if (r0 >= rows) return;
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
      if (W_IS_NK) {
        const int n = np * 16 + ((mi >> 1) << 3) + rr;
        const int k = ks * 16 + ((mi & 1) << 3);
        ldsm4(wbase + (uint32_t)(n * kGRow + k) * 2, b);
      } else {
        const int k = ks * 16 + ((mi & 1) << 3) + rr;
        const int n = np * 16 + ((mi >> 1) << 3);
        ldsm4_t(wbase + (uint32_t)(k * (kQ + 8) + n) * 2, b);
      }
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

}  // namespace

cudaError_t launch_gemm_heads(void* y, const void* x, const void* w, int rows, int heads,
                              bool w_is_nk, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((rows + 63) / 64, heads, kGD / 32);
  if (w_is_nk)
    gemm_heads_kernel<true><<<grid, 128, 0, stream>>>(
        static_cast<__nv_bfloat16*>(y), static_cast<const __nv_bfloat16*>(x),
        static_cast<const __nv_bfloat16*>(w), rows, heads);
  else
    gemm_heads_kernel<false><<<grid, 128, 0, stream>>>(
        static_cast<__nv_bfloat16*>(y), static_cast<const __nv_bfloat16*>(x),
        static_cast<const __nv_bfloat16*>(w), rows, heads);
  return cudaGetLastError();
}

}  // namespace pkv
