// Per-head projections for the latent (MLA-style) cache, on warp-level bf16
// tensor-core tiles: Y[b][h][:] = X[b][h][:] . W[h] for every row b and head
// h, with W[h] a 128 x 128 matrix.
//   * the query absorption q~_h = W_K[h]^T q_h takes W_K[h] stored [D][r]
//     as [K][N] (W_IS_NK = false);
//   * the output up-projection o_h = W_V[h] z_h takes W_V[h] stored [D][r]
//     as [N][K] (W_IS_NK = true).
// One CTA of 4 warps covers one head and 64 rows; a warp computes a 16 x 128
// tile with 128 m16n8k16 products, reading W straight from global memory
// (32 KiB per head, cached).  Output in bf16, fp32 accumulation.
#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kGD = 128;   // K = N = 128

__device__ __forceinline__ void mma16816g(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld_pair(const uint16_t* p0, const uint16_t* p1) {
  return (uint32_t)__ldg(p0) | ((uint32_t)__ldg(p1) << 16);
}

template <bool W_IS_NK>
__global__ void __launch_bounds__(128) gemm_heads_kernel(__nv_bfloat16* __restrict__ y,
                                                         const __nv_bfloat16* __restrict__ x,
                                                         const __nv_bfloat16* __restrict__ wts,
                                                         int rows, int heads) {
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = blockIdx.x * 64 + warp * 16;
  if (r0 >= rows) return;
  const uint16_t* w = reinterpret_cast<const uint16_t*>(wts) + (int64_t)h * kGD * kGD;
  // A fragments of X rows r0 + g and r0 + g + 8 (zero past the last row)
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
  float acc[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int col = n * 8 + g;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int k0 = ks * 16 + 2 * t;
      uint32_t b0, b1;
      if (W_IS_NK) {   // W[col][k] contiguous in k
        const uint32_t* wr = reinterpret_cast<const uint32_t*>(w + (int64_t)col * kGD);
        b0 = __ldg(wr + (k0 >> 1));
        b1 = __ldg(wr + ((k0 + 8) >> 1));
      } else {         // W[k][col]
        b0 = ld_pair(w + (int64_t)k0 * kGD + col, w + (int64_t)(k0 + 1) * kGD + col);
        b1 = ld_pair(w + (int64_t)(k0 + 8) * kGD + col, w + (int64_t)(k0 + 9) * kGD + col);
      }
      mma16816g(acc[n], af[ks][0], af[ks][1], af[ks][2], af[ks][3], b0, b1);
    }
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int col = n * 8 + 2 * t;
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
  const dim3 grid((rows + 63) / 64, heads);
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
