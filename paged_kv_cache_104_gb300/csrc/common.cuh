// Device helpers shared by the paged-KV kernels: mbarriers with bounded
// waits, 1-D bulk (TMA) copies, bf16 unpacking, error reporting.
//
// Every wait on an mbarrier is bounded: after about a second (kWaitLimitCycles
// SM cycles, or kWaitLimitIters polls) it gives up, records PKV_DEVERR_TIMEOUT
// in the caller's error word and returns false.  Kernels never trap.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// device error codes written into the library's error word (first one wins)
enum DevErr : int {
  DEVERR_NONE = 0,
  DEVERR_SLOT_RANGE = 1,    // kv_append: slot beyond the pool
  DEVERR_BLOCK_RANGE = 2,   // a block-table entry outside [0, num_blocks)
  DEVERR_SEQLEN_RANGE = 3,  // a sequence length < 1 or beyond its bound
  DEVERR_TIMEOUT = 4,       // an mbarrier wait ran out of time
  DEVERR_SMEM_LAYOUT = 5,   // dynamic shared memory not 1 KiB aligned (kernel skipped)
};

// Wait limits: 2^31 SM cycles (about 1 s at GB300 clocks), checked every 64
// polls with the SM-local cycle counter (cheap, unlike %globaltimer), and at
// most 2^28 polls in any case.
#ifdef PKV_TEST_WAIT_TIMEOUT
// Test build only (never the shipped library): waits give up after 2^22
// cycles, about 2 ms, so a test can make one run out quickly.
constexpr long long kWaitLimitCycles = 1ll << 22;
#else
constexpr long long kWaitLimitCycles = 1ll << 31;
#endif
constexpr unsigned int kWaitLimitIters = 1u << 28;

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most about
// one second.  Returns false (and records DEVERR_TIMEOUT) on time-out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned int it = 0; it < kWaitLimitIters; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && clock64() - t0 > kWaitLimitCycles) break;
  }
  record_error(err, DEVERR_TIMEOUT);
  return false;
}

// 1-D bulk copy global -> shared, completing on an mbarrier (TMA engine), with
// an L2 eviction-priority hint (createpolicy result).  dst, src 16-byte
// aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// fp16 store carrying an L2 eviction-priority hint.
__device__ __forceinline__ void st_global_hint_f16(__half* dst, __half v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(dst),
               "h"(__half_as_ushort(v)), "l"(policy)
               : "memory");
}

// Drop one 128-byte L2 line without writing it back: its contents become
// undefined.  For scratch that is dead once read; line must be 128-byte
// aligned and hold nothing else that is still live.
__device__ __forceinline__ void discard_l2_line(const void* line) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(__cvta_generic_to_global(line)) : "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Storage <-> fp32.  bf16 is the top half of a binary32, so widening is a
// shift; narrowing rounds to nearest even (__float2bfloat16_rn).
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// A measurement aid: the earliest start and the latest end of a grid's CTAs,
// in %globaltimer nanoseconds, into span[0] (atomic min) and span[1]
// (atomic max).  Called by one thread of a CTA; span null: nothing.
__device__ __forceinline__ void span_mark(unsigned long long* span, bool end) {
  if (span) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (end) atomicMax(span + 1, t);
    else atomicMin(span, t);
  }
}

// fp8 (E4M3) conversions, hardware rounding: f32 -> e4m3 rounds to nearest
// even and saturates finite values at +-448; e4m3 -> f16 is exact.
// Element order follows memory order: `lo` is the byte / half at the lower address.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPer16B = 4;
  __device__ __forceinline__ static void unpack(const uint4& c, float (&f)[4]) {
    f[0] = __uint_as_float(c.x);
    f[1] = __uint_as_float(c.y);
    f[2] = __uint_as_float(c.z);
    f[3] = __uint_as_float(c.w);
  }
  __device__ __forceinline__ static void store(float* p, float v) { *p = v; }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPer16B = 8;
  __device__ __forceinline__ static void unpack(const uint4& c, float (&f)[8]) {
    f[0] = bf16lo(c.x); f[1] = bf16hi(c.x);
    f[2] = bf16lo(c.y); f[3] = bf16hi(c.y);
    f[4] = bf16lo(c.z); f[5] = bf16hi(c.z);
    f[6] = bf16lo(c.w); f[7] = bf16hi(c.w);
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
};

}  // namespace pkv
