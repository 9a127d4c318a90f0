// Context identity and the per-context cache of kernel shared-memory
// attributes (see host_cache.h).
#include <cuda.h>

#include <map>
#include <mutex>
#include <utility>

#include "host_cache.h"

namespace pkv {
namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static const DriverFns fns = [] {
    DriverFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    return f;
  }();
  return fns;
}

std::mutex g_attr_mu;
// (context id, kernel) -> dynamic shared memory already allowed
std::map<std::pair<uint64_t, const void*>, int> g_attr;

}  // namespace

uint64_t current_context_id() {
  const DriverFns& f = driver_fns();
  if (!f.get_current || !f.get_id) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return (uint64_t)id;
}

cudaError_t allow_dynamic_smem(const void* func, int bytes) {
  const uint64_t ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (ctx != 0) {
    auto it = g_attr.find({ctx, func});
    if (it != g_attr.end() && it->second >= bytes) return cudaSuccess;
  }
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && ctx != 0) {
    if (g_attr.size() > 4096) g_attr.clear();   // stale contexts: start over
    int& v = g_attr[{ctx, func}];
    if (bytes > v) v = bytes;
  }
  return e;
}

}  // namespace pkv
