// Host-side state the launchers keep between calls: the identity of the
// current CUDA context, and the dynamic shared-memory size each kernel was
// last allowed per context.  Internal to the library; thread-safe.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Unique id of the context current on this thread (cuCtxGetId), or 0 when
// none is current or the driver cannot say.  A device reset destroys the
// primary context; the one created after it has another id, so state
// resolved in the old context (symbol addresses, function attributes) can be
// told apart from state valid now.
uint64_t current_context_id();

// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes), made only
// when this context has not already allowed func at least `bytes`.
cudaError_t allow_dynamic_smem(const void* func, int bytes);

template <typename F>
cudaError_t allow_dynamic_smem(F* func, int bytes) {
  return allow_dynamic_smem(reinterpret_cast<const void*>(func), bytes);
}

}  // namespace pkv
