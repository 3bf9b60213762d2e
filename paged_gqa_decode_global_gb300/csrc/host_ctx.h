// Host-side identity of the CUDA context current on the calling thread.
//
// Per-context state of the library (the shared-memory limit raised on each
// kernel instance, the allocation-free entry point's scratch address) is kept
// under the context's process-unique id rather than the device number: a
// caller may make a non-primary context current, or make the primary context
// again after cudaDeviceReset, and either starts from nothing.
#pragma once

#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

namespace pd {

// A driver entry point fetched through the runtime (the library does not
// link libcuda); nullptr if the driver lacks it.
inline void* driver_fn(const char* name) {
  void* sym = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &sym, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return sym;
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

// The two entry points, fetched once; nullptr if either is missing.
inline const CtxFns* ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    fns.get_current = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
    fns.get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
  });
  return (fns.get_current && fns.get_id) ? &fns : nullptr;
}

// The id of the context current on this thread, or 0 if there is none yet.
inline unsigned long long current_ctx_id(const CtxFns& f) {
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace pd
