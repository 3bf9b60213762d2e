// paged_decode_noalloc: one decode layer-step (stage 1 + merge) for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not allowed or not wise —
// a plugin inside an inference engine whose host owns every device allocation
// through its own arena, a serving loop that budgets all device memory up front,
// or any caller whose allocation would synchronise the device in the middle of
// a latency-critical step. Such callers cannot provide the workspace the other
// entry points take, so this one uses scratch memory the library carries itself.
//
// The scratch is a file-scope device array of kScratchBytes (8 MiB). Every GPU
// that loads this library holds it until the process exits. A __device__
// array has one address per CUDA context, so its address is looked up
// (cudaGetSymbolAddress) on the first call made in each context and kept under
// that context's unique id: a non-primary context, or a primary context made
// again after cudaDeviceReset, gets its own lookup. That first call in a
// context should therefore happen before any stream capture. All calls share
// the one array: calls that overlap on the GPU (two streams, or two host
// threads) race on it, so order them on one stream. Nothing here allocates:
// no cudaMalloc, no cudaFree, no library call that allocates.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "host_ctx.h"
#include "paged_decode.h"

namespace pd {
bool plan_is_valid(const pd_plan* plan);
}

namespace {

constexpr size_t kScratchBytes = 8u << 20;
constexpr int kMaxContexts = 64;

// Partials, log-sum-exps and the device error word of the calls below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
struct Entry {
  unsigned long long ctx_id;
  void* ptr;
};
Entry g_cache[kMaxContexts] = {};
int g_cached = 0;

// Device address of g_scratch in the current context.
pd_status scratch_for_current_context(void** out) {
  const pd::CtxFns* f = pd::ctx_fns();
  if (!f) return PD_ERR_CUDA;
  unsigned long long id = pd::current_ctx_id(*f);
  std::lock_guard<std::mutex> lock(g_mu);
  if (id != 0) {
    for (int i = 0; i < g_cached; ++i)
      if (g_cache[i].ctx_id == id) {
        *out = g_cache[i].ptr;
        return PD_OK;
      }
  }
  // first call in this context (with no context current yet, this runtime call
  // makes the current device's primary context current)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
    (void)cudaGetLastError();
    return PD_ERR_CUDA;
  }
  if (id == 0) id = pd::current_ctx_id(*f);
  if (id != 0 && g_cached < kMaxContexts) g_cache[g_cached++] = Entry{id, p};
  *out = p;
  return PD_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Everything the calls below would refuse, checked before anything is queued.
pd_status check_args(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, const int32_t* seq_lens, int32_t window, float scale,
                     const void* out) {
  if (!pd::plan_is_valid(plan) || plan->partial) return PD_ERR_INVALID_ARG;
  const pd_layer_desc& ly = plan->layer;
  if (ly.kv_dtype != PD_KV_BF16) return PD_ERR_INVALID_ARG;  // FP8 caches need scales: not served here
  if (window != ly.window || !std::isfinite(scale)) return PD_ERR_INVALID_ARG;
  if (plan->workspace_bytes > kScratchBytes) return PD_ERR_WORKSPACE_TOO_SMALL;
  if (plan->batch == 0) return PD_OK;
  if (!q || !k_pool || !block_tables || !seq_lens || !out) return PD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
      !aligned(seq_lens, 4))
    return PD_ERR_INVALID_ARG;
  if (ly.kv_shared) {
    if (v_pool && v_pool != k_pool) return PD_ERR_INVALID_ARG;
  } else if (!v_pool || v_pool == k_pool || !aligned(v_pool, 16)) {
    return PD_ERR_INVALID_ARG;
  }
  return PD_OK;
}

}  // namespace

extern "C" pd_status paged_decode_noalloc(const pd_plan* plan, const void* q, const void* k_pool,
                                          const void* v_pool, const int32_t* block_tables, const int32_t* seq_lens,
                                          int32_t window, float scale, void* out, uint32_t* device_flags,
                                          void* stream) {
  pd_status st = check_args(plan, q, k_pool, v_pool, block_tables, seq_lens, window, scale, out);
  if (st != PD_OK || plan->batch == 0) return st;
  if (device_flags && !aligned(device_flags, 4)) return PD_ERR_INVALID_ARG;
  void* scratch = nullptr;
  st = scratch_for_current_context(&scratch);
  if (st != PD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the error word starts at zero
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s) != cudaSuccess) return PD_ERR_CUDA;
  st = window > 0 ? paged_decode_window(plan, q, k_pool, v_pool, block_tables, seq_lens, window, scale, scratch,
                                        kScratchBytes, out, stream)
                  : paged_decode_global(plan, q, k_pool, v_pool, block_tables, seq_lens, scale, scratch,
                                        kScratchBytes, out, stream);
  if (st != PD_OK) return st;
  st = paged_decode_merge(plan, scratch, kScratchBytes, out, stream);
  if (st != PD_OK) return st;
  if (device_flags &&
      cudaMemcpyAsync(device_flags, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return PD_ERR_CUDA;
  return PD_OK;
}
