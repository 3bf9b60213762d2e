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
// that loads this library holds it until the process exits. Its device address
// is looked up once per device (cudaGetSymbolAddress, on the first call made
// while that device is current); that first call should therefore happen before
// any stream capture. All calls share the one array: calls that overlap on the
// GPU (two streams, or two host threads) race on it, so order them on one
// stream. Nothing here allocates: no cudaMalloc, no cudaFree, no library call
// that allocates.
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "paged_decode.h"

namespace {

constexpr size_t kScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

// Partials, log-sum-exps and the device error word of the calls below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
pd_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return PD_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PD_OK;
}

}  // namespace

extern "C" pd_status paged_decode_noalloc(const pd_plan* plan, const void* q, const void* k_pool,
                                          const void* v_pool, const int32_t* block_tables, const int32_t* seq_lens,
                                          int32_t window, float scale, void* out, uint32_t* device_flags,
                                          void* stream) {
  if (!plan) return PD_ERR_INVALID_ARG;
  if (plan->workspace_bytes > kScratchBytes) return PD_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  pd_status st = scratch_for_current_device(&scratch);
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
