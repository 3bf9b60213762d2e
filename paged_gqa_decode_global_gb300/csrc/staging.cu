// Copies for a decode loop whose inputs come from, and whose results go to,
// page-locked host memory, as one kernel in the stream's chain of programmatic
// dependent launches.
//
// Not an operation of the decode method itself: plumbing for the caller's
// loop. A decode step issued as memcpy + kernels + memcpy, or with its copies
// on other streams joined by event waits, ends that chain at every copy (a
// launch that follows a memcpy or an event wait cannot start before it
// completes), so the next step's stage 1 can no longer become resident and
// stream its older KV rows while the step in front drains. Here each copy is a
// kernel that lets the launch behind it start at once.
//
// Order: with after_wait = 0 the copies run, then the kernel waits for the
// launch in front of it (griddepcontrol.wait), so it completes only after that
// launch -- the chain's order of completions is kept, and a launch behind it
// that waits sees everything in front complete. With after_wait = 1 it waits
// first (for a result the launch in front writes).

#include <cuda_runtime.h>

#include <cstdint>

#include "paged_decode.h"

namespace pd {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;       // 16-byte loads a thread has in flight
constexpr int kMaxCopyBlocks = 1024;

__device__ __forceinline__ void copy_span(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  const size_t stride = (size_t)gridDim.x * kCopyThreads;
  size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x;
  // every load of a round issued before its stores: host memory is a long round trip away
  for (; i + (kCopyUnroll - 1) * stride < n; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

struct CopyList {
  const uint4* src[PD_MAX_STAGE_COPIES];
  uint4* dst[PD_MAX_STAGE_COPIES];
  size_t n[PD_MAX_STAGE_COPIES];  // 16-byte units; 0 for an unused slot
};

__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(const CopyList list, int after_wait) {
  asm volatile("griddepcontrol.launch_dependents;");
  if (after_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
  for (int c = 0; c < PD_MAX_STAGE_COPIES; ++c) copy_span(list.src[c], list.dst[c], list.n[c]);
  if (!after_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The address a kernel on the current device reaches `p` by: itself for
// device (or managed) memory of that device, the mapped device address for
// page-locked host memory; nullptr for pageable host memory, memory of another
// device, or a pointer the runtime does not know.
const void* device_address(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  switch (a.type) {
    case cudaMemoryTypeHost:
      return a.devicePointer;
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return a.device == dev ? a.devicePointer : nullptr;
    default:
      return nullptr;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, const void* b, size_t n) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + n && y < x + n;
}

}  // namespace
}  // namespace pd

extern "C" pd_status paged_decode_stage_copy(const pd_copy* copies, int32_t num_copies, int32_t after_wait,
                                             void* stream) {
  using namespace pd;
  if (after_wait != 0 && after_wait != 1) return PD_ERR_INVALID_ARG;
  if (num_copies < 0 || num_copies > PD_MAX_STAGE_COPIES || (num_copies > 0 && !copies)) return PD_ERR_INVALID_ARG;
  // every check that needs no CUDA call first, over the whole list
  for (int c = 0; c < num_copies; ++c) {
    const pd_copy& cp = copies[c];
    if (cp.bytes == 0) continue;
    if (cp.bytes & 15u) return PD_ERR_INVALID_ARG;
    if (!cp.dst || !cp.src || !aligned16(cp.dst) || !aligned16(cp.src)) return PD_ERR_INVALID_ARG;
    if (overlap(cp.dst, cp.src, cp.bytes)) return PD_ERR_INVALID_ARG;
  }
  CopyList list{};
  size_t longest = 0;
  for (int c = 0; c < num_copies; ++c) {
    const pd_copy& cp = copies[c];
    if (cp.bytes == 0) continue;
    const void* s = device_address(cp.src);
    const void* d = device_address(cp.dst);
    if (!s || !d || !aligned16(s) || !aligned16(d)) return PD_ERR_INVALID_ARG;
    list.src[c] = static_cast<const uint4*>(s);
    list.dst[c] = static_cast<uint4*>(const_cast<void*>(d));
    list.n[c] = cp.bytes / 16;
    if (list.n[c] > longest) longest = list.n[c];
  }
  size_t blocks = (longest + kCopyThreads - 1) / kCopyThreads;
  if (blocks > (size_t)kMaxCopyBlocks) blocks = kMaxCopyBlocks;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, stage_copy_kernel, list, (int)after_wait);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PD_ERR_CUDA;
  }
  return PD_OK;
}
