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
// Order: with after_wait = 0 both copies run, then the kernel waits for the
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

__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(const uint4* a_src, uint4* a_dst, size_t n_a,
                                                                  const uint4* b_src, uint4* b_dst, size_t n_b,
                                                                  int after_wait) {
  asm volatile("griddepcontrol.launch_dependents;");
  if (after_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
  copy_span(a_src, a_dst, n_a);
  copy_span(b_src, b_dst, n_b);
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

extern "C" pd_status paged_decode_stage_copy(void* in_dst, const void* in_src, size_t in_bytes, void* out_dst,
                                             const void* out_src, size_t out_bytes, int32_t after_wait,
                                             void* stream) {
  using namespace pd;
  if (after_wait != 0 && after_wait != 1) return PD_ERR_INVALID_ARG;
  if ((in_bytes | out_bytes) & 15u) return PD_ERR_INVALID_ARG;
  const void* ends[2][2] = {{in_src, in_dst}, {out_src, out_dst}};
  const size_t bytes[2] = {in_bytes, out_bytes};
  const void* dev[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};
  for (int c = 0; c < 2; ++c) {
    if (bytes[c] == 0) continue;
    for (int e = 0; e < 2; ++e) {
      if (!ends[c][e] || !aligned16(ends[c][e])) return PD_ERR_INVALID_ARG;
      dev[c][e] = device_address(ends[c][e]);
      if (!dev[c][e] || !aligned16(dev[c][e])) return PD_ERR_INVALID_ARG;
    }
    if (overlap(ends[c][0], ends[c][1], bytes[c])) return PD_ERR_INVALID_ARG;
  }
  const size_t n = (in_bytes > out_bytes ? in_bytes : out_bytes) / 16;
  size_t blocks = (n + kCopyThreads - 1) / kCopyThreads;
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
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, stage_copy_kernel, static_cast<const uint4*>(dev[0][0]),
                         static_cast<uint4*>(const_cast<void*>(dev[0][1])), in_bytes / 16,
                         static_cast<const uint4*>(dev[1][0]), static_cast<uint4*>(const_cast<void*>(dev[1][1])),
                         out_bytes / 16, (int)after_wait);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PD_ERR_CUDA;
  }
  return PD_OK;
}
