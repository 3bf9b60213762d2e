// Stage 2 of paged GQA decode attention (sm_103a): merge the KV pieces of every
// (request, query head) by their log-sum-exp weights, as its own launch (used
// when the pieces of one (request, KV head) are too many to merge in stage 1).
//
// Method: vLLM concepts page "模型库与算子层 — 概念", section "MLA 与 Sparse MLA
// （DSA）" — split-KV decode whose pieces each produce partial results carrying a
// log-sum-exp, combined afterwards:
//   M = max_s lse_s,  w_s = exp(lse_s - M) / sum_s' exp(lse_s' - M),  out = sum_s w_s o_s.
// Empty pieces carry lse = -inf (weight 0; their rows are not read); a row with
// no piece at all is zero, with lse -inf. The same kernel merges a stage-1
// workspace ([rows][S] pieces) and partial results gathered from several ranks
// ([S][rows]), to bf16, or to fp32 with the merged log-sum-exp.
//
// Grid (row, 128-dim slice of the row), 128 threads, launched behind stage 1
// as a programmatic dependent (it waits for stage 1 before reading). Every
// warp reduces the row's S log-sum-exps itself; then lane 4c + g of warp w
// sums float4 column 8w + c of the slice over pieces g, g + 4, g + 8, ...
// (eight lanes of one piece group read 128 contiguous bytes of a piece; a
// lane's first four pieces' rows are loaded together with the log-sum-exps,
// before the weights are known), and two shuffles add the four groups. The kernel holds no shared memory, so one of its CTAs fits
// beside a stage-1 CTA of the next launch on the same SM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pd_common.cuh"
#include "pd_kernels.h"

namespace pd {

namespace {

constexpr int kMergeMaxSplits = 1024;  // pieces of one row (the plan's cap, and the combine's rank limit)
constexpr int kMergeThreads = 128;  // 32 float4 columns x 4 piece groups: 128 dims a CTA
constexpr int kMergeGroups = 4;
constexpr int kPrefetch = 4;  // pieces per lane whose rows load with the log-sum-exps (S <= 16 in one go)

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  grid_dependency_wait();  // stage 1 (launched before this grid) has finished
  // the next kernel on the stream may become resident now (it waits for this
  // grid before it reads anything this grid writes)
  grid_launch_dependents();
  const size_t row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = p.num_splits;
  const float* lse = p.lse_part + row * p.lse_row_stride;
  const int g = lane % kMergeGroups;
  const int d4 = blockIdx.y * (kMergeThreads / kMergeGroups) + warp * (32 / kMergeGroups) + lane / kMergeGroups;
  const bool active = d4 < p.head_dim / 4;
  const float* src = p.o_part + row * p.row_stride + (size_t)d4 * 4;
  // the rows of this lane's first kPrefetch pieces do not depend on the
  // weights: their loads go out with the log-sum-exps'
  float4 pre[kPrefetch];
#pragma unroll
  for (int i = 0; i < kPrefetch; ++i) {
    const int s = g + i * kMergeGroups;
    pre[i] = (active && s < S) ? *reinterpret_cast<const float4*>(src + (size_t)s * p.piece_stride)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lse[s * p.lse_piece_stride]);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  float sum = 0.f;
  constexpr float kLog2e = 1.4426950408889634f;
  if (M != -INFINITY)
    for (int s = lane; s < S; s += 32) sum += exp2f((lse[s * p.lse_piece_stride] - M) * kLog2e);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  if (p.out_lse && blockIdx.y == 0 && threadIdx.x == 0) p.out_lse[row] = sum > 0.f ? M + __logf(sum) : -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (active && M != -INFINITY) {
    // an empty piece weighs 0 and its row may never have been written:
    // selected out, not multiplied
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) {
      const int s = g + i * kMergeGroups;
      if (s >= S) break;
      const float ws = exp2f((lse[s * p.lse_piece_stride] - M) * kLog2e) * inv;
      const bool use = ws != 0.f;
      acc.x = use ? fmaf(ws, pre[i].x, acc.x) : acc.x;
      acc.y = use ? fmaf(ws, pre[i].y, acc.y) : acc.y;
      acc.z = use ? fmaf(ws, pre[i].z, acc.z) : acc.z;
      acc.w = use ? fmaf(ws, pre[i].w, acc.w) : acc.w;
    }
#pragma unroll 4
    for (int s = g + kPrefetch * kMergeGroups; s < S; s += kMergeGroups) {
      const float ws = exp2f((lse[s * p.lse_piece_stride] - M) * kLog2e) * inv;
      if (ws == 0.f) continue;
      const float4 o = *reinterpret_cast<const float4*>(src + (size_t)s * p.piece_stride);
      acc.x = fmaf(ws, o.x, acc.x);
      acc.y = fmaf(ws, o.y, acc.y);
      acc.z = fmaf(ws, o.z, acc.z);
      acc.w = fmaf(ws, o.w, acc.w);
    }
  }
  // the four piece groups of a column sit in four neighbouring lanes
#pragma unroll
  for (int m = 1; m < kMergeGroups; m <<= 1) {
    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, m);
    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, m);
    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, m);
    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, m);
  }
  if (!active || g != 0) return;
  if (p.out) {
    __nv_bfloat162* out =
        reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(p.out) + row * p.head_dim) + d4 * 2;
    out[0] = __floats2bfloat162_rn(acc.x, acc.y);
    out[1] = __floats2bfloat162_rn(acc.z, acc.w);
  }
  if (p.out_f32) reinterpret_cast<float4*>(p.out_f32 + row * p.head_dim)[d4] = acc;
}

}  // namespace

int launch_merge(const MergeParams& p, int rows, void* stream) {
  if (rows <= 0) return 0;
  if (p.num_splits > kMergeMaxSplits || p.head_dim % 4 != 0) return static_cast<int>(cudaErrorInvalidValue);
  // launched with programmatic stream serialisation: its CTAs may become
  // resident while stage 1 drains and wait there for its completion
  cudaLaunchConfig_t cfg = {};
  constexpr int kCols = kMergeThreads / kMergeGroups;  // float4 columns a CTA
  cfg.gridDim = dim3(rows, (p.head_dim / 4 + kCols - 1) / kCols);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, merge_kernel, p);
  if (e != cudaSuccess) (void)cudaGetLastError();
  return static_cast<int>(e);
}

}  // namespace pd
