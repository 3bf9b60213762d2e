// Stage 2 of paged GQA decode attention (sm_103a): merge the KV pieces of every
// (request, query head) by their log-sum-exp weights.
//
// Method: vLLM concepts page "模型库与算子层 — 概念", section "MLA 与 Sparse MLA
// （DSA）" — split-KV decode whose pieces each produce partial results carrying a
// log-sum-exp, combined afterwards:
//   M = max_s lse_s,  w_s = exp(lse_s - M),  out = sum_s w_s o_s / sum_s w_s.
// Pieces with no attended token (lse = -inf) are skipped, so their partial rows
// are never read; a row with no piece at all is zero.
//
// One CTA per (request, query head) row; each thread owns 4 consecutive dims
// (one 16-byte fp32 load per piece); the output row is written as bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pd_kernels.h"

namespace pd {

namespace {

__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  const size_t row = blockIdx.x;
  const int S = p.num_splits;
  const int D = p.head_dim;
  const float* lse = p.lse_part + row * S;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, lse[s]);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + row * D;
  for (int d4 = threadIdx.x * 4; d4 < D; d4 += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const float l = lse[s];
        if (l == -INFINITY) continue;
        const float w = expf(l - M);
        const float4 o = *reinterpret_cast<const float4*>(p.o_part + (row * S + s) * D + d4);
        wsum += w;
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    reinterpret_cast<__nv_bfloat162*>(out + d4)[0] = lo;
    reinterpret_cast<__nv_bfloat162*>(out + d4)[1] = hi;
  }
}

}  // namespace

int launch_merge(const MergeParams& p, int rows, void* stream) {
  if (rows <= 0) return 0;
  const int threads = p.head_dim / 4 < 128 ? p.head_dim / 4 : 128;
  merge_kernel<<<rows, threads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace pd
