// The step before decode attention (sm_103a): per-head RMS norm of the new
// token's q, k and v, RoPE of q and k at the token's position, and the write of
// its k / v rows into the paged cache, in one launch.
//
// Method (Sparse-vLLM PR #27 "feat: support Gemma 4 and native multimodal
// inference", section "专用算子与性能优化": QKV norm + RoPE for Gemma 4; section
// "Gemma 4 文本推理": sliding-window and global layers carry their own RoPE
// parameters and RoPE cache; vLLM concepts page "模型库与算子层 — 概念": norm /
// RoPE folded into the paged KV-cache write).
//
// GB300 design: the work is B * (Hq + 2 Hkv) head rows of d <= 512 bf16, a few
// hundred KB per layer-step, so the launch is latency-bound: one warp per head
// row, 4 rows per CTA, every row read and written once with 16-byte accesses;
// the mean square is a warp reduction; a RoPE pair (i, i + rot/2) lies in
// different lanes, so the normalised row goes through shared memory once.
#include <cuda_bf16.h>

#include <cmath>

#include "paged_decode.h"
#include "pd_common.cuh"
#include "pd_variants.h"

namespace pd {
namespace {

constexpr int kRowsPerCta = 4;

struct PrepParams {
  const uint16_t* q_in;
  const uint16_t* k_in;
  const uint16_t* v_in;
  const uint16_t* q_w;
  const uint16_t* k_w;
  const uint16_t* v_w;  // may be null: unit weight
  const float* cos_sin;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  uint16_t* q_out;
  uint16_t* k_pool;
  uint16_t* v_pool;
  uint32_t* flags;
  float eps;
  int rot;
  int num_positions;
  int num_q_heads, num_kv_heads;
  int page_size, num_pages, max_pages;
  int rows;  // Hq + Hkv (+ Hkv when K != V)
};

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Lane l holds dims c*256 + 8l .. c*256 + 8l + 7 of chunk c.
template <int D>
__global__ void __launch_bounds__(32 * kRowsPerCta) qkv_norm_rope_write_kernel(const PrepParams p) {
  constexpr int NCH = D / 256;
  __shared__ float ybuf[kRowsPerCta][D];
  // launched as a programmatic dependent: let the decode behind this one
  // launch at once (it waits for this grid, and so for everything before it,
  // before it reads q or a new row; with early_kv its older rows stream in
  // meanwhile), then wait for the kernel before this one, which may have
  // written the new rows
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * kRowsPerCta + warp;
  if (r >= p.rows) return;

  // The source row and its weight do not depend on the length: their loads
  // go out first, the length and the page id (which place the result) in
  // their shadow.
  const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const bool is_q = r < Hq, is_k = !is_q && r < Hq + Hkv;
  const int head = is_q ? r : (is_k ? r - Hq : r - Hq - Hkv);
  const uint16_t* src = is_q ? p.q_in + ((size_t)b * Hq + head) * D
                             : (is_k ? p.k_in : p.v_in) + ((size_t)b * Hkv + head) * D;
  const uint16_t* w = is_q ? p.q_w : (is_k ? p.k_w : p.v_w);
  float x[NCH][8], wf[NCH][8];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    unpack8(__ldg(reinterpret_cast<const uint4*>(src + c * 256 + lane * 8)), x[c]);
    if (w) {
      unpack8(__ldg(reinterpret_cast<const uint4*>(w + c * 256 + lane * 8)), wf[c]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) wf[c][i] = 1.f;
    }
  }

  const int L = p.seq_lens[b];
  const long long cap = (long long)p.max_pages * p.page_size;
  if (L < 1 || L > cap || (p.rot > 0 && L - 1 >= p.num_positions)) {
    if (r == 0 && lane == 0) atomicOr(p.flags, kErrBadSeqLen);
    return;
  }
  const int pos = L - 1;
  uint16_t* dst;
  if (is_q) {
    dst = p.q_out + ((size_t)b * Hq + head) * D;
  } else {
    const int page = p.block_tables[(size_t)b * p.max_pages + pos / p.page_size];
    if ((unsigned)page >= (unsigned)p.num_pages) {
      if (lane == 0) atomicOr(p.flags, kErrBadPage);
      return;
    }
    dst = (is_k ? p.k_pool : p.v_pool) + (((size_t)page * Hkv + head) * p.page_size + pos % p.page_size) * D;
  }
  const bool rotate = is_q || is_k;  // v is not rotated

  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(x[c][i], x[c][i], ss);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(kFullMask, ss, m);
  const float inv_rms = 1.f / sqrtf(ss / D + p.eps);
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) x[c][i] = x[c][i] * inv_rms * wf[c][i];

  if (rotate && p.rot > 0) {
    float* y = ybuf[warp];
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i) y[c * 256 + lane * 8 + i] = x[c][i];
    __syncwarp();
    const int half = p.rot >> 1;
    const float* cs = p.cos_sin + (size_t)pos * p.rot;
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int dim = c * 256 + lane * 8 + i;
        if (dim < half) {
          x[c][i] = y[dim] * __ldg(cs + dim) - y[dim + half] * __ldg(cs + half + dim);
        } else if (dim < p.rot) {
          const int j = dim - half;
          x[c][i] = y[dim] * __ldg(cs + j) + y[j] * __ldg(cs + half + j);
        }
      }
  }

#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    uint4 o;
    o.x = pack2(x[c][0], x[c][1]);
    o.y = pack2(x[c][2], x[c][3]);
    o.z = pack2(x[c][4], x[c][5]);
    o.w = pack2(x[c][6], x[c][7]);
    *reinterpret_cast<uint4*>(dst + c * 256 + lane * 8) = o;
  }
}

// One thread per (position, pair); fp64 angle and sine / cosine, rounded to fp32.
__global__ void rope_table_kernel(double theta, int rot, int num_positions, float* out) {
  const int half = rot / 2;
  const long long n = (long long)num_positions * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(e / half), i = (int)(e % half);
    const double a = (double)pos * pow(theta, -2.0 * i / rot);
    double s, c;
    sincos(a, &s, &c);
    out[(size_t)pos * rot + i] = (float)c;
    out[(size_t)pos * rot + half + i] = (float)s;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pd

extern "C" {

pd_status paged_decode_rope_table(double theta, int32_t rotary_dim, int32_t num_positions, float* cos_sin,
                                  void* stream) {
  if (!(theta > 0.0) || !std::isfinite(theta) || rotary_dim < 2 || rotary_dim > 512 || rotary_dim % 2 ||
      num_positions < 1 || !cos_sin)
    return PD_ERR_INVALID_ARG;
  const long long n = (long long)num_positions * (rotary_dim / 2);
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const int blocks = (int)(want < 65536 ? want : 65536);
  pd::rope_table_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(theta, rotary_dim, num_positions,
                                                                                   cos_sin);
  return cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

pd_status paged_decode_qkv_norm_rope_write(const pd_layer_desc* layer, int32_t batch, int32_t rotary_dim,
                                           int32_t num_positions, float eps, const void* q_in, const void* k_in,
                                           const void* v_in, const void* q_norm_weight, const void* k_norm_weight,
                                           const void* v_norm_weight, const float* cos_sin,
                                           const int32_t* block_tables, const int32_t* seq_lens, void* q_out,
                                           void* k_pool, void* v_pool, uint32_t* device_flags, void* stream) {
  if (!layer) return PD_ERR_INVALID_ARG;
  const pd_layer_desc& ly = *layer;
  if (ly.num_q_heads <= 0 || ly.num_kv_heads <= 0 || ly.num_q_heads % ly.num_kv_heads != 0)
    return PD_ERR_INVALID_ARG;
  if (ly.page_size <= 0 || ly.num_pages <= 0 || ly.max_pages_per_seq <= 0) return PD_ERR_INVALID_ARG;
  if (ly.kv_shared != 0 && ly.kv_shared != 1) return PD_ERR_INVALID_ARG;
  if (ly.kv_dtype != PD_KV_BF16) return ly.kv_dtype == PD_KV_FP8_E4M3 ? PD_ERR_UNSUPPORTED : PD_ERR_INVALID_ARG;
  if (ly.head_dim != 256 && ly.head_dim != 512) return PD_ERR_UNSUPPORTED;
  if (batch < 0 || rotary_dim < 0 || rotary_dim % 2 || rotary_dim > ly.head_dim) return PD_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return PD_ERR_INVALID_ARG;
  if (rotary_dim > 0 && (!cos_sin || num_positions < 1)) return PD_ERR_INVALID_ARG;
  const bool kvs = ly.kv_shared != 0;
  if (!q_in || !k_in || !q_norm_weight || !k_norm_weight || !block_tables || !seq_lens || !q_out || !k_pool ||
      !device_flags)
    return PD_ERR_INVALID_ARG;
  if (!kvs && (!v_in || !v_pool)) return PD_ERR_INVALID_ARG;
  for (const void* ptr : {q_in, k_in, q_norm_weight, k_norm_weight, (const void*)q_out, (const void*)k_pool})
    if (!pd::aligned16(ptr)) return PD_ERR_INVALID_ARG;
  if (!kvs && (!pd::aligned16(v_in) || !pd::aligned16(v_pool))) return PD_ERR_INVALID_ARG;
  if (v_norm_weight && !pd::aligned16(v_norm_weight)) return PD_ERR_INVALID_ARG;
  if (batch == 0) return PD_OK;

  pd::PrepParams p;
  p.q_in = static_cast<const uint16_t*>(q_in);
  p.k_in = static_cast<const uint16_t*>(k_in);
  p.v_in = kvs ? nullptr : static_cast<const uint16_t*>(v_in);
  p.q_w = static_cast<const uint16_t*>(q_norm_weight);
  p.k_w = static_cast<const uint16_t*>(k_norm_weight);
  p.v_w = static_cast<const uint16_t*>(v_norm_weight);
  p.cos_sin = cos_sin;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.q_out = static_cast<uint16_t*>(q_out);
  p.k_pool = static_cast<uint16_t*>(k_pool);
  p.v_pool = kvs ? nullptr : static_cast<uint16_t*>(v_pool);
  p.flags = device_flags;
  p.eps = eps;
  p.rot = rotary_dim;
  p.num_positions = num_positions;
  p.num_q_heads = ly.num_q_heads;
  p.num_kv_heads = ly.num_kv_heads;
  p.page_size = ly.page_size;
  p.num_pages = ly.num_pages;
  p.max_pages = ly.max_pages_per_seq;
  p.rows = ly.num_q_heads + ly.num_kv_heads * (kvs ? 1 : 2);
  const dim3 grid((unsigned)batch, (unsigned)((p.rows + pd::kRowsPerCta - 1) / pd::kRowsPerCta));
  if (grid.y > 65535) return PD_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * pd::kRowsPerCta);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = ly.head_dim == 512 ? cudaLaunchKernelEx(&cfg, pd::qkv_norm_rope_write_kernel<512>, p)
                                           : cudaLaunchKernelEx(&cfg, pd::qkv_norm_rope_write_kernel<256>, p);
  if (e != cudaSuccess) (void)cudaGetLastError();
  return e == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

}  // extern "C"
