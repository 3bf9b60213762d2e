// Stage 1 of paged GQA decode attention (sm_103a): one CTA per
// (KV piece, KV head, request) streams the piece's K/V rows once from HBM and
// serves every query head of that KV head.
//
// Method (Sparse-vLLM PR #27 "feat: support Gemma 4 and native multimodal
// inference", section "专用算子与性能优化": a stage-1 decode pass whose program
// handles the GQA query heads of one KV head together, and grouped
// sliding-window/global decode; vLLM concepts page "模型库与算子层 — 概念",
// section "MLA 与 Sparse MLA（DSA）": split-KV pieces that each produce a partial
// result plus its log-sum-exp).
//
// GB300 design:
//   * warp NW (one elected lane) is the producer: per block of TB tokens it
//     issues one 1-D bulk TMA copy of the contiguous (page, KV head) rows of K
//     (and one of V) into a ring stage, completion counted on an mbarrier;
//   * consumer warp w owns ring stages w, w+NW, ... and processes blocks
//     w, w+NW, ... of the piece with its own online-softmax state, so warps
//     never wait on one another inside the loop;
//   * lanes split head_dim (16-byte chunks, conflict-free shared loads); q of
//     all G heads and the fp32 accumulators of all G heads stay in registers;
//   * QK: each lane forms TB*G partial dot products, one recursive-halving
//     reduce-scatter over the 32 lanes leaves one full dot product per lane;
//   * softmax in base 2 with q pre-scaled by scale*log2(e); PV broadcasts each
//     probability from the lane that owns it;
//   * at the end the NW warp states are merged in shared memory and the CTA
//     writes bf16 output (one piece) or an fp32 partial + log-sum-exp.
#include <cuda_bf16.h>

#include "pd_common.cuh"
#include "pd_kernels.h"

namespace pd {

namespace {

// Sum NV values per lane across the warp; afterwards lane l holds, in v[0], the
// full sum of value index l / (32 / NV). Recursive halving: at each level a lane
// keeps the half of its values selected by its lane bit and adds the partner's.
template <int NV>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lane) {
#pragma unroll
  for (int half = NV / 2, mask = 16; half >= 1; half >>= 1, mask >>= 1) {
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(kFullMask, send, mask);
    }
  }
  // remaining lane bits: plain butterfly so every replica holds the sum
#pragma unroll
  for (int mask = 16 / NV; mask >= 1; mask >>= 1) v[0] += __shfl_xor_sync(kFullMask, v[0], mask);
}

}  // namespace

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) stage1_kernel(const Stage1Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFFSET);
  uint64_t* empty_bar = full_bar + C::NST;
  uint32_t* stage_valid = reinterpret_cast<uint32_t*>(smem + C::VALID_OFFSET);
  float2* warp_ml = reinterpret_cast<float2*>(smem + C::ML_OFFSET);

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- attended range of this request and this piece -------------------------
  const int cap = p.max_pages * p.page_size;
  int L = p.seq_lens[b];
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadSeqLen);
    L = L < 0 ? 0 : cap;
  }
  const int lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
  const int base = (lo / C::TB) * C::TB;
  const long long piece_lo = (long long)base + (long long)split * p.chunk_tokens;
  const int tlo = (int)(piece_lo > lo ? piece_lo : lo);
  // the last piece takes whatever remains, so a device length longer than the
  // planned one is still attended in full
  const long long piece_hi = (split == p.num_splits - 1) ? (long long)L : piece_lo + p.chunk_tokens;
  const int thi = (int)(piece_hi < L ? piece_hi : L);
  const int blk_lo = (tlo / C::TB) * C::TB;
  const int nblk = (thi > tlo) ? (thi - blk_lo + C::TB - 1) / C::TB : 0;

  const size_t row_hq = (size_t)b * p.num_q_heads + (size_t)g * C::G;  // first query head row

  if (nblk == 0) {
    // nothing attended in this piece
    if (p.num_splits == 1) {
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + row_hq * C::D;
      for (int i = threadIdx.x; i < C::G * C::D; i += C::THREADS) o[i] = __float2bfloat16_rn(0.f);
    } else if (threadIdx.x < C::G) {
      p.lse_part[(row_hq + threadIdx.x) * p.num_splits + split] = -INFINITY;
    }
    return;
  }

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // ---- producer ------------------------------------------------------------------
  if (warp == C::NW) {
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      const int32_t* table = p.block_tables + (size_t)b * p.max_pages;
      int issued = 0;
#pragma unroll 1
      for (int j = 0; j < nblk; ++j) {
        const int st = j % C::NST;
        const int round = j / C::NST;
        if (round > 0 && !mbar_wait(&empty_bar[st], (round - 1) & 1)) {
          atomicOr(p.err, kErrTimeout);
          break;
        }
        const int t0 = blk_lo + j * C::TB;
        const int page = table[t0 / p.page_size];
        const bool ok = (unsigned)page < (unsigned)p.num_pages;
        stage_valid[st] = ok ? 1u : 0u;
        if (ok) {
          const size_t row = ((size_t)page * p.num_kv_heads + g) * p.page_size + (t0 % p.page_size);
          uint8_t* dst = smem + (size_t)st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[st], C::STAGE_BYTES);
          bulk_g2s(dst, p.k_pool + row * C::D, C::KV_BYTES, &full_bar[st], policy);
          if (!C::KVS) bulk_g2s(dst + C::KV_BYTES, p.v_pool + row * C::D, C::KV_BYTES, &full_bar[st], policy);
        } else {
          atomicOr(p.err, kErrBadPage);
          mbar_arrive(&full_bar[st]);
        }
        issued = j + 1;
      }
      // no copy may still be landing in shared memory when the CTA exits
#pragma unroll 1
      for (int st = 0; st < C::NST && st < issued; ++st) {
        const int j_last = st + C::NST * ((issued - 1 - st) / C::NST);
        if (!mbar_wait(&full_bar[st], (j_last / C::NST) & 1)) atomicOr(p.err, kErrTimeout);
      }
    }
    return;
  }

  // ---- consumers -----------------------------------------------------------------
  // q of the G heads for this lane's dims, pre-scaled to base-2 logits
  float qf[C::G][C::DPL];
#pragma unroll
  for (int h = 0; h < C::G; ++h) {
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.q + (row_hq + h) * C::D) + c * 32 + lane);
      float f[8];
      unpack_bf16x8(w, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) qf[h][c * 8 + i] = f[i] * p.scale_log2;
    }
  }

  float acc[C::G][C::DPL];
#pragma unroll
  for (int h = 0; h < C::G; ++h)
#pragma unroll
    for (int i = 0; i < C::DPL; ++i) acc[h][i] = 0.f;

  // this lane's value after the reduce-scatter: token vi / G, head vi % G
  const int vi = lane / C::R;
  const int my_tb = vi / C::G;
  float m_run = -INFINITY;  // running max (base-2 logits) of head vi % G
  float l_run = 0.f;        // running sum of 2^(s - m_run)

#pragma unroll 1
  for (int j = warp; j < nblk; j += C::NW) {
    const int st = j % C::NST;
    // every lane polls; the warp leaves together if any lane gave up
    const bool landed = mbar_wait(&full_bar[st], (j / C::NST) & 1);
    if (__any_sync(kFullMask, !landed)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      break;
    }
    const uint8_t* kst = smem + (size_t)st * C::STAGE_BYTES;
    const uint8_t* vst = C::KVS ? kst : kst + C::KV_BYTES;
    const bool stage_ok = stage_valid[st] != 0;
    const int t0 = blk_lo + j * C::TB;

    // QK: partial dot products over this lane's dims
    float part[C::NV];
#pragma unroll
    for (int tb = 0; tb < C::TB; ++tb) {
      float kf[C::DPL];
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        const uint4 w = lds128(kst + tb * C::ROW_BYTES + (c * 32 + lane) * 16);
        float f[8];
        unpack_bf16x8(w, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) kf[c * 8 + i] = f[i];
      }
#pragma unroll
      for (int h = 0; h < C::G; ++h) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < C::DPL; i += 2) {
          s0 = fmaf(qf[h][i], kf[i], s0);
          s1 = fmaf(qf[h][i + 1], kf[i + 1], s1);
        }
        part[tb * C::G + h] = s0 + s1;
      }
    }
    reduce_scatter<C::NV>(part, lane);

    // online softmax over the block, per head
    const int t = t0 + my_tb;
    const bool valid = stage_ok && t >= tlo && t < thi;
    const float s = valid ? part[0] : -INFINITY;
    float bmax = s;
#pragma unroll
    for (int mask = C::R * C::G; mask < 32; mask <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(kFullMask, bmax, mask));
    const float m_new = fmaxf(m_run, bmax);
    const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_run - m_new);
    const float pr = valid ? ex2(s - m_new) : 0.f;
    float bsum = pr;
#pragma unroll
    for (int mask = C::R * C::G; mask < 32; mask <<= 1) bsum += __shfl_xor_sync(kFullMask, bsum, mask);
    l_run = l_run * alpha + bsum;
    m_run = m_new;

    if (__any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll
      for (int h = 0; h < C::G; ++h) {
        const float a = __shfl_sync(kFullMask, alpha, h * C::R);
#pragma unroll
        for (int i = 0; i < C::DPL; ++i) acc[h][i] *= a;
      }
    }

    // PV (kept rolled: the block's rows are consumed one at a time)
#pragma unroll 1
    for (int tb = 0; tb < C::TB; ++tb) {
      float vf[C::DPL];
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        const uint4 w = lds128(vst + tb * C::ROW_BYTES + (c * 32 + lane) * 16);
        float f[8];
        unpack_bf16x8(w, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) vf[c * 8 + i] = f[i];
      }
#pragma unroll
      for (int h = 0; h < C::G; ++h) {
        const float ph = __shfl_sync(kFullMask, pr, (tb * C::G + h) * C::R);
#pragma unroll
        for (int i = 0; i < C::DPL; ++i) acc[h][i] = fmaf(ph, vf[i], acc[h][i]);
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
  }

  // ---- merge the NW warp states --------------------------------------------------
  named_bar_sync(1, C::NW * 32);  // every consumer is done with the ring
  float* comb = reinterpret_cast<float*>(smem);  // [NW][G][D]
#pragma unroll
  for (int h = 0; h < C::G; ++h) {
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      float4* dst = reinterpret_cast<float4*>(comb + ((size_t)warp * C::G + h) * C::D + (c * 32 + lane) * 8);
      dst[0] = make_float4(acc[h][c * 8 + 0], acc[h][c * 8 + 1], acc[h][c * 8 + 2], acc[h][c * 8 + 3]);
      dst[1] = make_float4(acc[h][c * 8 + 4], acc[h][c * 8 + 5], acc[h][c * 8 + 6], acc[h][c * 8 + 7]);
    }
  }
  if (my_tb == 0 && (lane % C::R) == 0) warp_ml[warp * C::G + vi] = make_float2(m_run, l_run);
  named_bar_sync(1, C::NW * 32);

  const int tid = threadIdx.x;
#pragma unroll 1
  for (int e = tid; e < C::G * C::D; e += C::NW * 32) {
    const int h = e / C::D;
    const int dim = e % C::D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) M = fmaxf(M, warp_ml[w * C::G + h].x);
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < C::NW; ++w) {
        const float2 ml = warp_ml[w * C::G + h];
        const float f = ex2(ml.x - M);  // 0 for a warp that saw no token
        Lsum = fmaf(f, ml.y, Lsum);
        O = fmaf(f, comb[((size_t)w * C::G + h) * C::D + dim], O);
      }
    }
    const float o = (Lsum > 0.f) ? O / Lsum : 0.f;
    if (p.num_splits == 1) {
      reinterpret_cast<__nv_bfloat16*>(p.out)[(row_hq + h) * C::D + dim] = __float2bfloat16_rn(o);
    } else {
      const size_t prow = (row_hq + h) * p.num_splits + split;
      p.o_part[prow * C::D + dim] = o;
      if (dim == 0) p.lse_part[prow] = (Lsum > 0.f) ? (M + log2f(Lsum)) * 0.69314718055994530942f : -INFINITY;
    }
  }
}

// ---- instantiation and dispatch -------------------------------------------------

#define PD_STAGE1_INSTANCE(ID, D, G, KVS, NW, SPW)                                                   \
  template __global__ void stage1_kernel<Stage1Cfg<D, G, KVS, NW, SPW>>(const Stage1Params);
PD_FOR_EACH_VARIANT(PD_STAGE1_INSTANCE)
#undef PD_STAGE1_INSTANCE

const void* stage1_kernel_ptr(int variant) {
  switch (variant) {
#define PD_STAGE1_CASE(ID, D, G, KVS, NW, SPW) \
  case ID:                                     \
    return reinterpret_cast<const void*>(&stage1_kernel<Stage1Cfg<D, G, KVS, NW, SPW>>);
    PD_FOR_EACH_VARIANT(PD_STAGE1_CASE)
#undef PD_STAGE1_CASE
    default:
      return nullptr;
  }
}

}  // namespace pd
