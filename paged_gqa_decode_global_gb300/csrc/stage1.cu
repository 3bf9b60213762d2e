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
//   * warp NW is the producer: its lanes fetch the page ids of 32 blocks at a
//     time and one lane issues, per block of 16 tokens, one tiled TMA copy of the block's K rows (and one of its V rows)
//     into a ring stage laid out [64-dim slab][token row][128 B] with the
//     128-byte swizzle, so the 8 rows an ldmatrix reads fall in 8 different
//     bank groups; completion is counted in bytes on the stage's mbarrier;
//   * consumer warp w owns ring stages w, w+NW, ... and processes blocks
//     w, w+NW, ... of the piece with its own online-softmax state, so warps
//     never wait on one another inside the loop;
//   * both contractions run on the tensor cores (mma.sync m16n8k16, bf16
//     inputs, fp32 accumulation), with the GQA group as the 8-wide N side:
//       QK: S[16 tok x 8 heads]  = K[16 x d] . q^T       (A = K rows, B = q)
//       PV: O^T[d x 8 heads]    += V^T[d x 16 tok] . P^T (A = V rows via
//           ldmatrix.trans, B = P transposed in registers with movmatrix);
//   * FP8 (e4m3) caches land in the ring as bytes; each lane loads its MMA
//     fragments straight from them with 16-byte shared loads and widens them
//     to f16 in registers (exact), taking the head dims in an order that
//     makes every load feed four MMAs (q and the output follow that order);
//     the products run in f16 with fp32 accumulation, the per-(page, KV head)
//     K scale multiplies the scores and the V scale the probabilities;
//   * the online softmax runs in base 2 on the S fragments (scale * log2 e
//     applied in fp32); each lane owns two heads, so the rescale of its O^T
//     fragments needs no communication;
//   * at the end the NW warp states are merged in shared memory and the CTA
//     writes bf16 output (one piece), or keeps its normalised result and
//     log-sum-exp for rank 0 of its thread-block cluster to merge over
//     distributed shared memory (up to 8 pieces), or writes an fp32 partial +
//     log-sum-exp for the merge kernel (more pieces);
//   * the grid is a programmatic dependent of the kernel before it: barriers
//     are set up while that kernel drains, and with early_kv the producer
//     already copies the cached rows that kernel cannot be writing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pd_common.cuh"
#include "pd_kernels.h"

namespace pd {

namespace {

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A . B + D, m16n8k16, bf16 x bf16 -> fp32.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A . B + D, m16n8k16, f16 x f16 -> fp32 (the FP8 path: e4m3 widens to f16 exactly).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four e4m3 bytes (little-endian in w) -> four f16 (exact), as two f16x2
// words: the hardware conversion takes a 16-bit pair, lower byte to lower half.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// FP8 QK order of the head dims. In k-step ks = 8*sl + 4*hf + jj the MMA's
// columns 2*(lane%4) + {0, 1} and + {8, 9} are the dims d + {0, 1} and
// d + {2, 3}, d = 128*sl + 16*(2*(lane%4) + hf) + 4*jj: four consecutive bytes
// of the 16-byte chunk 2*(lane%4) + hf of the 128-dim slab sl, so one load of a
// token row feeds four k-steps. (A sum over the dims may take them in any
// order, as long as q and K agree.)

// Lane r of each group of four lanes holds words v[0..3] of row r of a 4 x 4
// matrix of 32-bit words; afterwards it holds column r (v[s] = row s's word r):
// two butterfly rounds, each swapping the 2 x 2 blocks' off-diagonal halves.
__device__ __forceinline__ void quad_transpose(uint4& v, int lane) {
  const bool odd = (lane & 1) != 0;
  uint32_t s0 = odd ? v.x : v.y, s1 = odd ? v.z : v.w;
  s0 = __shfl_xor_sync(kFullMask, s0, 1);
  s1 = __shfl_xor_sync(kFullMask, s1, 1);
  if (odd) {
    v.x = s0;
    v.z = s1;
  } else {
    v.y = s0;
    v.w = s1;
  }
  const bool hi = (lane & 2) != 0;
  s0 = hi ? v.x : v.z;
  s1 = hi ? v.y : v.w;
  s0 = __shfl_xor_sync(kFullMask, s0, 2);
  s1 = __shfl_xor_sync(kFullMask, s1, 2);
  if (hi) {
    v.x = s0;
    v.y = s1;
  } else {
    v.z = s0;
    v.w = s1;
  }
}

// Transpose an 8x8 bf16 matrix held one row pair per lane (fragment layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace

// The query rows behind the CC columns of a CTA (CC = 8 MMA columns for each
// of its TW tiles). Decode variants: column c is query head g*G + c of
// request b. Column-tiled variants: column c is pair tile*8 + c of the
// request's T x group (token, head) pairs, token-major, where tile is the
// CTA's first 8-column tile: token j = pair / group, head g*group + pair %
// group, row (b*T + j)*Hq + head of q and out; pairs past T x group are unused
// columns.
template <class C>
struct ColMap {
  int b, g, tile, T, group, Hq;
  __device__ __forceinline__ ColMap(const Stage1Params& p) {
    b = blockIdx.z;
    Hq = p.num_q_heads;
    if constexpr (C::MQ) {
      g = blockIdx.y / p.col_tiles;
      tile = (blockIdx.y % p.col_tiles) * C::TW;
      T = p.query_tokens;
      group = p.group;
    } else {
      g = blockIdx.y;
      tile = 0;
      T = 1;
      group = C::G;
    }
  }
  __device__ __forceinline__ bool valid(int c) const {
    return C::MQ ? (c < C::CC && tile * C::G + c < T * group) : c < C::G;
  }
  __device__ __forceinline__ int token(int c) const { return C::MQ ? (tile * C::G + c) / group : 0; }
  __device__ __forceinline__ size_t row(int c) const {
    if constexpr (C::MQ) {
      const int pr = tile * C::G + c;
      return ((size_t)b * T + pr / group) * Hq + (size_t)g * group + pr % group;
    } else {
      return (size_t)b * Hq + (size_t)g * C::G + c;
    }
  }
};

// One CTA's piece: stream, attend, merge the warps, and leave the piece's result
// in `out` (one piece), in the workspace (pieces merged by a later launch) or in
// this CTA's shared memory (pieces merged across the cluster). Threads return
// from here at different points; none leaves the kernel early.
// What a thread of stage1_cta has done towards the cluster merge when every
// piece pushes into a region of rank 0's own (one cluster barrier):
constexpr int kMergeNothing = 0;   // not waited at the cluster barrier; the CTA pushed nothing
constexpr int kMergePushed = 1;    // waited there, and the CTA's result went out (rank 0: stayed local)
constexpr int kMergeToWait = 2;    // not waited; the CTA's result went out (the producer warp)

template <class C>
__device__ __forceinline__ int stage1_cta(const Stage1Params& p, uint8_t* smem) {
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFFSET);
  uint64_t* empty_bar = full_bar + C::NST;
  uint32_t* stage_valid = reinterpret_cast<uint32_t*>(smem + C::VALID_OFFSET);
  float2* stage_scale = reinterpret_cast<float2*>(smem + C::SCALE_OFFSET);  // FP8: (K, V) scale per block of a stage
  float2* warp_ml = reinterpret_cast<float2*>(smem + C::ML_OFFSET);

  // Prologue, before the previous kernel on the stream may have finished: the
  // producer's lane 0 prefetches the tensor maps (kernel parameters) and sets
  // up the ring's barriers. Then every thread waits for that kernel: nothing
  // below reads or writes global memory before it has completed -- except,
  // with early_kv, the producer warp's reads of the lengths, page ids, FP8
  // scales and the cached rows older than each request's newest query_tokens
  // positions (data the caller guarantees that kernel does not write): it
  // waits before the first copy of a block holding a newer row, before the
  // first copy that has to wait for a free stage, and before it leaves. It
  // writes nothing to global memory before that wait: a bad page id it meets
  // is recorded in a register and reaches the error word afterwards.
  const bool early = p.early_kv != 0 && threadIdx.x >= C::NW * 32;
  if (threadIdx.x == C::NW * 32) {
    prefetch_tensormap(&p.kmap);
    if (!C::KVS) prefetch_tensormap(&p.vmap);
#pragma unroll 1
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::TW);  // each team's warp for the stage releases it
    }
    fence_barrier_init();
  }
  if (!early) grid_dependency_wait();

  const ColMap<C> cm(p);
  const int split = blockIdx.x;
  const int g = cm.g;
  const int b = cm.b;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // consumer warps form TW teams of WB; team t serves the CTA's columns
  // [8t, 8t + 8) and its warps split the stage blocks
  const int team = warp / C::WB;
  const int cb = team * C::G;  // first CTA column of this warp's team

  // The consumers issue their q loads first, so that their latency overlaps
  // the length's (q does not depend on it); an empty piece drops them.
  // B fragments of q (heads on N, dims on K): lane holds head lane/4, dims
  // 2*(lane%4) + {0,1} and + {8,9} of every 16-dim step; heads past G are zero.
  const int qh = lane >> 2;
  uint32_t qb[C::KSTEPS][2];
  if (warp != C::NW) {
    const bool qv = cm.valid(cb + qh);
    const uint16_t* qrow = p.q + (qv ? cm.row(cb + qh) * C::D : 0);
    if constexpr (C::KV8) {
      // dims in the FP8 QK order (see the consumer loop): half hf of slab sl
      // gives lane r the 16 dims of chunk 2r + hf, four per k-step; the
      // products run in f16, so q rounds to f16 once here
#pragma unroll
      for (int sl = 0; sl < C::TMA_SLABS; ++sl) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint4 a = make_uint4(0u, 0u, 0u, 0u), c = a;
          if (qv) {
            const uint4* src = reinterpret_cast<const uint4*>(qrow + sl * 128 + (2 * (lane & 3) + hf) * 16);
            a = __ldg(src);
            c = __ldg(src + 1);
          }
          const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int ks = sl * 8 + hf * 4 + jj;
            qb[ks][0] = pack_f16x2(__uint_as_float(w[2 * jj] << 16), __uint_as_float(w[2 * jj] & 0xffff0000u));
            qb[ks][1] =
                pack_f16x2(__uint_as_float(w[2 * jj + 1] << 16), __uint_as_float(w[2 * jj + 1] & 0xffff0000u));
          }
        }
      }
    } else if constexpr (!C::MQ) {
      // decode: this lane's q dims 16 ks + 2r + {0, 1} and 16 ks + 8 + 2r +
      // {0, 1} as 4-byte loads (issued together here; the vector form below
      // measured slower for these instances)
      const int qk = (lane & 3) * 2;
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        if (qv) {
          qb[ks][0] = __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16 + qk));
          qb[ks][1] = __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16 + 8 + qk));
        } else {
          qb[ks][0] = 0u;
          qb[ks][1] = 0u;
        }
      }
    } else {
      // column-tiled instances, whose 4-byte loads issued in several round
      // trips (~2.5 us against ~0.7): lane r of a quad loads both 16-byte
      // halves of k-steps 4i + r (the quad reads 128 contiguous bytes); a
      // 4 x 4 transpose of 32-bit words across the quad then leaves with lane
      // r word r of every half: q dims 16 ks + 2r + {0, 1} and 16 ks + 8 + 2r
      // + {0, 1}
#pragma unroll
      for (int i = 0; i < C::KSTEPS / 4; ++i) {
        const int ks = 4 * i + (lane & 3);
        uint4 a = make_uint4(0u, 0u, 0u, 0u), c = a;
        if (qv) {
          a = __ldg(reinterpret_cast<const uint4*>(qrow + ks * 16));
          c = __ldg(reinterpret_cast<const uint4*>(qrow + ks * 16 + 8));
        }
        quad_transpose(a, lane);
        quad_transpose(c, lane);
        qb[4 * i + 0][0] = a.x;
        qb[4 * i + 1][0] = a.y;
        qb[4 * i + 2][0] = a.z;
        qb[4 * i + 3][0] = a.w;
        qb[4 * i + 0][1] = c.x;
        qb[4 * i + 1][1] = c.y;
        qb[4 * i + 2][1] = c.z;
        qb[4 * i + 3][1] = c.w;
      }
    }
  }


  // ---- attended range of this request and this piece -------------------------
  const int cap = p.max_pages * p.page_size;
  const int32_t* table = p.block_tables + (size_t)b * p.max_pages;
  // On a global layer a piece starts at split * chunk whatever the length, so
  // the producer fetches its first page ids while the length is in flight:
  // with one lane per stage, lane st those of stage block st; with the batch
  // walk, lane k that of block k.
  constexpr bool kLanePerStage = C::LANE_PER_STAGE;
  int page_spec[C::NSUB];
#pragma unroll
  for (int u = 0; u < C::NSUB; ++u) {
    page_spec[u] = -1;
    const int blk = kLanePerStage ? lane * C::NSUB + u : (u == 0 ? lane : -1);
    if (warp == C::NW && p.window == 0 && blk >= 0 && (!kLanePerStage || lane < C::NST)) {
      const long long t = (long long)split * p.chunk_tokens + (long long)blk * C::TB;
      if (t < cap) page_spec[u] = __ldg(table + t / p.page_size);
    }
  }
  int L = p.seq_lens[b];
  if (L < 0 || L > cap || (C::MQ && cm.T > 1 && L < cm.T)) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadSeqLen);
    L = L < 0 ? 0 : (L > cap ? cap : L);
  }
  // attended range [lo, hi) of this CTA's query rows: decode, the last W (or
  // all) positions; multi-token, the union of its tokens' causal ranges, token
  // j ending at its own position L - T + j (inclusive)
  int hi = L, lo;
  if constexpr (C::MQ) {
    const int j_first = cm.token(0);
    int j_last = cm.token(C::CC - 1);
    if (j_last > cm.T - 1) j_last = cm.T - 1;
    hi = L - cm.T + j_last + 1;
    if (hi < 0) hi = 0;
    const int first_hi = L - cm.T + j_first + 1;
    lo = (p.window > 0 && first_hi > p.window) ? first_hi - p.window : 0;
  } else {
    lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
  }
  const int base = (lo / C::TB) * C::TB;
  const long long piece_lo = (long long)base + (long long)split * p.chunk_tokens;
  const int tlo = (int)(piece_lo > lo ? piece_lo : lo);
  // the last piece takes whatever remains, so a device length longer than the
  // planned one is still attended in full
  const long long piece_hi = (split == p.num_splits - 1) ? (long long)hi : piece_lo + p.chunk_tokens;
  const int thi = (int)(piece_hi < hi ? piece_hi : hi);
  const int blk_lo = (tlo / C::TB) * C::TB;
  const int nblk = (thi > tlo) ? (thi - blk_lo + C::TB - 1) / C::TB : 0;
  // stages of this piece: NSUB consecutive blocks each (the last may hold fewer)
  const int nstg = (nblk + C::NSUB - 1) / C::NSUB;

  if (nblk == 0) {
    // nothing attended in this piece
    if (early) grid_dependency_wait();
    if (p.cluster_merge) {
      if (threadIdx.x < C::CC) reinterpret_cast<float*>(smem + C::CTA_LSE_OFFSET)[threadIdx.x] = -INFINITY;
    } else if (p.direct_out) {
      for (int i = threadIdx.x; i < C::CC * C::D; i += C::THREADS)
        if (cm.valid(i / C::D))
          reinterpret_cast<__nv_bfloat16*>(p.out)[cm.row(i / C::D) * C::D + i % C::D] = __float2bfloat16_rn(0.f);
    } else {
      // weight 0 and a zero partial row, so the merge needs no special case
      for (int i = threadIdx.x; i < C::CC * C::D; i += C::THREADS)
        if (cm.valid(i / C::D)) p.o_part[(cm.row(i / C::D) * p.num_splits + split) * C::D + i % C::D] = 0.f;
      if (threadIdx.x < C::CC && cm.valid(threadIdx.x))
        p.lse_part[cm.row(threadIdx.x) * p.num_splits + split] = -INFINITY;
    }
    return kMergeNothing;
  }

  // The ring's barriers (set up by the producer's lane 0 at entry) are
  // visible to the consumers once they pass named barrier 2, at which the
  // producer only arrives: it issues its first copies without waiting for
  // the consumers' q loads.
  if (warp == C::NW)
    named_bar_arrive(2, C::THREADS);
  else
    named_bar_sync(2, C::THREADS);
  // a merge launched behind this kernel may start its (waiting) CTAs now.
  // Every thread that signals has waited for the launch in front: a producer
  // lane with early_kv signals once it has (below), so that a launch behind
  // this one can rely on everything in front of this one being complete.
  if (!early) grid_launch_dependents();

  // ---- producer ------------------------------------------------------------------
  if (warp == C::NW) {
    if constexpr (kLanePerStage) {
    // Lane st owns ring stage st: it walks the stage blocks st, st + NST, ...
    // of the piece on its own, fetching the next one's page ids (and FP8
    // scales) while it waits for the stage to be released, then issuing that
    // block's copies. Stages never wait for one another, and each lane waits
    // only for the use of its stage it issued itself.
    const uint64_t policy = l2_evict_first_policy();
    bool waited = !early;  // this lane's dependency wait
    // error bits seen by this lane, published once this grid may write global
    // memory (after its dependency wait)
    uint32_t err_bits = 0;
    int last_jb = -1;  // the last stage block this lane issued
    // blocks ending after this position hold rows the previous kernel may write
    const int fresh_from = L - p.query_tokens;
    if (lane < C::NST) {
      const int st = lane;
      uint8_t* dst = smem + (size_t)st * C::STAGE_BYTES;
      // page ids (and scales) of stage block jb, fetched one use ahead
      auto fetch = [&](int jb, int (&pg)[C::NSUB], float2 (&sc)[C::NSUB]) {
#pragma unroll
        for (int u = 0; u < C::NSUB; ++u) {
          const int j = jb * C::NSUB + u;
          pg[u] = (jb < nstg && j < nblk) ? __ldg(table + (blk_lo + j * C::TB) / p.page_size) : -1;
          sc[u] = make_float2(1.f, 1.f);
          if constexpr (C::KV8) {
            if ((unsigned)pg[u] < (unsigned)p.num_pages) {
              const size_t si = (size_t)pg[u] * p.num_kv_heads + g;
              sc[u].x = __ldg(p.k_scale + si);
              sc[u].y = C::KVS ? sc[u].x : __ldg(p.v_scale + si);
            }
          }
        }
      };
      int pg[C::NSUB];
      float2 sc[C::NSUB];
      if (p.window == 0) {
        // the ids fetched before the length (a piece of a global layer starts at split * chunk)
#pragma unroll
        for (int u = 0; u < C::NSUB; ++u) {
          pg[u] = (st * C::NSUB + u < nblk) ? page_spec[u] : -1;
          sc[u] = make_float2(1.f, 1.f);
          if constexpr (C::KV8) {
            if ((unsigned)pg[u] < (unsigned)p.num_pages) {
              const size_t si = (size_t)pg[u] * p.num_kv_heads + g;
              sc[u].x = __ldg(p.k_scale + si);
              sc[u].y = C::KVS ? sc[u].x : __ldg(p.v_scale + si);
            }
          }
        }
      } else {
        fetch(st, pg, sc);
      }
#pragma unroll 1
      for (int jb = st; jb < nstg; jb += C::NST) {
        int pg_next[C::NSUB];
        float2 sc_next[C::NSUB];
        fetch(jb + C::NST, pg_next, sc_next);
        if (!waited && (jb >= C::NST || blk_lo + (jb + 1) * C::NSUB * C::TB > fresh_from)) {
          grid_dependency_wait();
          grid_launch_dependents();
          waited = true;
        }
        const int round = jb / C::NST;
        if (round > 0 && !mbar_wait(&empty_bar[st], (round - 1) & 1)) {
          err_bits |= kErrTimeout;
          break;
        }
        // blocks of this stage that exist and have a page in the pool
        uint32_t bits = 0;
#pragma unroll
        for (int u = 0; u < C::NSUB; ++u) {
          if (jb * C::NSUB + u >= nblk) continue;
          if ((unsigned)pg[u] < (unsigned)p.num_pages)
            bits |= 1u << u;
          else
            err_bits |= kErrBadPage;
        }
        stage_valid[st] = bits;
        if constexpr (C::KV8) {
#pragma unroll
          for (int u = 0; u < C::NSUB; ++u) stage_scale[st * C::NSUB + u] = sc[u];
        }
        if (bits) {
          mbar_arrive_expect_tx(&full_bar[st], __popc(bits) * C::BLOCK_TX + p.stall_bytes);
#pragma unroll
          for (int u = 0; u < C::NSUB; ++u) {
            if (!((bits >> u) & 1u)) continue;
            const int t0 = blk_lo + (jb * C::NSUB + u) * C::TB;
            const int row0 = (pg[u] * p.num_kv_heads + g) * p.page_size + (t0 % p.page_size);
            uint8_t* kd = dst + u * C::KV_BYTES;
            uint8_t* vd = dst + C::V_OFFSET + u * C::KV_BYTES;
            if (p.tma_rank == 3) {
              tma_load_3d(kd, &p.kmap, 0, row0, 0, &full_bar[st], policy);
              if (!C::KVS) tma_load_3d(vd, &p.vmap, 0, row0, 0, &full_bar[st], policy);
            } else {
              constexpr int SLAB_ELEMS = 128 / C::ELEM;
#pragma unroll
              for (int sl = 0; sl < C::TMA_SLABS; ++sl) {
                tma_load_2d(kd + sl * C::SLAB_BYTES, &p.kmap, sl * SLAB_ELEMS, row0, &full_bar[st], policy);
                if (!C::KVS)
                  tma_load_2d(vd + sl * C::SLAB_BYTES, &p.vmap, sl * SLAB_ELEMS, row0, &full_bar[st], policy);
              }
            }
          }
        } else {
          mbar_arrive(&full_bar[st]);
        }
        last_jb = jb;
#pragma unroll
        for (int u = 0; u < C::NSUB; ++u) {
          pg[u] = pg_next[u];
          sc[u] = sc_next[u];
        }
      }
    }
    if (!waited) {
      grid_dependency_wait();
      grid_launch_dependents();
    }
    // no copy may still be landing in shared memory when the CTA exits: each
    // lane waits for its stage's last copies
    if (last_jb >= 0 && !mbar_wait(&full_bar[lane], (last_jb / C::NST) & 1)) err_bits |= kErrTimeout;
    err_bits = __reduce_or_sync(kFullMask, err_bits);
    if (lane == 0 && err_bits) atomicOr(p.err, err_bits);
    } else {
    const uint64_t policy = l2_evict_first_policy();
    // page id of block `lane` of the first batch
    int page_next = -1;
    if (lane < nblk) page_next = (p.window == 0) ? page_spec[0] : __ldg(table + (blk_lo + lane * C::TB) / p.page_size);
    int* batch_row = reinterpret_cast<int*>(smem + C::BATCH_ROW_OFFSET);
    float2* batch_scale = reinterpret_cast<float2*>(smem + C::BATCH_SCALE_OFFSET);
    // The warp walks the blocks 32 at a time: lane k turns block j0 + k's page
    // id (fetched a batch ahead) into the pool row its copies start at (and,
    // FP8, fetches its scales) and leaves them in shared memory; lane 0 alone
    // then waits for each stage and issues its copies, with no warp-wide step
    // per block.
    int issued = 0;  // stage blocks issued (lane 0)
    bool stop = false;
    bool waited = !early;  // lane 0's dependency wait
    // error bits seen by lane 0, published once this grid may write global
    // memory (after its dependency wait)
    uint32_t err_bits = 0;
    // blocks ending after this position hold rows the previous kernel may write
    const int fresh_from = L - p.query_tokens;
    constexpr int kNoBlock = -1, kBadPage = -2;
#pragma unroll 1
    for (int j0 = 0; j0 < nblk && !stop; j0 += 32) {
      const int jk = j0 + lane;
      int row = kNoBlock;
      float2 sc = make_float2(1.f, 1.f);
      if (jk < nblk) {
        if ((unsigned)page_next < (unsigned)p.num_pages) {
          row = (page_next * p.num_kv_heads + g) * p.page_size + ((blk_lo + jk * C::TB) % p.page_size);
          if constexpr (C::KV8) {
            const size_t si = (size_t)page_next * p.num_kv_heads + g;
            sc.x = __ldg(p.k_scale + si);
            sc.y = C::KVS ? sc.x : __ldg(p.v_scale + si);
          }
        } else {
          row = kBadPage;
        }
      }
      const int jn = j0 + 32 + lane;
      page_next = (jn < nblk) ? __ldg(table + (blk_lo + jn * C::TB) / p.page_size) : -1;
      batch_row[lane] = row;
      if constexpr (C::KV8) batch_scale[lane] = sc;
      __syncwarp();
      if (lane == 0) {
        const int cnt = min(32, nblk - j0);
        // one stage per NSUB consecutive blocks (32 is a multiple of NSUB, so
        // a stage never straddles two batches)
#pragma unroll 1
        for (int k = 0; k < cnt; k += C::NSUB) {
          const int jb = (j0 + k) / C::NSUB;  // stage block
          if (!waited && (jb >= C::NST || blk_lo + (j0 + k + C::NSUB) * C::TB > fresh_from)) {
            grid_dependency_wait();
            grid_launch_dependents();
            waited = true;
          }
          const int st = jb % C::NST;
          const int round = jb / C::NST;
          if (round > 0 && !mbar_wait(&empty_bar[st], (round - 1) & 1)) {
            err_bits |= kErrTimeout;
            stop = true;
            break;
          }
          // blocks of this stage that exist and have a page in the pool
          int rows[C::NSUB];
          uint32_t bits = 0;
#pragma unroll
          for (int u = 0; u < C::NSUB; ++u) {
            rows[u] = (k + u < cnt) ? batch_row[k + u] : kNoBlock;
            if (rows[u] >= 0) bits |= 1u << u;
            if (rows[u] == kBadPage) err_bits |= kErrBadPage;
          }
          stage_valid[st] = bits;
          if constexpr (C::KV8) {
#pragma unroll
            for (int u = 0; u < C::NSUB; ++u) stage_scale[st * C::NSUB + u] = batch_scale[(k + u) & 31];
          }
          if (bits) {
            uint8_t* dst = smem + (size_t)st * C::STAGE_BYTES;
            mbar_arrive_expect_tx(&full_bar[st], __popc(bits) * C::BLOCK_TX + p.stall_bytes);
#pragma unroll
            for (int u = 0; u < C::NSUB; ++u) {
              if (!((bits >> u) & 1u)) continue;
              uint8_t* kd = dst + u * C::KV_BYTES;
              uint8_t* vd = dst + C::V_OFFSET + u * C::KV_BYTES;
              if (p.tma_rank == 3) {
                tma_load_3d(kd, &p.kmap, 0, rows[u], 0, &full_bar[st], policy);
                if (!C::KVS) tma_load_3d(vd, &p.vmap, 0, rows[u], 0, &full_bar[st], policy);
              } else {
                constexpr int SLAB_ELEMS = 128 / C::ELEM;
#pragma unroll
                for (int sl = 0; sl < C::TMA_SLABS; ++sl) {
                  tma_load_2d(kd + sl * C::SLAB_BYTES, &p.kmap, sl * SLAB_ELEMS, rows[u], &full_bar[st], policy);
                  if (!C::KVS)
                    tma_load_2d(vd + sl * C::SLAB_BYTES, &p.vmap, sl * SLAB_ELEMS, rows[u], &full_bar[st], policy);
                }
              }
            }
          } else {
            mbar_arrive(&full_bar[st]);
          }
          issued = jb + 1;
        }
      }
      // lane 0 is done with this batch's entries before they are rewritten
      stop = __shfl_sync(kFullMask, stop, 0);
    }
    if (early && !(lane == 0 && waited)) {
      grid_dependency_wait();
      grid_launch_dependents();
    }
    // no copy may still be landing in shared memory when the CTA exits (one
    // deadline for all stages)
    if (lane == 0) {
      const unsigned long long deadline = global_timer_ns() + kWaitTimeoutNs;
#pragma unroll 1
      for (int st = 0; st < C::NST && st < issued; ++st) {
        const int j_last = st + C::NST * ((issued - 1 - st) / C::NST);
        if (!mbar_wait_until(&full_bar[st], (j_last / C::NST) & 1, deadline)) {
          err_bits |= kErrTimeout;
          break;
        }
      }
      if (err_bits) atomicOr(p.err, err_bits);
    }
    }
    return (C::DED_SLOTS > 0 && p.cluster_merge == 2) ? kMergeToWait : kMergeNothing;
  }

  // ---- consumers -----------------------------------------------------------------
  // O^T accumulators: m-tile mt holds dims mt*16 + lane/4 (+8) x heads 2*(lane%4) (+1)
  float acc[C::MTILES][4];
#pragma unroll
  for (int mt = 0; mt < C::MTILES; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;

  // multi-token: the causal range [col_lo, col_hi) of this lane's two columns
  int col_lo[2] = {0, 0}, col_hi[2] = {0, 0};
  if constexpr (C::MQ) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = cb + (lane & 3) * 2 + cc;
      if (cm.valid(c)) {
        col_hi[cc] = L - cm.T + cm.token(c) + 1;
        col_lo[cc] = (p.window > 0 && col_hi[cc] > p.window) ? col_hi[cc] - p.window : 0;
      }
    }
  }

  // this lane's two heads and their running max / sum (base-2 logits)
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  // Per-lane ldmatrix offsets inside a stage. Byte (row r, 16-byte chunk c) of
  // a slab sits at r * 128 + ((c ^ (r % 8)) * 16): the 128-byte swizzle.
  // K (non-trans): lane supplies row (lane%8) + 8*((lane/8)%2), chunk 2*j + lane/16
  // V (trans):     lane supplies row (lane%8) + 8*(lane/16),    chunk 2*j + (lane/8)%2
  // for the 16-dim step j (mod 4) of a 64-dim slab.
  const int sw = lane & 7;
  const int kr = (lane & 7) | (((lane >> 3) & 1) << 3), kc = lane >> 4;
  const int vr = (lane & 7) | ((lane >> 4) << 3), vc = (lane >> 3) & 1;
  uint32_t koff[4], voff[4];
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    koff[jj] = (uint32_t)(kr * 128 + (((2 * jj + kc) ^ sw) << 4));
    voff[jj] = (uint32_t)(vr * 128 + (((2 * jj + vc) ^ sw) << 4));
  }
  const uint32_t ring = smem_u32(smem);

#pragma unroll 1
  for (int jb = warp % C::WB; jb < nstg; jb += C::WB) {
    const int st = jb % C::NST;
    // every lane polls; the warp leaves together if any lane gave up
    const bool landed = mbar_wait(&full_bar[st], (jb / C::NST) & 1);
    if (__any_sync(kFullMask, !landed)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      break;
    }
    const uint32_t kst = ring + st * C::STAGE_BYTES;
    const uint32_t vst = C::KVS ? kst : kst + C::V_OFFSET;
    const uint32_t valid_bits = stage_valid[st];
    const int t0 = blk_lo + jb * (C::NSUB * C::TB);  // first token of the stage
    const uint8_t* stg = smem + (size_t)st * C::STAGE_BYTES;
    float k_sc[C::NSUB], v_sc[C::NSUB];
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {
      k_sc[u] = 1.f;
      v_sc[u] = 1.f;
      if constexpr (C::KV8) {
        const float2 sc = stage_scale[st * C::NSUB + u];
        k_sc[u] = sc.x;
        v_sc[u] = sc.y;
      }
    }

    // QK on the tensor cores, block by block, four independent accumulation
    // chains each. s[u]: this lane's scores of block u: tokens t0 + 16u + lane/4
    // (s[u][0], s[u][1]) and + 8 (s[u][2], s[u][3]); heads 2*(lane%4) (s[u][0],
    // s[u][2]) and 2*(lane%4) + 1 (s[u][1], s[u][3])
    float s[C::NSUB][4];
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {
      float sacc[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) sacc[c][i] = 0.f;
      if constexpr (C::KV8) {
        // A fragments straight from the e4m3 rows: one 16-byte chunk of token
        // rows lane/4 and lane/4 + 8 holds this lane's part of four k-steps
        // (the dims are taken in the FP8 QK order; q follows it)
        const uint8_t* kb = stg + u * C::KV_BYTES;
#pragma unroll
        for (int sl = 0; sl < C::TMA_SLABS; ++sl) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint8_t* sp = kb + sl * C::SLAB_BYTES + qh * 128 + (((2 * (lane & 3) + hf) ^ qh) << 4);
            const uint4 ra = *reinterpret_cast<const uint4*>(sp);
            const uint4 rb = *reinterpret_cast<const uint4*>(sp + 8 * 128);
            const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
            const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              uint32_t a[4];
              e4m3x4_to_f16x4(wa[jj], a[0], a[2]);
              e4m3x4_to_f16x4(wb[jj], a[1], a[3]);
              const int ks = sl * 8 + hf * 4 + jj;
              mma_f16(sacc[jj], a, qb[ks][0], qb[ks][1]);
            }
          }
        }
      } else {
        const uint32_t kb = kst + u * C::KV_BYTES;
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ++ks) {
          uint32_t a[4];
          ldmatrix_x4(a, kb + (ks >> 2) * C::SLAB_BYTES + koff[ks & 3]);
          mma_bf16(sacc[ks & 3], a, qb[ks][0], qb[ks][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s[u][i] = ((sacc[0][i] + sacc[1][i]) + (sacc[2][i] + sacc[3][i])) * (p.scale_log2 * k_sc[u]);
    }

    // masks: rows outside the piece's range, of a skipped page, or (multi-token
    // columns) outside the column's own causal range
    bool va[C::NSUB], vb[C::NSUB];
    bool all_in = true;
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {
      const bool ok = (valid_bits >> u) & 1u;
      const int ta = t0 + u * C::TB + qh;
      va[u] = ok && ta >= tlo && ta < thi;
      vb[u] = ok && ta + 8 >= tlo && ta + 8 < thi;
      all_in = all_in && va[u] && vb[u];
      if constexpr (C::MQ) {
        if (!(va[u] && ta >= col_lo[0] && ta < col_hi[0])) s[u][0] = -INFINITY;
        if (!(va[u] && ta >= col_lo[1] && ta < col_hi[1])) s[u][1] = -INFINITY;
        if (!(vb[u] && ta + 8 >= col_lo[0] && ta + 8 < col_hi[0])) s[u][2] = -INFINITY;
        if (!(vb[u] && ta + 8 >= col_lo[1] && ta + 8 < col_hi[1])) s[u][3] = -INFINITY;
      } else {
        if (!va[u]) s[u][0] = s[u][1] = -INFINITY;
        if (!vb[u]) s[u][2] = s[u][3] = -INFINITY;
      }
    }

    // online softmax: max and sum over the stage's tokens (lane/4, the two
    // rows and the NSUB blocks)
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {
      bm0 = fmaxf(bm0, fmaxf(s[u][0], s[u][2]));
      bm1 = fmaxf(bm1, fmaxf(s[u][1], s[u][3]));
    }
#pragma unroll
    for (int mask = 4; mask < 32; mask <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(kFullMask, bm0, mask));
      bm1 = fmaxf(bm1, __shfl_xor_sync(kFullMask, bm1, mask));
    }
    const float mn0 = fmaxf(m_run[0], bm0), mn1 = fmaxf(m_run[1], bm1);
    const float alpha0 = (mn0 == -INFINITY) ? 1.f : ex2(m_run[0] - mn0);
    const float alpha1 = (mn1 == -INFINITY) ? 1.f : ex2(m_run[1] - mn1);
    const float ms0 = (mn0 == -INFINITY) ? 0.f : mn0, ms1 = (mn1 == -INFINITY) ? 0.f : mn1;
    float pr[C::NSUB][4];
    float bs0 = 0.f, bs1 = 0.f;
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {
      pr[u][0] = ex2(s[u][0] - ms0);
      pr[u][1] = ex2(s[u][1] - ms1);
      pr[u][2] = ex2(s[u][2] - ms0);
      pr[u][3] = ex2(s[u][3] - ms1);
      bs0 += pr[u][0] + pr[u][2];
      bs1 += pr[u][1] + pr[u][3];
    }
#pragma unroll
    for (int mask = 4; mask < 32; mask <<= 1) {
      bs0 += __shfl_xor_sync(kFullMask, bs0, mask);
      bs1 += __shfl_xor_sync(kFullMask, bs1, mask);
    }
    l_run[0] = l_run[0] * alpha0 + bs0;
    l_run[1] = l_run[1] * alpha1 + bs1;
    m_run[0] = mn0;
    m_run[1] = mn1;
    if (__any_sync(kFullMask, alpha0 != 1.f || alpha1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < C::MTILES; ++mt) {
        acc[mt][0] *= alpha0;
        acc[mt][1] *= alpha1;
        acc[mt][2] *= alpha0;
        acc[mt][3] *= alpha1;
      }
    }

    // Edge stage (window start, sequence end, skipped page): the masked rows
    // carry p = 0, but 0 * NaN is NaN, and a page's unused rows may hold any
    // bits, so their V values are zeroed in registers before the PV
    // contraction (several teams may read one stage: shared memory is left
    // as it landed). This lane's PV fragments of block u hold tokens
    // 2*(lane%4) + {0, 1} (halves of words 0 and 1) and + {8, 9} (words 2, 3).
    // (The FP8 path masks its own fragments in the PV loop.)
    bool edge = false;
    if constexpr (!C::KV8) edge = __any_sync(kFullMask, !all_in);

    // P^T as the B operand of each block: transpose the (token x head) 16-bit
    // fragments; on the FP8 path the block's V scale rides on P
    // (sum_t p_t (v_sc v8_t))
    uint32_t pb[C::NSUB][2];
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {
      if constexpr (C::KV8) {
        pb[u][0] = movmatrix_trans(pack_f16x2(pr[u][0] * v_sc[u], pr[u][1] * v_sc[u]));  // tokens 0..7
        pb[u][1] = movmatrix_trans(pack_f16x2(pr[u][2] * v_sc[u], pr[u][3] * v_sc[u]));  // tokens 8..15
      } else {
        pb[u][0] = movmatrix_trans(pack_bf16x2(pr[u][0], pr[u][1]));
        pb[u][1] = movmatrix_trans(pack_bf16x2(pr[u][2], pr[u][3]));
      }
    }

    // PV on the tensor cores
    if constexpr (C::KV8) {
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u) {
        // A fragments (dims x tokens) straight from the e4m3 rows: this lane
        // reads the 16-byte chunk lane/4 of tokens 2*(lane%4) + {0, 1, 8, 9}.
        // Byte 2w (2w + 1) of a chunk is taken as the dim of row lane/4
        // (lane/4 + 8) of m-tile w of the slab, so row i of m-tile w holds dim
        // 16*(i%8) + 2w + i/8 (the epilogue puts each back); a byte permute
        // pairs one dim of two tokens.
        const int tv = 2 * (lane & 3);
        const int t_a = t0 + u * C::TB + tv;
        const bool ok = (valid_bits >> u) & 1u;
        const bool ok0 = ok && t_a >= tlo && t_a < thi;
        const bool ok1 = ok && t_a + 1 >= tlo && t_a + 1 < thi;
        const bool ok2 = ok && t_a + 8 >= tlo && t_a + 8 < thi;
        const bool ok3 = ok && t_a + 9 >= tlo && t_a + 9 < thi;
        // a block every row of which is attended (all but the edge blocks) needs no zeroing
        const bool edge_u = __any_sync(kFullMask, !(ok0 && ok1 && ok2 && ok3));
        const uint8_t* vstg = (C::KVS ? stg : stg + C::V_OFFSET) + u * C::KV_BYTES;
#pragma unroll
        for (int sl = 0; sl < C::TMA_SLABS; ++sl) {
          const uint8_t* vp = vstg + sl * C::SLAB_BYTES;
          const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
          // rows the sequence does not cover may hold any bits: e4m3 zero instead
          uint4 r0 = *reinterpret_cast<const uint4*>(vp + tv * 128 + ((qh ^ tv) << 4));
          uint4 r1 = *reinterpret_cast<const uint4*>(vp + (tv + 1) * 128 + ((qh ^ (tv + 1)) << 4));
          uint4 r2 = *reinterpret_cast<const uint4*>(vp + (tv + 8) * 128 + ((qh ^ tv) << 4));
          uint4 r3 = *reinterpret_cast<const uint4*>(vp + (tv + 9) * 128 + ((qh ^ (tv + 1)) << 4));
          if (edge_u) {
            if (!ok0) r0 = zero;
            if (!ok1) r1 = zero;
            if (!ok2) r2 = zero;
            if (!ok3) r3 = zero;
          }
          const uint32_t x0[4] = {r0.x, r0.y, r0.z, r0.w}, x1[4] = {r1.x, r1.y, r1.z, r1.w};
          const uint32_t x2[4] = {r2.x, r2.y, r2.z, r2.w}, x3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
              const uint32_t sel = u2 ? 0x7362u : 0x5140u;
              uint32_t a[4];
              e4m3x4_to_f16x4(__byte_perm(x0[w], x1[w], sel), a[0], a[1]);
              e4m3x4_to_f16x4(__byte_perm(x2[w], x3[w], sel), a[2], a[3]);
              mma_f16(acc[sl * 8 + w * 2 + u2], a, pb[u][0], pb[u][1]);
            }
          }
        }
      }
    } else if (edge) {
      uint32_t vmask[C::NSUB][2];
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u) {
        const bool ok = (valid_bits >> u) & 1u;
        const int tv = t0 + u * C::TB + 2 * (lane & 3);
        const bool k0 = ok && tv >= tlo && tv < thi, k1 = ok && tv + 1 >= tlo && tv + 1 < thi;
        const bool k8 = ok && tv + 8 >= tlo && tv + 8 < thi, k9 = ok && tv + 9 >= tlo && tv + 9 < thi;
        vmask[u][0] = (k0 ? 0x0000ffffu : 0u) | (k1 ? 0xffff0000u : 0u);
        vmask[u][1] = (k8 ? 0x0000ffffu : 0u) | (k9 ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int mt = 0; mt < C::MTILES; ++mt) {
#pragma unroll
        for (int u = 0; u < C::NSUB; ++u) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, vst + u * C::KV_BYTES + (mt >> 2) * C::SLAB_BYTES + voff[mt & 3]);
          a[0] &= vmask[u][0];
          a[1] &= vmask[u][0];
          a[2] &= vmask[u][1];
          a[3] &= vmask[u][1];
          mma_bf16(acc[mt], a, pb[u][0], pb[u][1]);
        }
      }
    } else {
#pragma unroll
      for (int mt = 0; mt < C::MTILES; ++mt) {
#pragma unroll
        for (int u = 0; u < C::NSUB; ++u) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, vst + u * C::KV_BYTES + (mt >> 2) * C::SLAB_BYTES + voff[mt & 3]);
          mma_bf16(acc[mt], a, pb[u][0], pb[u][1]);
        }
      }
    }

    __syncwarp();
    asm volatile("" ::: "memory");
    if (lane == 0) mbar_arrive(&empty_bar[st]);
  }

  // ---- merge the NW warp states --------------------------------------------------
  named_bar_sync(1, C::NW * 32);  // every consumer is done with the ring
  // per-warp accumulators [NW][G][CS]: the 4-float pad of a head row puts the
  // heads 2 apart that a warp stores at once in different banks
  constexpr int CS = C::COMB_STRIDE;
  float* comb = reinterpret_cast<float*>(smem);
  const int h0 = (lane & 3) * 2;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = h0 + hh;
    if (h < C::G) {
      if constexpr (C::KV8) {
        // rows lane/4 and lane/4 + 8 of m-tile u of slab sl are dims
        // sl*128 + 16*(lane/4) + 2u + {0, 1}
        float* dst = comb + (warp * C::G + h) * CS + 16 * qh;
#pragma unroll
        for (int mt = 0; mt < C::MTILES; ++mt)
          *reinterpret_cast<float2*>(dst + (mt >> 3) * 128 + 2 * (mt & 7)) = make_float2(acc[mt][hh], acc[mt][2 + hh]);
      } else {
        float* dst = comb + (warp * C::G + h) * CS + qh;
#pragma unroll
        for (int mt = 0; mt < C::MTILES; ++mt) {
          dst[mt * 16] = acc[mt][hh];
          dst[mt * 16 + 8] = acc[mt][2 + hh];
        }
      }
      if (qh == 0) warp_ml[warp * C::G + h] = make_float2(m_run[hh], l_run[hh]);
    }
  }
  named_bar_sync(1, C::NW * 32);

  // merge coefficients, one thread per (warp, head), over the warps of its team:
  //   c_w = 2^(m_w - M) / sum_w' 2^(m_w' - M) l_w'  (0 for a warp that saw no token)
  // and the piece's natural-log log-sum-exp per CTA column
  const int tid = threadIdx.x;
  float* coef = reinterpret_cast<float*>(smem + C::COEF_OFFSET);  // [NW][G], then lse[CC]
  if (tid < C::NW * C::G) {
    const int w = tid / C::G, h = tid % C::G;
    const int w0 = (w / C::WB) * C::WB;  // the team's first warp
    float M = -INFINITY;
#pragma unroll
    for (int v = 0; v < C::WB; ++v) M = fmaxf(M, warp_ml[(w0 + v) * C::G + h].x);
    float Lsum = 0.f, mine = 0.f;
#pragma unroll
    for (int v = 0; v < C::WB; ++v) {
      const float2 ml = warp_ml[(w0 + v) * C::G + h];
      const float f = (M == -INFINITY) ? 0.f : ex2(ml.x - M);
      Lsum = fmaf(f, ml.y, Lsum);
      if (w0 + v == w) mine = f;
    }
    coef[w * C::G + h] = Lsum > 0.f ? mine / Lsum : 0.f;
    if (w == w0)
      coef[C::NW * C::G + (w / C::WB) * C::G + h] =
          (Lsum > 0.f) ? (M + __log2f(Lsum)) * 0.69314718055994530942f : -INFINITY;
  }
  named_bar_sync(1, C::NW * 32);
  const float* col_lse = coef + C::NW * C::G;  // [CC]

  // One-barrier cluster merge: once every CTA of the cluster has started
  // (each arrived at the barrier at kernel entry), ranks 1..S-1 store their
  // rows and lse straight into rank 0's region; rank 0 keeps its own locally.
  const bool fused = C::DED_SLOTS > 0 && p.cluster_merge == 2;
  bool to_rank0 = false;
  uint32_t remote_out = 0, remote_lse = 0;
  if (fused) {
    cluster_wait();
    const uint32_t rank = cluster_ctarank();
    if (rank != 0) {
      to_rank0 = true;
      remote_out = map_smem_rank(smem_u32(smem + C::DED_OFFSET) + (rank - 1) * (C::CC * C::D * 4), 0);
      remote_lse = map_smem_rank(smem_u32(smem + C::DED_LSE_OFFSET) + (rank - 1) * (C::CC * 4), 0);
    }
  }

  constexpr int D4 = C::D / 4;
#pragma unroll 2
  for (int e = tid; e < C::CC * D4; e += C::NW * 32) {
    const int h = e / D4;  // CTA column
    const int d4 = e % D4;
    if (C::MQ && !cm.valid(h)) continue;
    const int w0 = (h / C::G) * C::WB, hc = h % C::G;  // its team's first warp, its MMA column
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int v = 0; v < C::WB; ++v) {
      const float c = coef[(w0 + v) * C::G + hc];
      const float4 a = *reinterpret_cast<const float4*>(comb + ((w0 + v) * C::G + hc) * CS + d4 * 4);
      o.x = fmaf(c, a.x, o.x);
      o.y = fmaf(c, a.y, o.y);
      o.z = fmaf(c, a.z, o.z);
      o.w = fmaf(c, a.w, o.w);
    }
    if (p.direct_out) {
      __nv_bfloat162* dst =
          reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(p.out) + cm.row(h) * C::D) + d4 * 2;
      uint2 packed;
      packed.x = pack_bf16x2(o.x, o.y);
      packed.y = pack_bf16x2(o.z, o.w);
      *reinterpret_cast<uint2*>(dst) = packed;
    } else if (to_rank0) {
      st_dsmem_f32x4(remote_out + (h * D4 + d4) * 16, o);
      if (d4 == 0) st_dsmem_f32(remote_lse + h * 4, col_lse[h]);
    } else if (p.cluster_merge) {
      // kept in shared memory for rank 0 of the cluster (or to push from)
      reinterpret_cast<float4*>(smem + C::CTA_OUT_OFFSET)[h * D4 + d4] = o;
      if (d4 == 0) reinterpret_cast<float*>(smem + C::CTA_LSE_OFFSET)[h] = col_lse[h];
    } else {
      const size_t prow = cm.row(h) * p.num_splits + split;
      reinterpret_cast<float4*>(p.o_part + prow * C::D)[d4] = o;
      if (d4 == 0) p.lse_part[prow] = col_lse[h];
    }
  }
  return fused ? kMergePushed : kMergeNothing;
}

// Stage 2 inside the cluster (vLLM concepts page, "MLA 与 Sparse MLA（DSA）":
// the pieces' partial results, each with its log-sum-exp, are merged). The S
// CTAs of one (request, KV head) form a cluster; each holds its normalised
// result and log-sum-exp in shared memory. Ranks 1..S-1 push theirs into rank
// 0 with posted distributed-shared-memory stores -- into a region of rank 0's
// own when S - 1 results fit beside the ring (every CTA arrived at a cluster
// barrier when it started, which the pushers wait for), else into rank 0's
// ring once a first cluster barrier shows every CTA done with it; after the
// next cluster barrier rank 0 merges locally:
//   out = sum_r w_r o_r,  w_r = exp(lse_r - M) / sum_r' exp(lse_r' - M),  M = max_r lse_r
// in piece order; pieces with no attended token (lse = -inf) weigh nothing.
template <class C>
__device__ __forceinline__ void cluster_merge(const Stage1Params& p, uint8_t* smem, int state) {
  const int S = p.num_splits;
  const uint32_t rank = cluster_ctarank();
  const int tid = threadIdx.x;
  constexpr int D4 = C::D / 4;
  const float* my_lse = reinterpret_cast<const float*>(smem + C::CTA_LSE_OFFSET);
  const float4* my_out = reinterpret_cast<const float4*>(smem + C::CTA_OUT_OFFSET);
  const bool own_region = C::DED_SLOTS > 0 && p.cluster_merge == 2;
  const int push_off = own_region ? C::DED_OFFSET : C::PUSH_OFFSET;
  const int push_lse_off = own_region ? C::DED_LSE_OFFSET : C::PUSH_LSE_OFFSET;
  // (with its own region a CTA that attended something has pushed already --
  // all its threads have state kMergePushed or kMergeToWait -- and an empty
  // one, all of whose threads have state kMergeNothing, pushes its lse here)
  if (own_region) {
    if (state == kMergeNothing) __syncthreads();  // this CTA's lse is in place
    if (state != kMergePushed) cluster_wait();    // every CTA of the cluster has started
  } else {
    cluster_sync_all();  // every CTA of the cluster is done with its ring
  }
  if (rank != 0 && state == kMergeNothing) {
    const uint32_t slot = smem_u32(smem + push_off) + (rank - 1) * (C::CC * C::D * 4);
    const uint32_t lse_slot = smem_u32(smem + push_lse_off) + (rank - 1) * (C::CC * 4);
    if (tid < C::CC) st_dsmem_f32(map_smem_rank(lse_slot + tid * 4, 0), my_lse[tid]);
    const uint32_t remote = map_smem_rank(slot, 0);
    for (int e = tid; e < C::CC * D4; e += C::THREADS) {
      if (my_lse[e / D4] == -INFINITY) continue;  // nothing attended: only the lse is pushed
      st_dsmem_f32x4(remote + e * 16, my_out[e]);
    }
  }
  cluster_sync_all();  // the pushes are visible in rank 0
  if (rank != 0) return;
  const float* push_lse = reinterpret_cast<const float*>(smem + push_lse_off);
  const float4* push_out = reinterpret_cast<const float4*>(smem + push_off);
  float* wts = reinterpret_cast<float*>(smem + C::CTA_W_OFFSET);  // [S][CC]
  // one thread per (piece, head): w = exp(lse - M) / sum_r exp(lse_r - M),
  // every thread of a head reading that head's S log-sum-exps
  if (tid < S * C::CC) {
    const int r = tid / C::CC, h = tid % C::CC;
    float l[C::MAX_CLUSTER];
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < C::MAX_CLUSTER; ++q) {
      l[q] = q >= S ? -INFINITY : (q == 0 ? my_lse[h] : push_lse[(q - 1) * C::CC + h]);
      M = fmaxf(M, l[q]);
    }
    float sum = 0.f, mine = 0.f;
    constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
    for (int q = 0; q < C::MAX_CLUSTER; ++q) {
      const float e = (M == -INFINITY || q >= S) ? 0.f : ex2((l[q] - M) * kLog2e);
      sum += e;
      if (q == r) mine = e;
    }
    wts[r * C::CC + h] = sum > 0.f ? mine / sum : 0.f;
  }
  __syncthreads();
  const ColMap<C> cm(p);
#pragma unroll 1
  for (int e = tid; e < C::CC * D4; e += C::THREADS) {
    const int h = e / D4;
    if (C::MQ && !cm.valid(h)) continue;
    // all S pieces' weights and rows loaded before any is used; an empty
    // piece pushed no row (its slot may hold anything) and weighs 0: selected
    // out rather than multiplied
    float w[C::MAX_CLUSTER];
    float4 v[C::MAX_CLUSTER];
#pragma unroll
    for (int r = 0; r < C::MAX_CLUSTER; ++r) {
      if (r < S) {
        w[r] = wts[r * C::CC + h];
        v[r] = r == 0 ? my_out[e] : push_out[(r - 1) * C::CC * D4 + e];
      } else {
        w[r] = 0.f;
        v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < C::MAX_CLUSTER; ++r) {
      const bool use = w[r] != 0.f;
      acc.x = use ? fmaf(w[r], v[r].x, acc.x) : acc.x;
      acc.y = use ? fmaf(w[r], v[r].y, acc.y) : acc.y;
      acc.z = use ? fmaf(w[r], v[r].z, acc.z) : acc.z;
      acc.w = use ? fmaf(w[r], v[r].w, acc.w) : acc.w;
    }
    uint2 packed;
    packed.x = pack_bf16x2(acc.x, acc.y);
    packed.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + cm.row(h) * C::D + (e % D4) * 4) = packed;
  }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) stage1_kernel(const __grid_constant__ Stage1Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzle pattern repeats every 1024 bytes of shared address: start there
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  if (C::DED_SLOTS > 0 && p.cluster_merge == 2) cluster_arrive_relaxed();  // this CTA has started
  const int state = stage1_cta<C>(p, smem);
  if (p.cluster_merge) cluster_merge<C>(p, smem, state);
}

// ---- instantiation and dispatch -------------------------------------------------

#define PD_STAGE1_INSTANCE(ID, D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW)                       \
  template __global__ void stage1_kernel<Stage1Cfg<D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW>>( \
      const __grid_constant__ Stage1Params);
PD_FOR_EACH_VARIANT(PD_STAGE1_INSTANCE)
#undef PD_STAGE1_INSTANCE

const void* stage1_kernel_ptr(int variant) {
  switch (variant) {
#define PD_STAGE1_CASE(ID, D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW) \
  case ID:                                                        \
    return reinterpret_cast<const void*>(&stage1_kernel<Stage1Cfg<D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW>>);
    PD_FOR_EACH_VARIANT(PD_STAGE1_CASE)
#undef PD_STAGE1_CASE
    default:
      return nullptr;
  }
}

}  // namespace pd
