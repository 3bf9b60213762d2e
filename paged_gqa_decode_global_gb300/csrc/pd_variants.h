// Kernel instances of the stage-1 decode pass and their launch geometry.
// Shared by the host planner and the kernels so both agree on every size.
#pragma once

#include <cstdint>

namespace pd {

// Device error-word bits (mirrors PD_DEVFLAG_* of the public header).
constexpr uint32_t kErrBadPage = 0x1u;
constexpr uint32_t kErrBadSeqLen = 0x2u;
constexpr uint32_t kErrTimeout = 0x4u;

// Workspace: [error word, padded to 256 B][lse fp32 B*Hq*S][o_part fp32 B*Hq*S*D]
constexpr uint64_t kWorkspaceHeader = 256;

// Geometry of one stage-1 instance.
//   D   head_dim          G    query heads per KV head (GQA group)
//   KVS K=V shared pool   NW   consumer warps (+1 producer warp)
//   SPW ring stages owned by each consumer warp
template <int D_, int G_, bool KVS_, int NW_, int SPW_>
struct Stage1Cfg {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr bool KVS = KVS_;
  static constexpr int NW = NW_;
  static constexpr int SPW = SPW_;
  // Tokens per pipeline stage: the block a warp reduces at once. TB * G partial
  // dot products per lane feed one 32-lane reduce-scatter.
  static constexpr int TB = (G <= 4) ? 8 : 32 / G;
  static constexpr int NV = TB * G;   // partial dot products per lane per block (<= 32)
  static constexpr int R = 32 / NV;   // lanes that end up holding each full dot product
  static constexpr int NCH = D / 256; // 16-byte chunks per lane per token row
  static constexpr int DPL = NCH * 8; // head dims per lane
  static constexpr int NST = NW * SPW;
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int KV_BYTES = TB * ROW_BYTES;             // one of K or V per stage
  static constexpr int STAGE_BYTES = KV_BYTES * (KVS ? 1 : 2);
  static constexpr int RING_BYTES = NST * STAGE_BYTES;
  static constexpr int COMBINE_BYTES = NW * G * D * 4;         // per-warp accumulators (aliases the ring)
  static constexpr int BODY_BYTES = RING_BYTES > COMBINE_BYTES ? RING_BYTES : COMBINE_BYTES;
  static constexpr int BAR_OFFSET = BODY_BYTES;                // full[NST], empty[NST]
  static constexpr int VALID_OFFSET = BAR_OFFSET + NST * 16;   // u32 valid[NST]
  static constexpr int ML_OFFSET = VALID_OFFSET + NST * 4;     // float2 ml[NW][G]
  static constexpr int SMEM_BYTES = ML_OFFSET + NW * G * 8;
  static constexpr int THREADS = 32 * (NW + 1);
  static_assert(D % 256 == 0, "head_dim must be a multiple of 256");
  static_assert(NV <= 32 && (32 % NV) == 0, "block must fit one reduce-scatter");
  static_assert(16 % TB == 0, "a block must lie inside one 16-token page slice");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// The instances this library is built with, by variant id. Seven consumer
// warps plus the producer make two warps per SM sub-partition, which leaves each
// thread the full 255-register budget (q and accumulators of all G heads live in
// registers). Ring depth by stage size: 16 KiB x 14, 8 KiB x 28, 4 KiB x 56.
#define PD_FOR_EACH_VARIANT(X)      \
  X(0, 512, 1, false, 7, 2)         \
  X(1, 512, 2, false, 7, 2)         \
  X(2, 512, 4, false, 7, 2)         \
  X(3, 512, 1, true, 7, 4)          \
  X(4, 512, 2, true, 7, 4)          \
  X(5, 512, 4, true, 7, 4)          \
  X(6, 256, 1, false, 7, 4)         \
  X(7, 256, 2, false, 7, 4)         \
  X(8, 256, 4, false, 7, 4)         \
  X(9, 256, 8, false, 7, 8)         \
  X(10, 256, 1, true, 7, 8)         \
  X(11, 256, 2, true, 7, 8)         \
  X(12, 256, 4, true, 7, 8)         \
  X(13, 256, 8, true, 7, 8)

struct VariantInfo {
  int id, head_dim, group, kv_shared, nw, spw, block_tokens, threads, smem_bytes;
};

// Host-visible table, defined in plan.cu.
extern const VariantInfo kVariants[];
extern const int kNumVariants;

}  // namespace pd
