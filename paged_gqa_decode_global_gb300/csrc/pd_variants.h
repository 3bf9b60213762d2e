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
//   D   head_dim          G    query heads per KV head (GQA group, <= 8: the
//                              8-wide N side of the m16n8k16 MMAs)
//   KVS K=V shared pool   KV8  the KV cache holds e4m3 bytes (+ per-(page, KV
//                              head) scales) instead of bf16
//   NW  consumer warps (+1 producer warp)
//   SPW ring stages owned by each consumer warp
//   MQ  column-tiled (several query tokens per request, or one token with a
//       group of 9..16): the G = 8 MMA columns hold (token, head) pairs of
//       the request's T x group pairs, token-major, 8 per CTA, and each
//       column is masked causally by its own token's position
//   NSUB 16-token blocks per ring stage: each block is one tiled copy of K (and
//       one of V); the stage's blocks share its mbarrier round trip and one
//       online-softmax update
//   TW  column tiles per CTA (column-tiled instances): the NW consumer warps
//       form TW teams of NW / TW, team t serves the CTA's tile t (8 columns)
//       over every stage block, its warps splitting the blocks; one copy of
//       each block then feeds the TW teams
template <int D_, int G_, bool KVS_, bool KV8_, int NW_, int SPW_, bool MQ_ = false, int NSUB_ = 1, int TW_ = 1>
struct Stage1Cfg {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr bool KVS = KVS_;
  static constexpr bool KV8 = KV8_;
  static constexpr int NW = NW_;
  static constexpr int SPW = SPW_;
  static constexpr bool MQ = MQ_;
  static constexpr int NSUB = NSUB_;
  static constexpr int TW = TW_;
  static constexpr int WB = NW / TW;             // consumer warps of a team
  static constexpr int CC = TW * G;              // columns (query rows) of a CTA
  static constexpr int TB = 16;                  // tokens per block = the MMA's 16-row side
  static constexpr int KSTEPS = D / 16;          // QK k-steps
  static constexpr int MTILES = D / 16;          // PV m-tiles (head dims)
  static constexpr int NST = WB * SPW;          // stages: a team's warps own SPW each
  static constexpr int SLAB_BYTES = TB * 128;    // one 128-byte-wide slab of a 16-token block
  // what TMA lands per K (or V) block, [slab][16 rows][128 B] with the
  // 128-byte swizzle: bf16 rows (64 dims a slab) or e4m3 rows (128 dims)
  static constexpr int SLABS = D / 64;           // bf16 slabs
  static constexpr int ELEM = KV8 ? 1 : 2;
  static constexpr int TMA_SLABS = D * ELEM / 128;
  static constexpr int KV_BYTES = TMA_SLABS * SLAB_BYTES;       // one block of K (or V)
  static constexpr int BLOCK_TX = KV_BYTES * (KVS ? 1 : 2);     // bytes the copies of one block deliver
  // a stage: the K of its NSUB blocks, then (K != V) their V
  static constexpr int V_OFFSET = NSUB * KV_BYTES;
  static constexpr int STAGE_BYTES = NSUB * BLOCK_TX;
  static constexpr int RING_BYTES = NST * STAGE_BYTES;
  static constexpr int WORK_BYTES = RING_BYTES;
  static constexpr int COMB_STRIDE = D + 4;                    // floats per head row of the warp merge
  static constexpr int COMBINE_BYTES = NW * G * COMB_STRIDE * 4; // per-warp outputs (aliases the ring)
  static constexpr int BODY_BYTES = WORK_BYTES > COMBINE_BYTES ? WORK_BYTES : COMBINE_BYTES;
  // cluster merge (after the ring is drained): this CTA's result and lse, and
  // rank 0's merge weights; rank 0 then receives the results of ranks
  // 1..S-1, float [S-1][CC][D] + lse [S-1][CC], in what is left of the body
  static constexpr int CTA_OUT_OFFSET = (COMBINE_BYTES + 15) / 16 * 16;  // float [CC][D]
  static constexpr int CTA_LSE_OFFSET = CTA_OUT_OFFSET + CC * D * 4;     // float [CC]
  static constexpr int CTA_W_OFFSET = CTA_LSE_OFFSET + CC * 4;           // float [8][CC]
  // the pushes go after rank 0's weights, or into its warp-merge buffers
  // (dead once its result is out, which the first cluster barrier orders
  // before any push), whichever is larger
  static constexpr int TAIL_PUSH_OFFSET = (CTA_W_OFFSET + 8 * CC * 4 + 15) / 16 * 16;
  static constexpr int TAIL_PUSH_ROOM = BODY_BYTES - TAIL_PUSH_OFFSET;
  static constexpr int HEAD_PUSH_ROOM = CTA_OUT_OFFSET;
  static constexpr int PUSH_OFFSET = HEAD_PUSH_ROOM > TAIL_PUSH_ROOM ? 0 : TAIL_PUSH_OFFSET;
  static constexpr int PUSH_ROOM = HEAD_PUSH_ROOM > TAIL_PUSH_ROOM ? HEAD_PUSH_ROOM : TAIL_PUSH_ROOM;
  static constexpr int MAX_CLUSTER_FIT = 1 + (PUSH_ROOM > 0 ? PUSH_ROOM / ((CC * D + CC) * 4) : 0);
  static constexpr int MAX_CLUSTER = MAX_CLUSTER_FIT < 8 ? MAX_CLUSTER_FIT : 8;  // pieces one cluster merges
  static constexpr int PUSH_LSE_OFFSET = PUSH_OFFSET + (MAX_CLUSTER - 1) * CC * D * 4;
  static_assert(PUSH_LSE_OFFSET + (MAX_CLUSTER - 1) * CC * 4 <= PUSH_OFFSET + PUSH_ROOM,
                "cluster merge buffers fit in their region");
  static constexpr int BAR_OFFSET = BODY_BYTES;                // full[NST], empty[NST]
  static constexpr int VALID_OFFSET = BAR_OFFSET + NST * 16;   // u32 valid[NST]: one bit per block
  static constexpr int SCALE_OFFSET = (VALID_OFFSET + NST * 4 + 7) / 8 * 8;  // float2 (k, v) scale[NST][NSUB] (FP8)
  static constexpr int ML_OFFSET = SCALE_OFFSET + NST * NSUB * 8;  // float2 ml[NW][G]
  static constexpr int COEF_OFFSET = ML_OFFSET + NW * G * 8;   // float coef[NW][G], lse[CC]
  // Rings of 24..32 stages are fed by one producer lane per stage (each lane
  // waits for its own stage and issues its copies); other rings by the
  // producer warp's batch walk, lane 0 issuing in order.
  static constexpr bool LANE_PER_STAGE = NST >= 24 && NST <= 32;
  // the batch walk's 32 blocks: pool row of each (or a negative code) and,
  // FP8, its (K, V) scales
  static constexpr int BATCH_ROW_OFFSET = (COEF_OFFSET + (NW * G + CC) * 4 + 7) / 8 * 8;  // int [32]
  static constexpr int BATCH_SCALE_OFFSET = BATCH_ROW_OFFSET + (LANE_PER_STAGE ? 0 : 32 * 4);  // float2 [32]
  static constexpr int TAIL_END = (BATCH_SCALE_OFFSET + (LANE_PER_STAGE ? 0 : 32 * 8) + 15) / 16 * 16;
  // Pieces that can push into a region of their own, outside the ring (what
  // is left of the 227 KiB): with them the cluster merge needs one cluster
  // barrier (other ranks may store while rank 0 still streams); larger
  // clusters push into rank 0's drained ring after a first barrier.
  static constexpr int DED_ROOM = 227 * 1024 - 1024 - TAIL_END - 8 * CC * 4;
  static constexpr int DED_FIT = DED_ROOM > 0 ? DED_ROOM / (CC * D * 4) : 0;
  static constexpr int DED_SLOTS = DED_FIT < MAX_CLUSTER - 1 ? DED_FIT : MAX_CLUSTER - 1;
  static constexpr int DED_OFFSET = TAIL_END;                  // float [DED_SLOTS][CC][D]
  static constexpr int DED_LSE_OFFSET = DED_OFFSET + DED_SLOTS * CC * D * 4;  // float [DED_SLOTS][CC]
  // + 1 KiB so the ring can start on a 1024-byte boundary (the swizzle period)
  static constexpr int SMEM_BYTES = DED_LSE_OFFSET + (DED_SLOTS > 0 ? DED_SLOTS * CC * 4 : 0) + 1024;
  static constexpr int THREADS = 32 * (NW + 1);
  static_assert(D % 128 == 0, "head_dim must be a multiple of 128");
  static_assert(G >= 1 && G <= 8, "the GQA group is the MMA's 8-wide side");
  static_assert(16 % TB == 0, "a block must lie inside one 16-token page slice");
  static_assert(NSUB >= 1 && 32 % NSUB == 0, "a stage's blocks come from one batch of 32 page ids");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(SCALE_OFFSET % 8 == 0 && ML_OFFSET % 8 == 0, "float2 arrays need 8-byte alignment");
  static_assert(!MQ || G == 8, "multi-token variants use all 8 columns");
  static_assert(MAX_CLUSTER * CC <= THREADS, "one thread per (piece, column) computes the cluster merge weights");
  static_assert(NW % TW == 0 && (TW == 1 || MQ), "teams of equal size; several tiles only on column-tiled instances");
};

// The instances this library is built with, by variant id:
// X(id, head_dim, group, K=V, FP8, consumer warps, stages per warp, multi-token,
//   blocks per stage, column tiles per CTA).
// bf16: three consumer warps (the tensor cores leave the CUDA cores mostly
// idle) plus the producer; rings of 192 KiB: 32 KiB stages x 6 (d512 K!=V:
// one block a stage; d256 K!=V: two blocks), 16 KiB x 12 (d512 K=V: one block;
// d256 K=V and d128 K!=V: two blocks), 8 KiB x 24 (d128 K=V: two blocks).
// FP8: seven consumer warps (two per SM sub-partition hide the latency of
// widening e4m3 fragments to f16), one block a stage (two for the
// column-tiled d256 K=V instance), rings of 112-224 KiB.
// Column-tiled (ids 32-35): the group-8 geometry, any group up to 16 and any
// number of query tokens at run time, one tile of 8 columns per CTA (ids
// 44-47: the same over an FP8 cache); ids 48-51: two tiles per CTA, served by
// two teams of three consumer warps from one ring (bf16, more than 8 columns).
// head_dim 128: ids 36-43 (bf16, one query token).
// ids 52-59: the FP8 K!=V decode geometries with six consumer warps, whose
// smaller ring (192 KiB) leaves room beside it for the cluster's pushed
// results (one cluster barrier); for spans under 4096 tokens, where the
// launch's fixed costs weigh more than the seventh warp's arithmetic.
#define PD_FOR_EACH_VARIANT(X) \
  X(0, 512, 1, false, false, 3, 2, false, 1, 1)  \
  X(1, 512, 2, false, false, 3, 2, false, 1, 1)  \
  X(2, 512, 4, false, false, 3, 2, false, 1, 1)  \
  X(3, 512, 8, false, false, 3, 2, false, 1, 1)  \
  X(4, 512, 1, true, false, 3, 4, false, 1, 1)   \
  X(5, 512, 2, true, false, 3, 4, false, 1, 1)   \
  X(6, 512, 4, true, false, 3, 4, false, 1, 1)   \
  X(7, 512, 8, true, false, 3, 4, false, 1, 1)   \
  X(8, 256, 1, false, false, 3, 2, false, 2, 1)  \
  X(9, 256, 2, false, false, 3, 2, false, 2, 1)  \
  X(10, 256, 4, false, false, 3, 2, false, 2, 1) \
  X(11, 256, 8, false, false, 3, 2, false, 2, 1) \
  X(12, 256, 1, true, false, 3, 4, false, 2, 1)  \
  X(13, 256, 2, true, false, 3, 4, false, 2, 1)  \
  X(14, 256, 4, true, false, 3, 4, false, 2, 1)  \
  X(15, 256, 8, true, false, 3, 4, false, 2, 1)  \
  X(16, 512, 1, false, true, 7, 2, false, 1, 1)  \
  X(17, 512, 2, false, true, 7, 2, false, 1, 1)  \
  X(18, 512, 4, false, true, 7, 2, false, 1, 1)  \
  X(19, 512, 8, false, true, 7, 2, false, 1, 1)  \
  X(20, 512, 1, true, true, 7, 4, false, 1, 1)   \
  X(21, 512, 2, true, true, 7, 4, false, 1, 1)   \
  X(22, 512, 4, true, true, 7, 4, false, 1, 1)   \
  X(23, 512, 8, true, true, 7, 4, false, 1, 1)   \
  X(24, 256, 1, false, true, 7, 4, false, 1, 1)  \
  X(25, 256, 2, false, true, 7, 4, false, 1, 1)  \
  X(26, 256, 4, false, true, 7, 4, false, 1, 1)  \
  X(27, 256, 8, false, true, 7, 4, false, 1, 1)  \
  X(28, 256, 1, true, true, 7, 4, false, 1, 1)   \
  X(29, 256, 2, true, true, 7, 4, false, 1, 1)   \
  X(30, 256, 4, true, true, 7, 4, false, 1, 1)   \
  X(31, 256, 8, true, true, 7, 4, false, 1, 1)   \
  X(32, 512, 8, false, false, 3, 2, true, 1, 1)  \
  X(33, 512, 8, true, false, 3, 4, true, 1, 1)   \
  X(34, 256, 8, false, false, 3, 2, true, 2, 1)  \
  X(35, 256, 8, true, false, 3, 4, true, 2, 1)   \
  X(36, 128, 1, false, false, 3, 4, false, 2, 1) \
  X(37, 128, 2, false, false, 3, 4, false, 2, 1) \
  X(38, 128, 4, false, false, 3, 4, false, 2, 1) \
  X(39, 128, 8, false, false, 3, 4, false, 2, 1) \
  X(40, 128, 1, true, false, 3, 8, false, 2, 1)  \
  X(41, 128, 2, true, false, 3, 8, false, 2, 1)  \
  X(42, 128, 4, true, false, 3, 8, false, 2, 1)  \
  X(43, 128, 8, true, false, 3, 8, false, 2, 1)  \
  X(44, 512, 8, false, true, 7, 2, true, 1, 1)   \
  X(45, 512, 8, true, true, 7, 4, true, 1, 1)    \
  X(46, 256, 8, false, true, 7, 4, true, 1, 1)   \
  X(47, 256, 8, true, true, 7, 4, true, 2, 1)    \
  X(48, 512, 8, false, false, 6, 2, true, 1, 2)  \
  X(49, 512, 8, true, false, 6, 4, true, 1, 2)   \
  X(50, 256, 8, false, false, 6, 2, true, 2, 2)  \
  X(51, 256, 8, true, false, 6, 4, true, 2, 2)  \
  X(52, 512, 1, false, true, 6, 2, false, 1, 1) \
  X(53, 512, 2, false, true, 6, 2, false, 1, 1) \
  X(54, 512, 4, false, true, 6, 2, false, 1, 1) \
  X(55, 512, 8, false, true, 6, 2, false, 1, 1) \
  X(56, 256, 1, false, true, 6, 4, false, 1, 1) \
  X(57, 256, 2, false, true, 6, 4, false, 1, 1) \
  X(58, 256, 4, false, true, 6, 4, false, 1, 1) \
  X(59, 256, 8, false, true, 6, 4, false, 1, 1)

struct VariantInfo {
  int id, head_dim, group, kv_shared, kv_fp8, nw, spw, block_tokens, threads, smem_bytes, max_cluster, multi,
      ded_slots, blocks_per_stage, tiles;
};

// Host-visible table, defined in plan.cu.
extern const VariantInfo kVariants[];
extern const int kNumVariants;

}  // namespace pd
