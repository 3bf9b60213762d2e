// Kernel parameter blocks and launch entry points shared by the C ABI layer.
#pragma once

#include <cstdint>

#include <cuda.h>  // CUtensorMap (the encoder itself is fetched from the driver at run time)

#include "pd_variants.h"

namespace pd {

struct Stage1Params {
  // TMA descriptors of the K and V pools (V's = K's for a K=V layer), viewed as
  // rank 3 {64 dims, rows = pages*Hkv*P, D/64 slabs} (tma_rank 3) or as rank 2
  // {D, rows} (tma_rank 2); a 16-row box lands as [slab][row][128 B], 128-byte swizzled.
  CUtensorMap kmap;
  CUtensorMap vmap;
  int32_t tma_rank;
  const uint16_t* q;            // bf16 [B, Hq, D] ([B, T, Hq, D] on multi-token variants)
  const uint16_t* k_pool;       // bf16 [num_pages, Hkv, P, D] (FP8: e4m3 bytes, read only by TMA)
  const uint16_t* v_pool;       // bf16, == k_pool for a K=V layer
  const float* k_scale;         // FP8: [num_pages, Hkv] scale of each (page, KV head) of K
  const float* v_scale;         // FP8: same for V (== k_scale for a K=V layer)
  const int32_t* block_tables;  // [B, max_pages]
  const int32_t* seq_lens;      // [B]
  void* out;                    // bf16 [B, Hq, D] (written when num_splits == 1)
  float* lse_part;              // [B, Hq, S] natural-log log-sum-exp of each piece
  float* o_part;                // [B, Hq, S, D] normalised partial outputs
  uint32_t* err;                // device error word
  int32_t direct_out;           // one piece and a bf16 result wanted: the CTA writes `out` itself
  int32_t cluster_merge;        // the S pieces of a (request, KV head) are one cluster; rank 0 merges:
                                // 1 = they push into rank 0's drained ring (two cluster barriers),
                                // 2 = into rank 0's region of its own (one barrier; S - 1 <= DED_SLOTS)
  int32_t stall_bytes;          // tests only: bytes expected per stage beyond what the copies deliver
  int32_t early_kv;             // no kernel still running when this grid starts writes a length,
                                // page id, scale or cached row older than the newest query_tokens
                                // positions: the producer copies such rows before its dependency wait
  float scale_log2;             // softmax scale * log2(e)
  int32_t window;               // 0 = global layer
  int32_t num_pages, max_pages, page_size;
  int32_t num_q_heads, num_kv_heads;
  int32_t num_splits, chunk_tokens;
  // multi-token variants: T query tokens per request (q and out [B, T, Hq, D]),
  // the GQA group at run time, and the CTAs (column tiles of 8 (token, head)
  // pairs) per KV head: blockIdx.y = KV head * col_tiles + tile
  int32_t query_tokens, group, col_tiles;
};

struct MergeParams {
  // piece s of row r: o_part[r * row_stride + s * piece_stride + d] (floats),
  // lse_part[r * lse_row_stride + s * lse_piece_stride]; stage 1's workspace
  // is [rows][S][D] / [rows][S], a cross-rank combine's input [S][rows][D] / [S][rows]
  const float* lse_part;
  const float* o_part;
  int64_t row_stride, piece_stride, lse_row_stride, lse_piece_stride;
  void* out;              // bf16 [rows, D], or null
  float* out_f32;         // fp32 [rows, D], or null
  float* out_lse;         // fp32 [rows] natural-log log-sum-exp of the merged row, or null
  int32_t num_splits;
  int32_t head_dim;
};

// Address of the stage-1 kernel of a variant (nullptr if unknown).
const void* stage1_kernel_ptr(int variant);

// Launch the merge for rows = B * Hq; returns the CUDA error code.
int launch_merge(const MergeParams& p, int rows, void* stream);

}  // namespace pd
