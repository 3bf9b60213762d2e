// C ABI entry points: argument checks, kernel launch on the caller's stream,
// device error-word readback. Declarations and contracts: include/paged_decode.h.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "host_ctx.h"
#include "paged_decode.h"
#include "pd_kernels.h"

namespace pd {
bool plan_is_valid(const pd_plan* plan);
}

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxContexts = 64;

// Per CUDA context, one bit per variant whose dynamic shared-memory limit has
// been raised there (a function attribute belongs to the context it was set in).
struct SmemReady {
  unsigned long long ctx_id;
  uint64_t bits;
};
#define PD_VARIANT_ID_FITS_A_BIT(ID, ...) static_assert((ID) >= 0 && (ID) < 64, "one bit per variant id");
PD_FOR_EACH_VARIANT(PD_VARIANT_ID_FITS_A_BIT)
#undef PD_VARIANT_ID_FITS_A_BIT
std::mutex g_smem_mu;
SmemReady g_smem_ready[kMaxContexts] = {};
int g_smem_contexts = 0;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ---- TMA descriptors ----------------------------------------------------------
// cuTensorMapEncodeTiled is a driver entry point; it is looked up once through
// the runtime so the library does not link the driver library directly.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static std::atomic<EncodeTiledFn> cached{nullptr};
  EncodeTiledFn fn = cached.load(std::memory_order_acquire);
  if (fn) return fn;
  void* sym = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &sym, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !sym) {
    (void)cudaGetLastError();
    return nullptr;
  }
  fn = reinterpret_cast<EncodeTiledFn>(sym);
  cached.store(fn, std::memory_order_release);
  return fn;
}

// Rank the pools are viewed at: 3 ({64 dims, rows, slabs}, one copy per block)
// when the driver accepts that view, else 2 ({D, rows}, one copy per slab).
std::atomic<int> g_tma_rank{0};

// Describe a pool [num_pages, Hkv, P, D] bf16 for 16-row boxes that land as
// [slab][row][128 B] with the 128-byte swizzle.
pd_status encode_pool_map(CUtensorMap* map, const void* pool, const pd_layer_desc& ly, int rank) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return PD_ERR_CUDA;
  // 128-byte rows of the swizzle: 64 bf16 or 128 e4m3 elements
  const bool fp8 = ly.kv_dtype == PD_KV_FP8_E4M3;
  const cuuint64_t elem = fp8 ? 1 : 2;
  const cuuint64_t span = 128 / elem;
  const CUtensorMapDataType type = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t rows = (cuuint64_t)ly.num_pages * ly.num_kv_heads * ly.page_size;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r;
  if (rank == 3) {
    const cuuint64_t dims[3] = {span, rows, (cuuint64_t)ly.head_dim / span};
    const cuuint64_t strides[2] = {(cuuint64_t)ly.head_dim * elem, 128};
    const cuuint32_t box[3] = {(cuuint32_t)span, 16, (cuuint32_t)(ly.head_dim / span)};
    r = fn(map, type, 3, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)ly.head_dim, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ly.head_dim * elem};
    const cuuint32_t box[2] = {(cuuint32_t)span, 16};
    r = fn(map, type, 2, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? PD_OK : PD_ERR_CUDA;
}

pd_status encode_pool_maps(pd::Stage1Params& p, const void* k_pool, const void* v_pool, const pd_layer_desc& ly) {
  int rank = g_tma_rank.load(std::memory_order_acquire);
  if (rank == 0) {
    rank = encode_pool_map(&p.kmap, k_pool, ly, 3) == PD_OK ? 3 : 2;
    g_tma_rank.store(rank, std::memory_order_release);
  }
  pd_status st = encode_pool_map(&p.kmap, k_pool, ly, rank);
  if (st != PD_OK) return st;
  if (v_pool == k_pool) {
    p.vmap = p.kmap;
  } else {
    st = encode_pool_map(&p.vmap, v_pool, ly, rank);
    if (st != PD_OK) return st;
  }
  p.tma_rank = rank;
  return PD_OK;
}

pd_status ensure_smem_attr(int variant, const void* fn, int smem_bytes) {
  const pd::CtxFns* f = pd::ctx_fns();
  const unsigned long long id = f ? pd::current_ctx_id(*f) : 0;
  const uint64_t bit = 1ull << variant;
  std::lock_guard<std::mutex> lock(g_smem_mu);
  SmemReady* e = nullptr;
  if (id != 0) {
    for (int i = 0; i < g_smem_contexts; ++i)
      if (g_smem_ready[i].ctx_id == id) e = &g_smem_ready[i];
    if (e && (e->bits & bit)) return PD_OK;
  }
  // the first launch of this instance in this context (or no context id to
  // key on: set it every time)
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess) {
    (void)cudaGetLastError();
    return PD_ERR_CUDA;
  }
  const unsigned long long now = f ? pd::current_ctx_id(*f) : 0;  // the runtime call may have made one current
  if (now == 0) return PD_OK;
  if (!e || now != id) {
    e = nullptr;
    for (int i = 0; i < g_smem_contexts; ++i)
      if (g_smem_ready[i].ctx_id == now) e = &g_smem_ready[i];
    if (!e && g_smem_contexts < kMaxContexts) {
      e = &g_smem_ready[g_smem_contexts++];
      *e = SmemReady{now, 0};
    }
  }
  if (e) e->bits |= bit;
  return PD_OK;
}

pd_status stage1(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool, const float* k_scale,
                 const float* v_scale, const int32_t* block_tables, const int32_t* seq_lens, int32_t window,
                 float scale, void* workspace, size_t workspace_bytes, void* out, void* stream) {
  if (!pd::plan_is_valid(plan)) return PD_ERR_INVALID_ARG;
  const pd_layer_desc& ly = plan->layer;
  const bool fp8 = ly.kv_dtype == PD_KV_FP8_E4M3;
  if (fp8) {
    if (!k_scale || !aligned(k_scale, 4)) return PD_ERR_INVALID_ARG;
    if (ly.kv_shared) {
      if (v_scale && v_scale != k_scale) return PD_ERR_INVALID_ARG;
      v_scale = k_scale;
    } else if (!v_scale || !aligned(v_scale, 4)) {
      return PD_ERR_INVALID_ARG;
    }
  }
  if (window != ly.window) return PD_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PD_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return PD_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return PD_ERR_WORKSPACE_TOO_SMALL;
  if (plan->batch == 0) return PD_OK;
  if (!q || !k_pool || !block_tables || !seq_lens || !out) return PD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
      !aligned(seq_lens, 4))
    return PD_ERR_INVALID_ARG;
  if (ly.kv_shared) {
    if (v_pool && v_pool != k_pool) return PD_ERR_INVALID_ARG;
    v_pool = k_pool;
  } else {
    if (!v_pool || v_pool == k_pool || !aligned(v_pool, 16)) return PD_ERR_INVALID_ARG;
  }

  const void* fn = pd::stage1_kernel_ptr(plan->variant);
  if (!fn) return PD_ERR_INVALID_ARG;
  pd_status st = ensure_smem_attr(plan->variant, fn, plan->smem_bytes);
  if (st != PD_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  pd::Stage1Params p;
  std::memset(&p, 0, sizeof(p));
  st = encode_pool_maps(p, k_pool, v_pool, ly);
  if (st != PD_OK) return st;
  p.q = static_cast<const uint16_t*>(q);
  p.k_pool = static_cast<const uint16_t*>(k_pool);
  p.v_pool = static_cast<const uint16_t*>(v_pool);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse_part = reinterpret_cast<float*>(ws + plan->lse_offset);
  p.o_part = reinterpret_cast<float*>(ws + plan->opart_offset);
  p.err = reinterpret_cast<uint32_t*>(ws);
  p.direct_out = (plan->num_splits == 1 && !plan->partial) ? 1 : 0;
  if (plan->merge_mode == 2)
    p.cluster_merge = (plan->num_splits - 1 <= pd::kVariants[plan->variant].ded_slots) ? 2 : 1;
  else
    p.cluster_merge = 0;
  p.stall_bytes = plan->test_stall_bytes;
  p.early_kv = plan->early_kv;
  p.scale_log2 = scale * kLog2e;
  p.window = ly.window;
  p.num_pages = ly.num_pages;
  p.max_pages = ly.max_pages_per_seq;
  p.page_size = ly.page_size;
  p.num_q_heads = ly.num_q_heads;
  p.num_kv_heads = ly.num_kv_heads;
  p.num_splits = plan->num_splits;
  p.chunk_tokens = plan->chunk_tokens;
  p.query_tokens = plan->query_tokens;
  p.group = ly.num_q_heads / ly.num_kv_heads;
  p.col_tiles = plan->grid_y / ly.num_kv_heads;

  void* args[] = {&p};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan->grid_x, plan->grid_y, plan->grid_z);
  cfg.blockDim = dim3(plan->threads_per_cta);
  cfg.dynamicSmemBytes = plan->smem_bytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  int na = 0;
  // programmatic dependent launch: the grid may start (set up its barriers on
  // free SMs) while the previous kernel on the stream drains; it touches no
  // global memory before that kernel has finished (griddepcontrol.wait)
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (p.cluster_merge) {
    // the S pieces of one (request, KV head) are consecutive in x: one cluster
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = plan->num_splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PD_ERR_CUDA;
  }
  return PD_OK;
}

// The merge of a plan's workspace ([rows][S] pieces) into bf16 `out`, or into
// fp32 `o_f32` with the merged log-sum-exp `lse`.
pd_status merge_workspace(const pd_plan* plan, const uint8_t* ws, void* out, float* o_f32, float* lse, void* stream) {
  pd::MergeParams p = {};
  p.lse_part = reinterpret_cast<const float*>(ws + plan->lse_offset);
  p.o_part = reinterpret_cast<const float*>(ws + plan->opart_offset);
  p.row_stride = (int64_t)plan->num_splits * plan->layer.head_dim;
  p.piece_stride = plan->layer.head_dim;
  p.lse_row_stride = plan->num_splits;
  p.lse_piece_stride = 1;
  p.out = out;
  p.out_f32 = o_f32;
  p.out_lse = lse;
  p.num_splits = plan->num_splits;
  p.head_dim = plan->layer.head_dim;
  const long long rows = (long long)plan->batch * plan->query_tokens * plan->layer.num_q_heads;
  if (rows > 0x7fffffffLL) return PD_ERR_UNSUPPORTED;
  if (pd::launch_merge(p, (int)rows, stream) != 0) return PD_ERR_CUDA;
  return PD_OK;
}

}  // namespace

extern "C" {

pd_status paged_decode_global(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_tables, const int32_t* seq_lens, float scale,
                              void* workspace, size_t workspace_bytes, void* out, void* stream) {
  if (!plan || plan->layer.window != 0 || plan->layer.kv_dtype != PD_KV_BF16) return PD_ERR_INVALID_ARG;
  return stage1(plan, q, k_pool, v_pool, nullptr, nullptr, block_tables, seq_lens, 0, scale, workspace,
                workspace_bytes, out, stream);
}

pd_status paged_decode_window(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_tables, const int32_t* seq_lens, int32_t window,
                              float scale, void* workspace, size_t workspace_bytes, void* out, void* stream) {
  if (!plan || window <= 0 || plan->layer.window != window || plan->layer.kv_dtype != PD_KV_BF16)
    return PD_ERR_INVALID_ARG;
  return stage1(plan, q, k_pool, v_pool, nullptr, nullptr, block_tables, seq_lens, window, scale, workspace,
                workspace_bytes, out, stream);
}

pd_status paged_decode_global_fp8(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                                  const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                  const int32_t* seq_lens, float scale, void* workspace, size_t workspace_bytes,
                                  void* out, void* stream) {
  if (!plan || plan->layer.window != 0 || plan->layer.kv_dtype != PD_KV_FP8_E4M3) return PD_ERR_INVALID_ARG;
  return stage1(plan, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, 0, scale, workspace,
                workspace_bytes, out, stream);
}

pd_status paged_decode_window_fp8(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                                  const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                  const int32_t* seq_lens, int32_t window, float scale, void* workspace,
                                  size_t workspace_bytes, void* out, void* stream) {
  if (!plan || window <= 0 || plan->layer.window != window || plan->layer.kv_dtype != PD_KV_FP8_E4M3)
    return PD_ERR_INVALID_ARG;
  return stage1(plan, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, window, scale, workspace,
                workspace_bytes, out, stream);
}

pd_status paged_decode_merge(const pd_plan* plan, const void* workspace, size_t workspace_bytes, void* out,
                             void* stream) {
  if (!pd::plan_is_valid(plan)) return PD_ERR_INVALID_ARG;
  // mode 0: one piece, nothing to merge; mode 2: merged inside the stage-1 clusters
  if (plan->merge_mode != 1 || plan->batch == 0) return PD_OK;
  if (!workspace || !aligned(workspace, 256) || !out || !aligned(out, 16)) return PD_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return PD_ERR_WORKSPACE_TOO_SMALL;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  return merge_workspace(plan, ws, out, nullptr, nullptr, stream);
}

pd_status paged_decode_global_partial(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                                      const int32_t* block_tables, const int32_t* seq_lens, float scale,
                                      void* workspace, size_t workspace_bytes, float* o_out, float* lse_out,
                                      void* stream) {
  if (!plan || !pd::plan_is_valid(plan) || !plan->partial) return PD_ERR_INVALID_ARG;
  if (plan->batch > 0 && (!o_out || !lse_out || !aligned(o_out, 16) || !aligned(lse_out, 4)))
    return PD_ERR_INVALID_ARG;
  // stage 1 writes only the workspace for a partial plan; its `out` is not touched
  pd_status st = stage1(plan, q, k_pool, v_pool, nullptr, nullptr, block_tables, seq_lens, 0, scale, workspace,
                        workspace_bytes, o_out, stream);
  if (st != PD_OK || plan->batch == 0) return st;
  return merge_workspace(plan, static_cast<const uint8_t*>(workspace), nullptr, o_out, lse_out, stream);
}

pd_status paged_decode_combine(int32_t num_parts, int32_t rows, int32_t head_dim, const float* o_parts,
                               const float* lse_parts, void* out, void* stream) {
  if (num_parts < 1 || num_parts > 1024 || rows < 0 || head_dim <= 0 || head_dim % 4 != 0) return PD_ERR_INVALID_ARG;
  if (rows == 0) return PD_OK;
  if (!o_parts || !lse_parts || !out || !aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(out, 8))
    return PD_ERR_INVALID_ARG;
  pd::MergeParams p = {};
  p.lse_part = lse_parts;
  p.o_part = o_parts;
  p.row_stride = head_dim;
  p.piece_stride = (int64_t)rows * head_dim;
  p.lse_row_stride = 1;
  p.lse_piece_stride = rows;
  p.out = out;
  p.num_splits = num_parts;
  p.head_dim = head_dim;
  if (pd::launch_merge(p, rows, stream) != 0) return PD_ERR_CUDA;
  return PD_OK;
}

pd_status paged_decode_check_device_error(const pd_plan* plan, void* workspace, size_t workspace_bytes,
                                          void* stream, uint32_t* flags) {
  (void)plan;
  if (!workspace || workspace_bytes < sizeof(uint32_t)) return PD_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PD_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return PD_ERR_CUDA;
  if (flags) *flags = word;
  if (word != 0) {
    if (cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess) return PD_ERR_CUDA;
    return PD_ERR_DEVICE_FAULT;
  }
  return PD_OK;
}

}  // extern "C"
