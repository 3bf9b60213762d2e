/*
 * paged_decode.h — C ABI of the GB300 (sm_103a) paged GQA decode-attention library.
 *
 * One new query token per request attends over that request's cached keys and
 * values, which live in fixed-size pages of a per-layer pool and are found
 * through a block table. Both kinds of attention layer of a Gemma-4-style
 * model are served:
 *   - global layers (every cached token is attended; head_dim 512 in Gemma 4),
 *     optionally with one tensor used as both K and V ("K=V" storage);
 *   - sliding-window layers (only the last `window` tokens; head_dim 256),
 * each with its own query/KV head counts, query heads grouped on KV heads (GQA).
 *
 * Sources (page title, section):
 *   [PR27-text] Sparse-vLLM PR #27 "feat: support Gemma 4 and native multimodal
 *               inference", section "Gemma 4 文本推理" (text inference):
 *               heterogeneous sliding/global layers with their own head_dim and
 *               KV-head count, K=V or K!=V storage, per-layer KV storage.
 *   [PR27-ops]  same page, section "专用算子与性能优化" (dedicated operators and
 *               performance): a stage-1 decode pass for head_dim 512 that serves
 *               several GQA query heads of one KV head per program; grouped
 *               sliding-window and global decode; window starts that are not
 *               32-token aligned.
 *   [vLLM-attn] "模型库与算子层 — 概念" (vLLM model library & operator layer,
 *               concepts), section "注意力层" (attention layer): decode is the
 *               single-token incremental attention; paged KV cache with logical
 *               layout [L, B, H, N, C]; block sizes are multiples of 16.
 *   [vLLM-MLA]  same page, section "MLA 与 Sparse MLA（DSA）": split-KV decode —
 *               the KV sequence is cut into num_kv_splits pieces whose partial
 *               results carry a log-sum-exp and are merged afterwards; the partial
 *               buffer is reserved once for the worst case so no call allocates
 *               and CUDA-graph capture works.
 *
 * Data layout (all device pointers, row-major, contiguous, 16-byte aligned):
 *   q            bf16  [batch, num_q_heads, head_dim]
 *   k_pool       bf16  [num_pages, num_kv_heads, page_size, head_dim]
 *                      (FP8 layers: e4m3 bytes, plus fp32 scales [num_pages, num_kv_heads])
 *   v_pool       bf16  same shape as k_pool; NULL or == k_pool iff kv_shared
 *   block_tables int32 [batch, max_pages_per_seq]; entry i of request b is the
 *                      pool page holding its tokens [i*page_size, (i+1)*page_size)
 *   seq_lens     int32 [batch]; cached tokens of each request, INCLUDING the new
 *                      token (whose K/V the caller has already written)
 *   out          bf16  [batch, num_q_heads, head_dim]
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).
 * The attended positions of request b are [0, L) on a global layer and
 * [max(0, L - window), L) on a window layer (exactly the last `window` tokens,
 * the current one included); an empty range gives a zero output row.
 *
 * Ownership: the caller allocates and owns every buffer (inputs, the workspace
 * and out). The library allocates and frees nothing, keeps no state between
 * calls, and never synchronises except in paged_decode_check_device_error.
 * Every launch is ordered on the given stream (a cudaStream_t passed as void*;
 * NULL = the legacy default stream). The kernels go out as programmatic
 * dependents (they may become resident while the kernel before them drains,
 * and wait for it before touching what it may write; see pd_plan.early_kv for
 * the one exception a caller can opt into), and each lets the launch behind it
 * start early: a caller's kernel launched behind one of them with
 * programmatic stream serialisation must wait for it (griddepcontrol.wait,
 * cudaGridDependencySynchronize) before reading its output. Kernels launched
 * without that attribute, copies and events are ordered as usual.
 *
 * Errors: no exception or trap crosses this boundary. Host-side argument checks
 * return a status without launching anything. Conditions only the GPU can see
 * (a block-table entry outside the pool, a device seq_len outside
 * [0, max_pages_per_seq * page_size], a pipeline wait that timed out) set bits in
 * an error word at the start of the workspace: the offending page is skipped
 * (its tokens are masked out), the length clamped; paged_decode_check_device_error
 * reports PD_ERR_DEVICE_FAULT. The error word must be zero before the first
 * call: zero the workspace once after allocating it. Calls that share a
 * workspace must not overlap on the GPU: order them on one stream.
 */
#ifndef PAGED_DECODE_H
#define PAGED_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PD_OK = 0,
  PD_ERR_INVALID_ARG = 1,          /* bad pointer, shape, length or scale */
  PD_ERR_UNSUPPORTED = 2,          /* valid but not built: head_dim / group size */
  PD_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < plan->workspace_bytes */
  PD_ERR_CUDA = 4,                 /* a CUDA runtime call failed */
  PD_ERR_DEVICE_FAULT = 5          /* the device error word is non-zero */
} pd_status;

/* Bits of the device error word (paged_decode_check_device_error, *flags). */
#define PD_DEVFLAG_BAD_PAGE 0x1u     /* a block-table entry outside [0, num_pages) */
#define PD_DEVFLAG_BAD_SEQLEN 0x2u   /* a device seq_len outside the block table */
#define PD_DEVFLAG_WAIT_TIMEOUT 0x4u /* a pipeline wait gave up after ~1 s */

/* Element type of the KV cache (pd_layer_desc.kv_dtype). */
#define PD_KV_BF16 0      /* bf16 K/V rows */
#define PD_KV_FP8_E4M3 1  /* OCP e4m3 bytes; the value is byte * scale[page, KV head] */

/* One attention layer's shape. */
typedef struct {
  int32_t num_q_heads;        /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;       /* Hkv */
  int32_t head_dim;           /* d: 256 or 512 (128: bf16 cache, one query token) */
  int32_t page_size;          /* P: tokens per page, a multiple of 16 */
  int32_t num_pages;          /* pages in the pool */
  int32_t max_pages_per_seq;  /* block-table row length */
  int32_t window;             /* 0 = global layer; > 0 = sliding window of this many tokens */
  int32_t kv_shared;          /* 1 = one pool is both K and V (K=V storage) */
  int32_t kv_dtype;           /* PD_KV_BF16 or PD_KV_FP8_E4M3 */
} pd_layer_desc;

/* Launch plan: a plain value filled by paged_decode_plan, copyable, reusable for
 * any call with the same layer, batch and no longer sequences than it was made
 * for. Callers read workspace_bytes and num_splits; the other fields are the
 * library's. Every launch call checks the fields against one another first (the
 * grid against the pieces and batch, the workspace offsets and size against
 * what the launches write) and returns PD_ERR_INVALID_ARG for a plan that no
 * longer agrees with itself, before any CUDA call. */
typedef struct {
  pd_layer_desc layer;
  int32_t batch;
  int32_t num_splits;       /* S: KV pieces per (request, KV head); 1 = no merge needed */
  int32_t chunk_tokens;     /* tokens per piece */
  int32_t block_tokens;     /* tokens per pipeline stage */
  int32_t variant;          /* kernel instance */
  int32_t grid_x, grid_y, grid_z;
  int32_t threads_per_cta;
  int32_t smem_bytes;
  int32_t sm_count;
  int32_t max_seq_len;      /* longest sequence the plan was made for */
  int32_t merge_mode;       /* 0: S = 1, stage 1 writes out and there is nothing to merge;
                               1: paged_decode_merge launches the merge;
                               2: 2 <= S <= 8, stage 1 runs each (request, KV head)'s pieces as
                                  one thread-block cluster that merges them and writes out */
  int32_t test_stall_bytes;  /* 0. Tests set it > 0 to make stage 1 expect more bytes per stage
                                than its copies deliver, so its pipeline waits run out (~1 s) and
                                report PD_DEVFLAG_WAIT_TIMEOUT without any fault */
  int32_t query_tokens;     /* T: query tokens per request (1 = decode; > 1 = paged_decode_plan_multi) */
  int32_t partial;          /* 1: made by paged_decode_plan_partial (fp32 pieces always left for a merge) */
  int32_t early_kv;         /* 0 (as planned). A caller may set 1 when no kernel that can still be
                               running as stage 1 starts writes block_tables, seq_lens, the FP8 scales
                               or a cached row other than each request's newest query_tokens positions.
                               Those kernels are the one launched just before stage 1 on its stream and,
                               if that one lets its dependents start before it waits for its own
                               predecessor (paged_decode_qkv_norm_rope_write does), the one before it,
                               and so on; this library's decode and merge kernels let them start only
                               after that wait. A decode behind the new-token step, or behind another
                               layer's decode, qualifies. Stage 1 then copies the older rows of its first
                               pipeline stages while those kernels run (programmatic dependent launch);
                               q, the newest rows and every write (the device error word included)
                               wait for them as usual */
  uint64_t workspace_bytes; /* bytes the caller must provide */
  uint64_t lse_offset;      /* byte offset of the fp32 [batch, T, Hq, S] log-sum-exp part */
  uint64_t opart_offset;    /* byte offset of the fp32 [batch, T, Hq, S, d] partial outputs */
  uint32_t magic;
  uint32_t version;
} pd_plan;

/*
 * Choose the split count and launch shape for one decode step of one layer
 * ([vLLM-MLA]: split-KV with a worst-case-sized partial buffer; [PR27-ops]: the
 * stage-1 pass). Pure host function: no CUDA call.
 *   layer         the layer shape; window and kv_shared included
 *   batch         number of requests (>= 0)
 *   seq_lens_host host array [batch] of sequence lengths, each in
 *                 [0, max_pages_per_seq * page_size] — the plan stays valid for any
 *                 later call whose lengths do not exceed max(seq_lens_host)
 *   sm_count      streaming multiprocessors of the target GPU (> 0)
 *   plan          output
 * Groups (Hq / Hkv) of 1..16 are served: 1, 2, 4 and 8 by one CTA per
 * (request, KV head, piece) that reads each KV byte once for all query heads;
 * the others by CTAs of 8-column tiles of query heads (3, 5, 6, 7: one tile;
 * 9..16: two, a CTA each over short contexts, one CTA for both over long ones;
 * head_dim 256 or 512 -- at head_dim 128 only 1, 2, 4 and 8).
 * Returns PD_ERR_INVALID_ARG for a malformed shape or length, PD_ERR_UNSUPPORTED
 * for a head_dim or group size no kernel instance of the library serves (group > 16).
 */
pd_status paged_decode_plan(const pd_layer_desc* layer, int32_t batch, const int32_t* seq_lens_host,
                            int32_t sm_count, pd_plan* plan);

/*
 * Plan for several new tokens per request: speculative-decode verification or
 * a chunk of prefill over the paged cache (Sparse-vLLM PR #27, section
 * "专用算子与性能优化", reuses a paged prefill plan next to decode; the vLLM
 * concepts page, section "MLA 与 Sparse MLA（DSA）", lists causal multi-token
 * verification over a paged cache). Request b's T query tokens are its last T
 * cached positions (their K/V already written; seq_lens counts them); token j
 * at position L_b - T + j attends causally: positions up to its own, and on a
 * window layer only the last `window` of them (its own included) -- for each
 * token, exactly the decode of that token at length L_b - T + 1 + j.
 *   query_tokens  T, 1..256 (T = 1 is paged_decode_plan)
 *   seq_lens_host each in [T, max_pages_per_seq * page_size]
 *   other arguments as for paged_decode_plan
 * With such a plan, paged_decode_global / paged_decode_window /
 * paged_decode_merge / paged_decode_noalloc take q and out as bf16
 * [batch, T, Hq, d]; a device length below T sets PD_DEVFLAG_BAD_SEQLEN and the
 * tokens before position 0 attend nothing (zero output). The (token, head)
 * pairs of one KV head are served 8 per CTA, so for T * group <= 8 every KV
 * byte is still read once. bf16 or FP8 caches (an FP8 plan goes with
 * paged_decode_global_fp8 / paged_decode_window_fp8), head_dim 256 or 512,
 * group Hq / Hkv up to 16.
 */
pd_status paged_decode_plan_multi(const pd_layer_desc* layer, int32_t batch, int32_t query_tokens,
                                  const int32_t* seq_lens_host, int32_t sm_count, pd_plan* plan);

/*
 * Stage 1 on a global layer (plan->layer.window == 0): for every (request,
 * KV head, KV piece) one CTA streams the piece's pages once and serves all
 * query heads of that KV head ([PR27-ops] grouped decode, [vLLM-attn] decode).
 * With plan->num_splits == 1 it writes `out` directly; otherwise it writes the
 * partial outputs and log-sum-exps into the workspace and paged_decode_merge
 * must follow on the same stream.
 *   scale     softmax scale applied to q.k (finite, usually 1/sqrt(head_dim))
 *   workspace device buffer of at least plan->workspace_bytes, 256-byte aligned
 * Returns PD_ERR_INVALID_ARG (NULL/misaligned pointer, v_pool inconsistent with
 * kv_shared, non-finite scale, window layer), PD_ERR_WORKSPACE_TOO_SMALL,
 * PD_ERR_CUDA (launch failure).
 */
pd_status paged_decode_global(const pd_plan* plan, const void* q, const void* k_pool,
                              const void* v_pool, const int32_t* block_tables,
                              const int32_t* seq_lens, float scale, void* workspace,
                              size_t workspace_bytes, void* out, void* stream);

/*
 * Stage 1 on a sliding-window layer: as paged_decode_global, attending only
 * the last `window` positions of each request; pages wholly before the window
 * are never read, and the window may start at any token offset ([PR27-ops]:
 * window starts need no 32-token alignment). `window` must equal
 * plan->layer.window (> 0).
 */
pd_status paged_decode_window(const pd_plan* plan, const void* q, const void* k_pool,
                              const void* v_pool, const int32_t* block_tables,
                              const int32_t* seq_lens, int32_t window, float scale,
                              void* workspace, size_t workspace_bytes, void* out, void* stream);

/*
 * Stage 1 over an FP8 KV cache (plan->layer.kv_dtype == PD_KV_FP8_E4M3): as
 * paged_decode_global / paged_decode_window, with k_pool / v_pool holding OCP
 * e4m3 bytes [num_pages, Hkv, P, head_dim] and k_scale / v_scale fp32
 * [num_pages, Hkv]: the cached value of an element is its e4m3 value times the
 * scale of its (page, KV head). For a K=V layer v_pool and v_scale are NULL or
 * equal to k_pool and k_scale. q stays bf16 (it is rounded once to f16 for the
 * tensor cores; |q| must stay below 65504). window = 0 on a global layer.
 * FP8 KV caches halve the bytes of this bandwidth-bound pass; the vLLM
 * concepts page records FP8 KV-cache support in Blackwell attention backends
 * (sections "JIT 预热基础设施" and "MLA 与 Sparse MLA（DSA）"). Errors as for the
 * bf16 calls; a bf16 plan is rejected with PD_ERR_INVALID_ARG.
 */
pd_status paged_decode_global_fp8(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                                  const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                  const int32_t* seq_lens, float scale, void* workspace, size_t workspace_bytes,
                                  void* out, void* stream);
pd_status paged_decode_window_fp8(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                                  const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                  const int32_t* seq_lens, int32_t window, float scale, void* workspace,
                                  size_t workspace_bytes, void* out, void* stream);

/*
 * Stage 2 ([vLLM-MLA]: the pieces' partial results are merged): for each
 * (request, query head), out = sum_s w_s o_s / sum_s w_s with
 * w_s = exp(lse_s - max lse); pieces with no attended token weigh nothing; a
 * row with none at all is zero. The launch may start while stage 1 is still
 * running (programmatic dependent launch) and waits for it before reading the
 * partials. With plan->merge_mode 0 (one piece) there is nothing to merge and
 * with mode 2 stage 1 merged the pieces itself: it returns PD_OK without
 * launching, so it is always safe to call after stage 1.
 */
pd_status paged_decode_merge(const pd_plan* plan, const void* workspace, size_t workspace_bytes,
                             void* out, void* stream);

/*
 * Synchronise `stream`, read the device error word of `workspace`, store it in
 * *flags (may be NULL) and reset it to zero. Returns PD_ERR_DEVICE_FAULT if it
 * was non-zero, PD_ERR_CUDA if the synchronisation or copy failed.
 */
pd_status paged_decode_check_device_error(const pd_plan* plan, void* workspace,
                                          size_t workspace_bytes, void* stream, uint32_t* flags);

/*
 * One decode layer-step (stage 1, then the merge) for callers that cannot
 * allocate device memory. The source pages have no counterpart to this entry
 * point; it exists for callers such as a plugin inside an inference engine that
 * owns all device memory, or a serving loop that must not call cudaMalloc (which
 * can synchronise the device) mid-step. Instead of a caller-provided workspace
 * it uses an 8 MiB scratch array compiled into the library, which every GPU that
 * loads the library holds until the process exits.
 *   plan, q, k_pool, v_pool, block_tables, seq_lens, scale, out: as for
 *                 paged_decode_global / paged_decode_window
 *   window        0 on a global layer, else plan->layer.window
 *   device_flags  optional device pointer: receives the device error word
 *                 (PD_DEVFLAG_*) of this call; NULL to ignore it
 *   stream        cudaStream_t as void*
 * Every argument is checked before anything is queued: PD_ERR_INVALID_ARG for
 * what paged_decode_global / paged_decode_window refuse, and for an FP8 plan
 * (its scales have no argument here) or a plan from paged_decode_plan_partial;
 * PD_ERR_WORKSPACE_TOO_SMALL when the plan needs more than 8 MiB of scratch
 * (plan->workspace_bytes > 8 MiB). With batch 0 nothing is launched and
 * device_flags is not written. Otherwise it returns the statuses of the calls
 * it makes. The array has one device address per CUDA context; the first call
 * in a context (the device's primary context, another context made current by
 * the caller, or a primary context made again after cudaDeviceReset) looks it
 * up, so make that call before any stream capture. All calls share the one
 * array and each starts by clearing its error word: calls that overlap on the
 * GPU race, so order them on one stream. It allocates nothing.
 */
pd_status paged_decode_noalloc(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens, int32_t window, float scale,
                               void* out, uint32_t* device_flags, void* stream);

/* ---- Sequence-sharded decode: partial results and their combine ----------------
 *
 * Decode context parallelism (vLLM concepts page "模型库与算子层 — 概念", sections
 * on the MLA backends: DCP, an all-gather of each rank's partial outputs and
 * log-sum-exps ahead of the merge): the cached tokens of every request are
 * spread over R ranks, each rank attends its own tokens and produces a
 * normalised fp32 partial output plus its log-sum-exp, the ranks exchange
 * them (an all-gather, the caller's collective), and every rank merges the R
 * partials. The split of one request's tokens over several pieces inside a
 * rank and the merge across ranks are the same log-sum-exp arithmetic.
 */

/*
 * Plan for paged_decode_global_partial: as paged_decode_plan for a global bf16
 * layer (window 0; PD_ERR_UNSUPPORTED otherwise), with fp32 pieces always left
 * in the workspace (no in-cluster merge).
 */
pd_status paged_decode_plan_partial(const pd_layer_desc* layer, int32_t batch, const int32_t* seq_lens_host,
                                    int32_t sm_count, pd_plan* plan);

/*
 * This rank's part of a sharded decode: attention of q over the tokens of this
 * rank's cache (k_pool, v_pool, block_tables, seq_lens describe the local
 * tokens, as for paged_decode_global), written as
 *   o_out   device fp32 [batch, Hq, d]: the normalised partial output,
 *   lse_out device fp32 [batch, Hq]: its natural-log log-sum-exp (-inf and a
 *           zero row where the rank holds no token of the request).
 * plan from paged_decode_plan_partial; o_out 16-byte aligned. Errors as for
 * paged_decode_global.
 */
pd_status paged_decode_global_partial(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                                      const int32_t* block_tables, const int32_t* seq_lens, float scale,
                                      void* workspace, size_t workspace_bytes, float* o_out, float* lse_out,
                                      void* stream);

/*
 * Merge num_parts partial results of the same rows (one per rank, gathered):
 *   o_parts   device fp32 [num_parts, rows, head_dim] (16-byte aligned)
 *   lse_parts device fp32 [num_parts, rows]
 *   out       device bf16 [rows, head_dim]
 * out = sum_r w_r o_r, w_r = exp(lse_r - M) / sum_r' exp(lse_r' - M), M =
 * max_r lse_r; parts with lse = -inf weigh nothing (a row with none is zero).
 * num_parts 1..1024, head_dim a multiple of 4. Returns PD_ERR_INVALID_ARG for a
 * bad argument, PD_ERR_CUDA if the launch fails.
 */
pd_status paged_decode_combine(int32_t num_parts, int32_t rows, int32_t head_dim, const float* o_parts,
                               const float* lse_parts, void* out, void* stream);

/* ---- The step before decode: QKV norm, RoPE, paged-cache write -----------------
 *
 * Gemma 4 layers normalise the new token's q, k and v per head and apply RoPE
 * to q and k with the layer's own parameters (sliding-window and global layers
 * differ); the normalised, rotated k and the normalised v then go into the
 * paged cache (Sparse-vLLM PR #27 "feat: support Gemma 4 and native multimodal
 * inference", sections "Gemma 4 文本推理" and "专用算子与性能优化"; the vLLM
 * concepts page "模型库与算子层 — 概念" describes folding norm / RoPE into the
 * paged KV-cache write). One launch does all three for a batch of new tokens.
 */

/*
 * Fill a layer's RoPE table: cos_sin[p * rotary_dim + i] = cos(p * f_i) and
 * cos_sin[p * rotary_dim + rotary_dim/2 + i] = sin(p * f_i), with
 * f_i = theta^(-2i / rotary_dim), for p < num_positions and i < rotary_dim / 2.
 * The angles and their sine / cosine are evaluated in fp64 and rounded to fp32.
 *   theta          RoPE base (> 0, finite)
 *   rotary_dim     even, 2..512
 *   num_positions  rows of the table (>= 1)
 *   cos_sin        device fp32 [num_positions, rotary_dim], caller-owned
 *   stream         cudaStream_t as void*
 * Once per layer kind, before the first paged_decode_qkv_norm_rope_write.
 * Returns PD_ERR_INVALID_ARG for a bad argument, PD_ERR_CUDA if the launch fails.
 */
pd_status paged_decode_rope_table(double theta, int32_t rotary_dim, int32_t num_positions, float* cos_sin,
                                  void* stream);

/*
 * For every request b, with pos = seq_lens[b] - 1 (the new token's position;
 * seq_lens counts it, as in decode):
 *   q_out[b, h]                    = rope(norm(q_in[b, h], q_norm_weight), pos)
 *   k_pool[page, g, pos % P, :]    = rope(norm(k_in[b, g], k_norm_weight), pos)
 *   v_pool[page, g, pos % P, :]    = norm(v_in[b, g], v_norm_weight)   (K != V layers)
 * with page = block_tables[b][pos / P], norm(x, w)_i = x_i / sqrt(mean(x^2) +
 * eps) * w_i (a model that scales by 1 + w passes 1 + w), and rope turning the
 * pairs (i, i + rotary_dim/2), i < rotary_dim/2, by the angles of table row
 * pos: (y_i, y_j) -> (y_i cos - y_j sin, y_j cos + y_i sin); dims past
 * rotary_dim pass through. Arithmetic in fp32, results rounded once to bf16.
 *   layer          the decode layer descriptor (bf16 cache only: an FP8 cache
 *                  keeps one scale per page, which a single appended row
 *                  cannot set -> PD_ERR_UNSUPPORTED; head_dim 256 or 512)
 *   batch          requests (0: nothing is launched)
 *   rotary_dim     even, 0..head_dim (0: no rotation, cos_sin may be NULL)
 *   num_positions  rows of cos_sin
 *   eps            >= 0, finite
 *   q_in           device bf16 [batch, Hq, d]
 *   k_in, v_in     device bf16 [batch, Hkv, d]; v_in unused (may be NULL) when
 *                  layer->kv_shared (the cached row is the rotated k)
 *   q_norm_weight, k_norm_weight  device bf16 [d]
 *   v_norm_weight  device bf16 [d], or NULL for unit weights
 *   cos_sin        device fp32 [num_positions, rotary_dim] (paged_decode_rope_table)
 *   block_tables, seq_lens: as for decode
 *   q_out          device bf16 [batch, Hq, d] (the decode call's q)
 *   k_pool, v_pool device bf16 pools [num_pages, Hkv, P, d]; v_pool unused when
 *                  layer->kv_shared
 *   device_flags   device uint32 word, caller-owned and zeroed by the caller;
 *                  PD_DEVFLAG_BAD_SEQLEN is or-ed in (and nothing of that
 *                  request is written) when seq_lens[b] is outside
 *                  [1, max_pages * P] or pos >= num_positions while rotating;
 *                  PD_DEVFLAG_BAD_PAGE (and the cache rows are not written,
 *                  q_out is) when the page id is outside the pool
 *   stream         cudaStream_t as void*
 * q_in / k_in / v_in / q_out / pools must be 16-byte aligned. Only the new
 * token's rows of the pools are written. Requests must not share a slot.
 * Launched as a programmatic dependent that lets the kernel behind it start at
 * once, before it waits for the kernel before it: a decode with
 * pd_plan.early_kv behind it streams its older rows meanwhile (a kernel behind
 * it that reads what this one writes must wait for it, griddepcontrol.wait).
 * Returns PD_ERR_INVALID_ARG / PD_ERR_UNSUPPORTED without launching, PD_ERR_CUDA
 * if the launch fails.
 */
pd_status paged_decode_qkv_norm_rope_write(const pd_layer_desc* layer, int32_t batch, int32_t rotary_dim,
                                           int32_t num_positions, float eps, const void* q_in, const void* k_in,
                                           const void* v_in, const void* q_norm_weight, const void* k_norm_weight,
                                           const void* v_norm_weight, const float* cos_sin,
                                           const int32_t* block_tables, const int32_t* seq_lens, void* q_out,
                                           void* k_pool, void* v_pool, uint32_t* device_flags, void* stream);

/* ---- Host-in/host-out decode loops ---------------------------------------------
 *
 * Not an operation of the decode method: plumbing for a caller whose inputs
 * (q, block table, lengths) come from, and whose results go to, page-locked
 * host memory every step. A step issued as memcpy + decode + memcpy, or with
 * its copies on other streams joined by event waits, ends the chain of
 * programmatic dependent launches at every copy, so the next stage 1 cannot
 * start while the step in front drains. This call copies as one kernel that
 * lets the launch behind it start at once.
 */
#define PD_MAX_STAGE_COPIES 4

typedef struct {
  void* dst;
  const void* src;
  size_t bytes;   /* a multiple of 16; 0: the entry is skipped (its pointers may be NULL) */
} pd_copy;

/*
 * Copies copies[0 .. num_copies) (num_copies 0..PD_MAX_STAGE_COPIES; the kernel
 * is launched even when nothing is copied):
 *   after_wait 0  the copies run, then the kernel waits for the launch in front
 *                 of it (griddepcontrol.wait), so it completes after that launch:
 *                 for data that nothing possibly still running writes or reads.
 *                 Possibly still running as it starts: the launch in front and,
 *                 if that one lets its dependents start before its own wait, the
 *                 one before it, and so on. This library's decode and merge
 *                 kernels let them start after their wait;
 *                 paged_decode_qkv_norm_rope_write and this copy before.
 *   after_wait 1  the kernel waits first: for data the launch in front writes
 *                 or, behind a launch that lets its dependents start before its
 *                 own wait, for anything that launch's predecessors touch
 *   stream        cudaStream_t as void*
 * Every pointer of a non-empty copy is device memory of the current device or
 * page-locked host memory (cudaHostAlloc / cudaHostRegister, reached through its
 * device address), 16-byte aligned; a copy's source and destination do not
 * overlap, nor do the copies of one call.
 *
 * A decode loop with one step of look-ahead for q: two q buffers and two result
 * buffers used alternately. Without pd_plan.early_kv: copy(step 0's inputs in,
 * 0); per step i: decode(i) [+ merge(i)], then copy(step i+1's inputs in, step
 * i-1's result out, 0); at the end copy(the last result out, 1). With
 * pd_plan.early_kv stage 1 reads its block table and lengths before its wait,
 * so the copy in front of it must not write them: the block table and lengths
 * go two steps ahead (three buffers), copied for steps 0 and 1 with an ordinary
 * copy before the loop and for step i+2 by step i's copy. A loop whose last
 * kernel of a step lets its dependents start before its own wait
 * (paged_decode_qkv_norm_rope_write alone) copies after it with after_wait 1:
 * the next step's inputs in and that step's own result out.
 *
 * Returns PD_ERR_INVALID_ARG without launching (pageable or foreign memory,
 * misalignment, a size off 16, overlap, more than PD_MAX_STAGE_COPIES copies,
 * after_wait not 0 or 1), PD_ERR_CUDA if the launch fails.
 */
pd_status paged_decode_stage_copy(const pd_copy* copies, int32_t num_copies, int32_t after_wait, void* stream);

/* Static, human-readable name of a status. */
const char* paged_decode_status_string(pd_status status);

/* ABI version of this library (bumped when pd_plan or a signature changes). */
int32_t paged_decode_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_DECODE_H */
