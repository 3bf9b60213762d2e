// Host-side planner of the paged decode library: argument validation, the
// choice of kernel instance, the KV split count and the workspace size.
// Pure host code: no CUDA call.
//
// Split-KV with a worst-case-sized partial buffer follows the vLLM concepts page
// "模型库与算子层 — 概念", section "MLA 与 Sparse MLA（DSA）" (num_kv_splits pieces,
// partial results plus log-sum-exp, the buffer reserved up front). The split
// count itself is this library's own choice: the pages give no rule for it.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <deque>
#include <queue>
#include <vector>

#include "paged_decode.h"
#include "pd_kernels.h"

namespace pd {

#define PD_VARIANT_ROW(ID, D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW)                                         \
  VariantInfo{ID,                                                                                         \
              D,                                                                                          \
              G,                                                                                          \
              KVS ? 1 : 0,                                                                                \
              KV8 ? 1 : 0,                                                                                \
              NW,                                                                                         \
              SPW,                                                                                        \
              Stage1Cfg<D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW>::TB,                                        \
              Stage1Cfg<D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW>::THREADS,                                   \
              Stage1Cfg<D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW>::SMEM_BYTES,                                \
              Stage1Cfg<D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW>::MAX_CLUSTER,                               \
              MQ ? 1 : 0,                                                                                 \
              Stage1Cfg<D, G, KVS, KV8, NW, SPW, MQ, NSUB, TW>::DED_SLOTS,                                 \
              NSUB,                                                                                       \
              TW},
const VariantInfo kVariants[] = {PD_FOR_EACH_VARIANT(PD_VARIANT_ROW)};
#undef PD_VARIANT_ROW
const int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

}  // namespace pd

namespace {

constexpr uint32_t kPlanMagic = 0x50444543u;  // "PDEC"
constexpr int32_t kAbiVersion = 5;
// Pieces per (request, KV head) are capped at what the merge kernel takes
// (and far above what the cost model ever picks: a few waves of the GPU).
constexpr int kMaxSplits = 1024;

// Query tokens per request a plan may carry (multi-token variants).
constexpr int kMaxQueryTokens = 256;

// Largest GQA group (query heads per KV head) a plan accepts.
constexpr int kMaxGroup = 16;

// Decode (one query token) with a group of 1, 2, 4 or 8: the instance of
// exactly this group. Several query tokens, or any other group up to
// kMaxGroup (3, 5..7, 9..16): the column-tiled instance (CTAs of 8 columns of
// (token, head) pairs), which takes the group at run time.
bool tiled(int query_tokens, int group) { return query_tokens > 1 || group > 8 || (group & (group - 1)) != 0; }

// Column-tiled plans with more than one 8-column tile use, over a bf16 cache,
// the instances whose CTA serves two tiles from one ring (one copy of every
// block for both); other plans those with one tile per CTA.
// Where two instances serve the same shape (the FP8 K != V decode ones, with
// seven and with six consumer warps), `nw` > 0 asks for that many warps; 0
// takes the first in the table.
const pd::VariantInfo* find_variant(int head_dim, int group, int kv_shared, int kv_fp8, int multi, int tiles,
                                    int nw = 0) {
  if (group < 1 || group > kMaxGroup) return nullptr;
  for (int i = 0; i < pd::kNumVariants; ++i) {
    const pd::VariantInfo& v = pd::kVariants[i];
    if (v.head_dim != head_dim || v.kv_shared != kv_shared || v.kv_fp8 != kv_fp8 || v.multi != multi) continue;
    if (v.tiles != tiles || (nw > 0 && v.nw != nw)) continue;
    if (multi || v.group == group) return &v;
  }
  return nullptr;
}

// 8-column tiles of a column-tiled plan: its T x group (token, head) pairs, 8 at a time.
int col_tiles(int query_tokens, int group) { return (query_tokens * group + 7) / 8; }

// CTAs per (KV head, piece) of a plan on instance v.
int col_groups(const pd::VariantInfo& v, int query_tokens, int group) {
  return v.multi ? (col_tiles(query_tokens, group) + v.tiles - 1) / v.tiles : 1;
}

uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Cost model of one stage-1 launch, in microseconds. Units (a CTA, or a
// thread-block cluster of S CTAs) go to `slots` resident positions in launch
// order (split index fastest), each to the position that frees first. A CTA
// spends cta_fixed_us before its first bytes arrive (empty_cta_us if its range
// is empty), then streams its tokens. The n CTAs streaming at a moment share
//   agg(n) = ((n * cap)^-4 + hbm^-4)^(-1/4)   tokens / us
// equally: `cap` is what one CTA of the instance streams on its own (its ring
// latency or its per-block arithmetic, whichever binds), `hbm` the memory's
// rate; the smooth minimum fits the rates measured on a GB300 with 16, 32, 64,
// 96, 144 and 152 CTAs to a few percent. A unit ends `tail_us` after its last
// CTA. More than one piece adds the merge launch and its traffic (merge mode 1)
// or the in-cluster merge (mode 2).
struct CostModel {
  double cap_tok_per_us;  // one CTA alone
  double hbm_tok_per_us;  // all CTAs together
  double cta_fixed_us;    // launch, first copies in flight, epilogue
  double empty_cta_us;
  double merge_fixed_us;
  double merge_us_per_byte;
  double cluster_merge_us;
  int slots;                          // resident CTAs (one per SM: shared memory bound)
  std::vector<double> per_cta_rate;   // [n] = agg(n) / n, n = 0..slots
};

constexpr int kMaxClusterSplits = 8;

// Clusters of S CTAs (one CTA per SM, ~230 KB of shared memory each) resident
// at once on a 152-SM GB300, as cudaOccupancyMaxActiveClusters reports: the
// GPCs hold unequal numbers of SMs, so sizes 7 and 8 fit 15 clusters, not 16.
// Other SM counts scale it. Only the cost model uses it.
int cluster_slots(int splits, int sm_count) {
  static const int kGb300[kMaxClusterSplits + 1] = {0, 152, 76, 46, 36, 28, 23, 15, 15};
  if (splits < 1 || splits > kMaxClusterSplits) return 0;
  return (int)((long long)kGb300[splits] * sm_count / 152);
}

// Tokens per microsecond one stage-1 CTA streams when few CTAs run (measured
// on a GB300 with 16 CTAs over 2 x 65536 tokens, 4 KV heads): per (head_dim,
// K=V, FP8) for CTAs of one 8-column tile (decode, or query tokens and heads
// in one tile), and for bf16 CTAs of two tiles.
double cta_tokens_per_us(const pd::VariantInfo& v) {
  const bool kvs = v.kv_shared != 0;
  if (v.tiles == 2) {
    if (v.head_dim == 512) return kvs ? 48.5 : 47.2;
    return 67.0;  // d256 (K=V not measured: the K != V figure)
  }
  if (v.kv_fp8) {
    // (the six-warp K != V instances: the seven-warp figure scaled by 6 / 7)
    const double warps = v.nw == 6 ? 6.0 / 7.0 : 1.0;
    if (v.head_dim == 512) return kvs ? 85.1 : 49.4 * warps;
    return kvs ? 120.0 : 98.0 * warps;
  }
  if (v.head_dim == 512) return kvs ? 61.7 : 55.4;
  if (v.head_dim == 256) return kvs ? 90.5 : 74.6;
  return kvs ? 165.5 : 74.7;
}

// `tokens(u, i)`: unit u's CTA i's token count (<= 0: an empty range). Units
// start at non-decreasing times and every CTA's fixed phase (and an empty
// CTA's) has the same length, so the fixed phases, the empty CTAs and the
// slots freed each end in the order they began: three FIFO queues; only the
// streaming CTAs need a heap. Returns 1e300 as soon as the clock passes
// `limit` by more than rounding (a launch that long cannot be the one chosen).
template <class UnitTokens>
double simulate_fluid(long long num_units, int ctas_per_unit, const UnitTokens& tokens, int slots, double tail_us,
                      const CostModel& cm, double limit = 1e300) {
  struct Ev {
    double t;
    long long u;
    long long tok;
  };
  struct Stream {
    double v_end;  // service level (tokens per streaming CTA) at which it is done
    long long u;
    bool operator>(const Stream& o) const { return v_end > o.v_end; }
  };
  std::deque<Ev> fixed_q, empty_q;  // a CTA's fixed phase ends / an empty CTA ends
  std::deque<double> free_q;        // a slot frees
  std::priority_queue<Stream, std::vector<Stream>, std::greater<Stream>> streams;
  std::vector<int> left;  // CTAs of each started unit still running
  left.reserve((size_t)std::min<long long>(num_units, 1 << 20));
  long long next = 0;
  double t = 0.0, level = 0.0, makespan = 0.0;
  auto start_unit = [&](double at) {
    const long long u = next++;
    left.push_back(ctas_per_unit);
    for (int i = 0; i < ctas_per_unit; ++i) {
      const long long n = tokens(u, i);
      if (n > 0)
        fixed_q.push_back({at + cm.cta_fixed_us, u, n});
      else
        empty_q.push_back({at + cm.empty_cta_us, u, 0});
    }
  };
  auto cta_done = [&](long long u) {
    if (--left[(size_t)u] == 0) free_q.push_back(t + tail_us);
  };
  for (int s = 0; s < slots && next < num_units; ++s) start_unit(0.0);
  while (!fixed_q.empty() || !empty_q.empty() || !free_q.empty() || !streams.empty()) {
    if (t > limit * (1.0 + 1e-6)) return 1e300;
    const size_t n = streams.size();
    const double rate = n ? cm.per_cta_rate[std::min(n, cm.per_cta_rate.size() - 1)] : 0.0;
    const double t_stream = n ? t + (streams.top().v_end - level) / rate : 1e300;
    const double t_fixed = fixed_q.empty() ? 1e300 : fixed_q.front().t;
    const double t_empty = empty_q.empty() ? 1e300 : empty_q.front().t;
    const double t_free = free_q.empty() ? 1e300 : free_q.front();
    const double t_wall = std::min(t_fixed, std::min(t_empty, t_free));
    if (n && t_stream <= t_wall) {
      t = std::max(t, t_stream);
      level = streams.top().v_end;
      const long long u = streams.top().u;
      streams.pop();
      cta_done(u);
      continue;
    }
    if (n) level += rate * (t_wall - t);
    t = std::max(t, t_wall);
    if (t_wall == t_fixed) {
      streams.push({level + (double)fixed_q.front().tok, fixed_q.front().u});
      fixed_q.pop_front();
    } else if (t_wall == t_empty) {
      const long long u = empty_q.front().u;
      empty_q.pop_front();
      cta_done(u);
    } else {
      free_q.pop_front();
      makespan = std::max(makespan, t);
      if (next < num_units) start_unit(t);
    }
  }
  return makespan;
}

// Tokens of piece s of a request whose block-aligned span is n tokens (the
// last piece takes the remainder).
long long piece_tokens(int n, int chunk, int splits, int s) {
  const long long lo = (long long)s * chunk;
  return (s == splits - 1) ? n - lo : std::min<long long>(chunk, n - lo);
}

// One launch with a CTA per (request, KV head CTA, piece), then the merge launch.
double simulate(const std::vector<int>& n_tok, int hkv, int chunk, int splits, const CostModel& cm,
                uint64_t merge_bytes, double limit = 1e300) {
  const long long units = (long long)n_tok.size() * hkv * splits;
  auto tok = [&](long long u, int) {
    return piece_tokens(n_tok[(size_t)(u / ((long long)hkv * splits))], chunk, splits, (int)(u % splits));
  };
  const double merge_us = splits > 1 ? cm.merge_fixed_us + merge_bytes * cm.merge_us_per_byte : 0.0;
  const double makespan = simulate_fluid(units, 1, tok, cm.slots, 0.0, cm, limit - merge_us);
  return makespan >= 1e300 ? 1e300 : makespan + merge_us;
}

// The same launch with the S pieces of each (request, KV head) run as one
// thread-block cluster, merged in the cluster: only cluster_slots(S) clusters
// are resident at a time.
double simulate_clusters(const std::vector<int>& n_tok, int hkv, int chunk, int splits, const CostModel& cm,
                         double limit = 1e300) {
  const int cl_slots = cluster_slots(splits, cm.slots);
  if (cl_slots <= 0) return 1e300;
  const long long units = (long long)n_tok.size() * hkv;
  auto tok = [&](long long u, int i) { return piece_tokens(n_tok[(size_t)(u / hkv)], chunk, splits, i); };
  return simulate_fluid(units, splits, tok, cl_slots, cm.cluster_merge_us, cm, limit);
}

}  // namespace

namespace {
pd_status plan_impl(const pd_layer_desc* layer, int32_t batch, int32_t query_tokens, const int32_t* seq_lens_host,
                    int32_t sm_count, int partial, pd_plan* plan);
}

extern "C" {

int32_t paged_decode_abi_version(void) { return kAbiVersion; }

const char* paged_decode_status_string(pd_status status) {
  switch (status) {
    case PD_OK:
      return "ok";
    case PD_ERR_INVALID_ARG:
      return "invalid argument";
    case PD_ERR_UNSUPPORTED:
      return "unsupported head_dim / group size";
    case PD_ERR_WORKSPACE_TOO_SMALL:
      return "workspace too small";
    case PD_ERR_CUDA:
      return "CUDA runtime error";
    case PD_ERR_DEVICE_FAULT:
      return "device reported a bad page, a bad length or a timed-out wait";
  }
  return "unknown status";
}

pd_status paged_decode_plan(const pd_layer_desc* layer, int32_t batch, const int32_t* seq_lens_host,
                            int32_t sm_count, pd_plan* plan) {
  return paged_decode_plan_multi(layer, batch, 1, seq_lens_host, sm_count, plan);
}

pd_status paged_decode_plan_multi(const pd_layer_desc* layer, int32_t batch, int32_t query_tokens,
                                  const int32_t* seq_lens_host, int32_t sm_count, pd_plan* plan) {
  return plan_impl(layer, batch, query_tokens, seq_lens_host, sm_count, 0, plan);
}

pd_status paged_decode_plan_partial(const pd_layer_desc* layer, int32_t batch, const int32_t* seq_lens_host,
                                    int32_t sm_count, pd_plan* plan) {
  if (layer && (layer->window != 0 || layer->kv_dtype != PD_KV_BF16)) return PD_ERR_UNSUPPORTED;
  return plan_impl(layer, batch, 1, seq_lens_host, sm_count, 1, plan);
}

}  // extern "C"

namespace {

pd_status plan_impl(const pd_layer_desc* layer, int32_t batch, int32_t query_tokens, const int32_t* seq_lens_host,
                    int32_t sm_count, int partial, pd_plan* plan) {
  if (!layer || !plan) return PD_ERR_INVALID_ARG;
  if (query_tokens < 1 || query_tokens > kMaxQueryTokens) return PD_ERR_INVALID_ARG;
  const int T = query_tokens;
  const pd_layer_desc& ly = *layer;
  if (ly.num_q_heads <= 0 || ly.num_kv_heads <= 0 || ly.num_q_heads % ly.num_kv_heads != 0)
    return PD_ERR_INVALID_ARG;
  if (ly.head_dim <= 0 || ly.page_size <= 0 || ly.page_size % 16 != 0) return PD_ERR_INVALID_ARG;
  if (ly.num_pages <= 0 || ly.max_pages_per_seq <= 0 || ly.window < 0) return PD_ERR_INVALID_ARG;
  if (ly.kv_shared != 0 && ly.kv_shared != 1) return PD_ERR_INVALID_ARG;
  if (ly.kv_dtype != PD_KV_BF16 && ly.kv_dtype != PD_KV_FP8_E4M3) return PD_ERR_INVALID_ARG;
  if (batch < 0 || batch > 65535 || ly.num_kv_heads > 65535 || sm_count <= 0) return PD_ERR_INVALID_ARG;
  if (batch > 0 && !seq_lens_host) return PD_ERR_INVALID_ARG;
  const long long cap = (long long)ly.max_pages_per_seq * ly.page_size;
  if (cap > 0x7fffffffLL) return PD_ERR_INVALID_ARG;
  // pool rows are addressed with 32-bit TMA coordinates
  if ((long long)ly.num_pages * ly.num_kv_heads * ly.page_size > 0x7fffffffLL) return PD_ERR_UNSUPPORTED;
  int32_t max_len = 0;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens_host[b] < (T > 1 ? T : 0) || seq_lens_host[b] > cap) return PD_ERR_INVALID_ARG;
    max_len = std::max(max_len, seq_lens_host[b]);
  }
  const int group = ly.num_q_heads / ly.num_kv_heads;
  const bool multi = tiled(T, group);
  const bool fp8 = ly.kv_dtype == PD_KV_FP8_E4M3;
  // Two tiles per CTA read each block once for both; separate CTAs read it
  // once each, the second read an L2 hit when the context is short. Measured
  // (16 query / 4 KV heads, d 512): 4 tiles over 8 x 1024 tokens 22.1 us with
  // two tiles a CTA against 25.7 us; 2 tiles over 4 x 32768 tokens 165 us
  // against 192 us; 2 tiles over 8 x 1024 tokens 21.3 us against 20.2 us.
  int longest_span = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = seq_lens_host[b];
    const int first_hi = L - T + 1;
    const int lo = (ly.window > 0 && first_hi > ly.window) ? first_hi - ly.window : 0;
    longest_span = std::max(longest_span, L - lo);
  }
  const int tiles_needed = multi ? col_tiles(T, group) : 1;
  const int want_tiles = (multi && !fp8 && (tiles_needed >= 3 || (tiles_needed == 2 && longest_span >= 4096))) ? 2 : 1;
  // FP8 K != V decode over spans under 4096 tokens: the six-warp instance,
  // whose cluster merges need one barrier (same-box: 64 MiB 11.13 -> 10.39
  // us, windows of 1024 -1.6%); longer spans keep the seventh warp's
  // arithmetic (1 GiB: 84.1 us against 86.0 with six).
  const int want_nw = (fp8 && !ly.kv_shared && !multi && longest_span < 4096) ? 6 : 0;
  const pd::VariantInfo* v = find_variant(ly.head_dim, group, ly.kv_shared, fp8, multi, want_tiles, want_nw);
  if (!v && want_nw > 0) v = find_variant(ly.head_dim, group, ly.kv_shared, fp8, multi, want_tiles);
  if (!v && want_tiles > 1) v = find_variant(ly.head_dim, group, ly.kv_shared, fp8, multi, 1);
  if (!v) return PD_ERR_UNSUPPORTED;
  const int TB = v->block_tokens;
  // CTAs per (piece, KV head): one, or the column groups of a tiled plan
  const int groups = col_groups(*v, T, group);
  if ((long long)ly.num_kv_heads * groups > 65535) return PD_ERR_UNSUPPORTED;
  const int hkv_ctas = ly.num_kv_heads * groups;

  // block-aligned attended span of each request (several query tokens: the
  // union of their ranges, from the first token's window start)
  std::vector<int> n_tok(batch);
  int max_n = 0;
  long long total = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = seq_lens_host[b];
    const int first_hi = L - T + 1;
    const int lo = (ly.window > 0 && first_hi > ly.window) ? first_hi - ly.window : 0;
    n_tok[b] = L > 0 ? L - (lo / TB) * TB : 0;
    max_n = std::max(max_n, n_tok[b]);
    total += n_tok[b];
  }

  CostModel cm;
  const double kv_bytes_per_token =
      (double)ly.head_dim * (ly.kv_dtype == PD_KV_FP8_E4M3 ? 1.0 : 2.0) * (ly.kv_shared ? 1.0 : 2.0);
  // ~7.3 TB/s of HBM on a 152-SM GB300, in proportion for other SM counts
  cm.hbm_tok_per_us = 7.3e12 / 1e6 / kv_bytes_per_token * sm_count / 152.0;
  cm.cap_tok_per_us = cta_tokens_per_us(*v);
  cm.cta_fixed_us = 2.0;
  cm.empty_cta_us = 0.2;
  cm.merge_fixed_us = 2.0;
  cm.merge_us_per_byte = 1.0 / 7.0e6;
  cm.cluster_merge_us = 0.5;
  cm.slots = sm_count;  // one resident CTA per SM (shared memory bound)
  cm.per_cta_rate.assign((size_t)sm_count + 1, 0.0);
  for (int n = 1; n <= sm_count; ++n) {
    const double agg = std::pow(std::pow(n * cm.cap_tok_per_us, -4.0) + std::pow(cm.hbm_tok_per_us, -4.0), -0.25);
    cm.per_cta_rate[(size_t)n] = agg / n;
  }

  // pieces are whole stages where possible (a stage holds blocks_per_stage blocks)
  const uint64_t unit = 16ull * v->blocks_per_stage;
  int best_chunk = std::max(16, (int)align_up((uint64_t)std::max(max_n, 1), 16));
  int best_splits = 1;
  bool best_cluster = false;
  if (max_n > 0) {
    // candidates: multiples of 16 on a geometric grid, from the point where the
    // launch would need more than ~8 waves up to one piece per request
    const long long work = total * hkv_ctas;
    const int c_min = (int)std::max<long long>(64, align_up((uint64_t)(work / (8LL * cm.slots) + 1), unit));
    const int c_max = (int)align_up((uint64_t)max_n, 16);
    std::vector<int> cands;
    for (double c = c_min; c < c_max; c *= 1.08) cands.push_back((int)align_up((uint64_t)c, unit));
    for (int w = 1; w <= 8; ++w) {
      // pieces sized so B * Hkv * S lands on exactly w waves for the longest request
      const long long per_wave = (long long)w * cm.slots;
      const long long pairs = (long long)batch * hkv_ctas;
      const long long s = std::max<long long>(1, per_wave / std::max<long long>(1, pairs));
      cands.push_back((int)align_up((uint64_t)((max_n + s - 1) / s), unit));
    }
    cands.push_back(c_max);
    std::sort(cands.begin(), cands.end());
    cands.erase(std::unique(cands.begin(), cands.end()), cands.end());
    // A launch lasts at least as long as all its tokens take at the memory's
    // rate, and as its longest piece takes at one CTA's rate after the fixed
    // start (the model's shared rate is below both); a candidate whose bound
    // exceeds the best cost so far cannot be chosen, so it is not simulated.
    // The "exactly w waves" sizes, usually near the best, seed that cost.
    const double total_tok = (double)total * hkv_ctas;
    auto merge_bytes_of = [&](int s) {
      return (uint64_t)batch * T * ly.num_q_heads * s * (ly.head_dim + 1) * 4ull * 2ull;
    };
    auto stream_bound = [&](int c) {
      return std::max(total_tok / cm.hbm_tok_per_us, cm.cta_fixed_us + std::min(c, max_n) / cm.cap_tok_per_us);
    };
    // and, each CTA holding its slot for at least its fixed start plus its
    // tokens at one CTA's rate, at least the sum of those over the slots (a
    // cluster: its longest piece, and its merge)
    auto slot_bound = [&](int c, int s) {
      double direct = 0.0, clustered = 0.0;
      for (int b = 0; b < batch; ++b) {
        const int busy = n_tok[b] > 0 ? std::min(s, (n_tok[b] + c - 1) / c) : 0;
        direct += busy * cm.cta_fixed_us + (s - busy) * cm.empty_cta_us;
        clustered += (n_tok[b] > 0 ? cm.cta_fixed_us + std::min(c, n_tok[b]) / cm.cap_tok_per_us : cm.empty_cta_us) +
                     cm.cluster_merge_us;
      }
      direct = (direct * hkv_ctas + total_tok / cm.cap_tok_per_us) / cm.slots;
      const int cl_slots = cluster_slots(s, cm.slots);
      clustered = cl_slots > 0 ? clustered * hkv_ctas / cl_slots : 1e300;
      return std::make_pair(direct, clustered);
    };
    auto may_cluster = [&](int s) { return !partial && s >= 2 && s <= std::min(kMaxClusterSplits, v->max_cluster); };
    double best = 1e300;
    for (int w = 1; w <= 2; ++w) {
      const long long pairs = (long long)batch * hkv_ctas;
      const long long sw = std::max<long long>(1, (long long)w * cm.slots / std::max<long long>(1, pairs));
      const int c = (int)align_up((uint64_t)((max_n + sw - 1) / sw), unit);
      const int s = (max_n + c - 1) / c;
      if (c < 16 || s > kMaxSplits) continue;
      best = std::min(best, simulate(n_tok, hkv_ctas, c, s, cm, merge_bytes_of(s)));
      if (may_cluster(s)) best = std::min(best, simulate_clusters(n_tok, hkv_ctas, c, s, cm));
    }
    const double seed = best;
    best = 1e300;
    for (int c : cands) {
      if (c < 16) continue;
      const int s = (max_n + c - 1) / c;
      if (s > kMaxSplits) continue;
      const uint64_t merge_bytes = merge_bytes_of(s);
      const auto slots_b = slot_bound(c, s);
      const double merge_us = s > 1 ? cm.merge_fixed_us + merge_bytes * cm.merge_us_per_byte : 0.0;
      const double bound_direct = std::max(stream_bound(c), slots_b.first) + merge_us;
      const double bound_cluster = std::max(stream_bound(c) + cm.cluster_merge_us, slots_b.second);
      // (the margin keeps rounding from dropping a candidate that ties the best)
      const double limit = std::min(best, seed);
      const double prune_at = limit * (1.0 + 1e-6);
      const bool try_cluster = may_cluster(s) && bound_cluster <= prune_at;
      if (bound_direct > prune_at && !try_cluster) continue;
      double cost = bound_direct > prune_at ? 1e300 : simulate(n_tok, hkv_ctas, c, s, cm, merge_bytes, limit);
      bool cluster = false;
      if (try_cluster) {
        const double cc = simulate_clusters(n_tok, hkv_ctas, c, s, cm, limit);
        if (cc < cost) {
          cost = cc;
          cluster = true;
        }
      }
      if (cost < best * (1.0 - 1e-9) || (cost <= best && s < best_splits)) {
        best = cost;
        best_chunk = c;
        best_splits = s;
        best_cluster = cluster;
      }
    }
  }

  std::memset(plan, 0, sizeof(*plan));
  plan->layer = ly;
  plan->batch = batch;
  plan->num_splits = best_splits;
  plan->chunk_tokens = best_chunk;
  plan->block_tokens = TB;
  plan->variant = v->id;
  plan->grid_x = best_splits;
  plan->grid_y = hkv_ctas;
  plan->query_tokens = T;
  plan->grid_z = batch;
  plan->threads_per_cta = v->threads;
  plan->smem_bytes = v->smem_bytes;
  plan->sm_count = sm_count;
  plan->max_seq_len = max_len;
  const uint64_t rows = (uint64_t)batch * T * ly.num_q_heads;
  if (best_splits > 1 && best_cluster) {
    // merged inside each cluster: the workspace holds only the error word
    plan->merge_mode = 2;
    plan->lse_offset = pd::kWorkspaceHeader;
    plan->opart_offset = pd::kWorkspaceHeader;
    plan->workspace_bytes = pd::kWorkspaceHeader;
  } else if (best_splits > 1 || partial) {
    // (a partial plan always leaves fp32 pieces for the merge, even one)
    plan->merge_mode = 1;
    plan->lse_offset = pd::kWorkspaceHeader;
    plan->opart_offset = align_up(plan->lse_offset + rows * best_splits * 4ull, 256);
    plan->workspace_bytes = plan->opart_offset + rows * best_splits * (uint64_t)ly.head_dim * 4ull;
  } else {
    plan->merge_mode = 0;
    plan->lse_offset = pd::kWorkspaceHeader;
    plan->opart_offset = pd::kWorkspaceHeader;
    plan->workspace_bytes = pd::kWorkspaceHeader;
  }
  plan->partial = partial;
  plan->magic = kPlanMagic;
  plan->version = kAbiVersion;
  return PD_OK;
}

}  // namespace

namespace pd {

bool plan_is_valid(const pd_plan* plan) {
  if (!plan || plan->magic != kPlanMagic || plan->version != (uint32_t)kAbiVersion) return false;
  if (plan->variant < 0 || plan->variant >= kNumVariants) return false;
  const VariantInfo& v = kVariants[plan->variant];
  const pd_layer_desc& ly = plan->layer;
  if (ly.num_kv_heads <= 0 || ly.num_q_heads % ly.num_kv_heads != 0) return false;
  const int group = ly.num_q_heads / ly.num_kv_heads;
  if (v.multi) {
    if (group > kMaxGroup || plan->query_tokens < 1 || plan->query_tokens > kMaxQueryTokens) return false;
    if (!tiled(plan->query_tokens, group)) return false;
    if (plan->grid_y != ly.num_kv_heads * col_groups(v, plan->query_tokens, group)) return false;
  } else {
    if (group != v.group || plan->query_tokens != 1 || plan->grid_y != ly.num_kv_heads) return false;
  }
  if (ly.head_dim != v.head_dim || ly.kv_shared != v.kv_shared) return false;
  if ((ly.kv_dtype == PD_KV_FP8_E4M3) != (v.kv_fp8 == 1)) return false;
  if (plan->num_splits < 1 || plan->num_splits > kMaxSplits || plan->chunk_tokens < 16 || plan->chunk_tokens % 16 != 0)
    return false;
  if (plan->batch < 0 || plan->grid_x != plan->num_splits || plan->grid_z != plan->batch) return false;
  if (plan->block_tokens != v.block_tokens) return false;
  if (plan->threads_per_cta != v.threads || plan->smem_bytes != v.smem_bytes) return false;
  if (plan->merge_mode < 0 || plan->merge_mode > 2) return false;
  if (plan->test_stall_bytes < 0 || plan->test_stall_bytes > (1 << 16) || plan->test_stall_bytes % 16 != 0)
    return false;
  if (plan->partial != 0 && plan->partial != 1) return false;
  if (plan->early_kv != 0 && plan->early_kv != 1) return false;
  if (plan->partial ? (plan->merge_mode != 1 || plan->query_tokens != 1 || ly.window != 0)
                    : ((plan->num_splits == 1) != (plan->merge_mode == 0)))
    return false;
  if (plan->merge_mode == 2 && plan->num_splits > std::min(kMaxClusterSplits, v.max_cluster)) return false;
  // The workspace the plan asks for must hold what its launches write: the
  // error word, and in merge mode 1 the [rows][S] log-sum-exps and the
  // [rows][S][d] fp32 partials at their offsets (a plan edited by hand to more
  // pieces is refused here instead of writing past the caller's buffer).
  if (plan->workspace_bytes < pd::kWorkspaceHeader) return false;
  if (plan->merge_mode == 1) {
    if (plan->lse_offset < pd::kWorkspaceHeader || plan->lse_offset % 256 != 0 || plan->opart_offset % 256 != 0)
      return false;
    uint64_t lse_bytes = 0, opart_bytes = 0, lse_end = 0, opart_end = 0;
    const uint64_t rows = (uint64_t)plan->batch * (uint64_t)plan->query_tokens * (uint64_t)ly.num_q_heads;
    if (__builtin_mul_overflow(rows, (uint64_t)plan->num_splits * 4ull, &lse_bytes) ||
        __builtin_mul_overflow(lse_bytes, (uint64_t)ly.head_dim, &opart_bytes) ||
        __builtin_add_overflow(plan->lse_offset, lse_bytes, &lse_end) ||
        __builtin_add_overflow(plan->opart_offset, opart_bytes, &opart_end))
      return false;
    if (plan->opart_offset < lse_end || plan->workspace_bytes < opart_end) return false;
  }
  return true;
}

}  // namespace pd
