// C ABI of libkvsel: argument checks, workspace layout, per-call sequence tables,
// tracing, and the order of kernel launches for each entry point.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.cuh"

namespace kvsel {

// ----------------------------------------------------------------------------- tracing
namespace {
struct Pending {
  std::string name;
  cudaEvent_t a, b;
};
struct TraceState {
  std::mutex mu;
  bool on = false;
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> pool;
};
TraceState& trace() {
  static TraceState t;
  return t;
}
std::atomic<int64_t> g_launches{0};

cudaEvent_t take_event(TraceState& t) {
  if (!t.pool.empty()) {
    cudaEvent_t e = t.pool.back();
    t.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

TraceScope::TraceScope(const char* n, cudaStream_t s) : name(n), stream(s), start(nullptr), on(false) {
  TraceState& t = trace();
  std::lock_guard<std::mutex> lk(t.mu);
  if (!t.on) return;
  start = take_event(t);
  if (start && cudaEventRecord(start, s) == cudaSuccess) on = true;
}

TraceScope::~TraceScope() {
  if (!on) return;
  TraceState& t = trace();
  std::lock_guard<std::mutex> lk(t.mu);
  cudaEvent_t end = take_event(t);
  if (end && cudaEventRecord(end, stream) == cudaSuccess) {
    t.pending.push_back(Pending{name, start, end});
  } else {
    t.pool.push_back(start);
    if (end) t.pool.push_back(end);
  }
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Raises a kernel's dynamic shared-memory limit to `bytes` when a launch needs more than it was
// last given.  The default limit counts static and dynamic shared memory together against 48 KB,
// so a kernel with a large static footprint needs the attribute for small dynamic sizes too; the
// attribute is per device, so the cache is too.
cudaError_t set_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<int, const void*>, size_t>> given;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  for (auto& e : given)
    if (e.first.first == dev && e.first.second == func) {
      if (e.second >= bytes) return cudaSuccess;
      const cudaError_t st = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
      if (st == cudaSuccess) e.second = bytes;
      return st;
    }
  const cudaError_t st = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (st == cudaSuccess) given.push_back({{dev, func}, bytes});
  return st;
}

// ----------------------------------------------------------------------------- geometry
static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int64_t total_units(const kvsel_desc& d) { return (int64_t)d.batch * d.n_layers * d.h_kv; }
static int64_t nseg1(const kvsel_desc& d, int b) { return cdiv(d.prefix_lens[b] + d.window, kScoreSeg1); }

struct WsLayout {
  size_t lse_off, part_off, norm_off, cnt_off, total;
};

static WsLayout ws_layout(const kvsel_desc& d) {
  WsLayout w{};
  const int64_t R = (int64_t)(d.h_q / d.h_kv) * d.window;
  const int64_t units = total_units(d);
  size_t off = sizeof(DeviceError);
  w.lse_off = off;
  off = align_up(off + (size_t)(units * R) * sizeof(float), KVSEL_WS_ALIGN);
  w.part_off = off;
  int64_t parts = 0;
  for (int b = 0; b < d.batch; ++b) parts += (int64_t)d.n_layers * d.h_kv * nseg1(d, b) * R;
  off = align_up(off + (size_t)parts * sizeof(float2), KVSEL_WS_ALIGN);
  w.norm_off = off;
  off = align_up(off + (size_t)units * sizeof(float), KVSEL_WS_ALIGN);
  w.cnt_off = off;
  off = align_up(off + (size_t)units * sizeof(int32_t), KVSEL_WS_ALIGN);
  w.total = off;
  return w;
}

// ----------------------------------------------------------------------------- checks
static kvsel_status check_desc(const kvsel_desc* d) {
  if (d == nullptr || d->prefix_lens == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (d->n_layers < 1 || d->h_kv < 1 || d->h_q < 1 || d->h_q % d->h_kv != 0) return KVSEL_ERR_INVALID_ARG;
  if (d->batch < 1 || d->batch > KVSEL_MAX_BATCH) return KVSEL_ERR_INVALID_ARG;
  if (d->window < 1 || d->window > KVSEL_MAX_WINDOW) return KVSEL_ERR_INVALID_ARG;
  if (d->group_reduce != KVSEL_REDUCE_SUM && d->group_reduce != KVSEL_REDUCE_MAX &&
      d->group_reduce != KVSEL_REDUCE_MEAN)
    return KVSEL_ERR_INVALID_ARG;
  if (d->page_reduce != KVSEL_REDUCE_SUM && d->page_reduce != KVSEL_REDUCE_MAX) return KVSEL_ERR_INVALID_ARG;
  if (d->pool_type != KVSEL_POOL_MAX && d->pool_type != KVSEL_POOL_AVG) return KVSEL_ERR_INVALID_ARG;
  if (d->score_mode != KVSEL_SCORE_SOFTMAX && d->score_mode != KVSEL_SCORE_LOGITS) return KVSEL_ERR_INVALID_ARG;
  if (d->pool_k < 1 || d->pool_k % 2 == 0 || d->pool_k > 63) return KVSEL_ERR_INVALID_ARG;
  if (d->page_size < 1 || d->page_size > KVSEL_MAX_PAGE) return KVSEL_ERR_INVALID_ARG;
  for (int b = 0; b < d->batch; ++b) {
    const int64_t L = d->prefix_lens[b];
    if (L < 1 || L + d->window >= (int64_t(1) << 31)) return KVSEL_ERR_INVALID_ARG;
  }
  if (total_units(*d) > (int64_t(1) << 24)) return KVSEL_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return KVSEL_ERR_UNSUPPORTED;
  if ((int64_t)(d->h_q / d->h_kv) * d->window > KVSEL_MAX_ROWS) return KVSEL_ERR_UNSUPPORTED;
  return KVSEL_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

kvsel_status check_score_args(const kvsel_desc* desc, const void* q, const void* k, const float* scores,
                              const float* page_scores) {
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  if (q == nullptr || k == nullptr || scores == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(scores)) return KVSEL_ERR_INVALID_ARG;
  if (desc->page_size > 1 && page_scores == nullptr) return KVSEL_ERR_INVALID_ARG;
  return KVSEL_OK;
}

static kvsel_status check_ws(const kvsel_desc& d, void* ws, size_t ws_bytes) {
  if (ws == nullptr || ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0) return KVSEL_ERR_WORKSPACE;
  if (ws_bytes < ws_layout(d).total) return KVSEL_ERR_WORKSPACE;
  return KVSEL_OK;
}

ScoreShape make_shape(const kvsel_desc& d) {
  ScoreShape sh;
  sh.n_layers = d.n_layers; sh.h_q = d.h_q; sh.h_kv = d.h_kv; sh.d = d.head_dim; sh.W = d.window;
  sh.G = d.h_q / d.h_kv; sh.R = sh.G * d.window;
  sh.group_reduce = d.group_reduce; sh.pool_k = d.pool_k; sh.page_size = d.page_size;
  sh.page_reduce = d.page_reduce;
  sh.pool_type = d.pool_type;
  sh.logits = d.score_mode == KVSEL_SCORE_LOGITS ? 1 : 0;
  sh.lse_given = 0;
  sh.seg1 = sh.seg2 = 0;    // set by the launcher
  sh.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.head_dim));
  sh.scale_nat = (float)(1.0 / std::sqrt((double)d.head_dim));
  sh.gscale = d.group_reduce == KVSEL_REDUCE_MEAN ? (float)(1.0 / ((double)sh.R)) : 1.0f;
  return sh;
}

// Sequence table: element offsets of each sequence in the packed layouts.
static SeqTable make_table(const kvsel_desc& d, int32_t layers_in_scores) {
  SeqTable t;
  memset(&t, 0, sizeof(t));
  t.batch = d.batch;
  int64_t k_off = 0, s_off = 0, p_off = 0;
  for (int b = 0; b < d.batch; ++b) {
    SeqInfo& s = t.s[b];
    s.L = (int32_t)d.prefix_lens[b];
    s.n_keys = s.L + d.window;
    s.k_off = k_off;
    s.s_off = s_off;
    s.p_off = p_off;
    s.unit0 = b * d.n_layers * d.h_kv;
    k_off += (int64_t)d.n_layers * d.h_kv * s.n_keys * d.head_dim;
    s_off += (int64_t)layers_in_scores * d.h_kv * s.L;
    p_off += (int64_t)layers_in_scores * d.h_kv * cdiv(s.L, d.page_size);
  }
  return t;
}

// Sequence table for `rows` score rows per sequence (top-k inputs): s_off / p_off become the
// offsets of each sequence's [rows][L_b] token scores / [rows][ceil(L_b / P)] page scores.
static SeqTable make_table_rows(const kvsel_desc& d, int32_t rows) {
  SeqTable t = make_table(d, d.n_layers);
  int64_t s_off = 0, p_off = 0;
  for (int b = 0; b < d.batch; ++b) {
    t.s[b].s_off = s_off;
    t.s[b].p_off = p_off;
    s_off += (int64_t)rows * t.s[b].L;
    p_off += (int64_t)rows * cdiv(t.s[b].L, d.page_size);
  }
  return t;
}

// Shared checks of a top-k request (token or page mode).
static kvsel_status check_topk(const kvsel_desc& d, int32_t k, int32_t n_recent) {
  if (k < 0 || n_recent < 0) return KVSEL_ERR_INVALID_ARG;
  const int P = d.page_size;
  if (P == 1) {
    if (n_recent != 0) return KVSEL_ERR_INVALID_ARG;
    for (int b = 0; b < d.batch; ++b)
      if (k > d.prefix_lens[b]) return KVSEL_ERR_INVALID_ARG;
  } else {
    if (d.window % P != 0) return KVSEL_ERR_UNSUPPORTED;
    for (int b = 0; b < d.batch; ++b) {
      const int64_t L = d.prefix_lens[b];
      const int64_t n_pages = cdiv(L, P);
      if (n_recent > n_pages || k > n_pages - n_recent) return KVSEL_ERR_INVALID_ARG;
      if (L % P != 0 && n_recent < 1) return KVSEL_ERR_INVALID_ARG;
    }
  }
  return KVSEL_OK;
}

}  // namespace kvsel

using namespace kvsel;

// ============================================================================= C ABI
extern "C" {

const char* kvsel_version(void) { return "kvsel 0.2 (sm_103a)"; }

const char* kvsel_status_string(kvsel_status s) {
  switch (s) {
    case KVSEL_OK: return "ok";
    case KVSEL_ERR_INVALID_ARG: return "invalid argument";
    case KVSEL_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case KVSEL_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case KVSEL_ERR_CUDA: return "CUDA error";
    case KVSEL_ERR_TIMEOUT: return "bounded device wait timed out";
    case KVSEL_ERR_DEVICE: return "device-side index out of range";
  }
  return "unknown status";
}

kvsel_status kvsel_workspace_size(const kvsel_desc* desc, size_t* bytes) {
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  if (bytes == nullptr) return KVSEL_ERR_INVALID_ARG;
  *bytes = ws_layout(*desc).total;
  return KVSEL_OK;
}

kvsel_status kvsel_score(const kvsel_desc* desc, const void* q, const void* k, float* scores,
                         float* page_scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx("kvsel_score");
  kvsel_status st = check_score_args(desc, q, k, scores, page_scores);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if ((st = check_ws(d, ws, ws_bytes)) != KVSEL_OK) return st;
  const WsLayout w = ws_layout(d);
  auto ws_base = [](void* p) { return static_cast<char*>(p); };

  const ScoreShape sh = make_shape(d);
  const SeqTable base = make_table(d, d.n_layers);
  return launch_score(sh, base, q, k, scores, page_scores, reinterpret_cast<float*>(ws_base(ws) + w.lse_off),
                      reinterpret_cast<float2*>(ws_base(ws) + w.part_off), reinterpret_cast<DeviceError*>(ws),
                      stream);
}

kvsel_status kvsel_score_from_lse(const kvsel_desc* desc, const void* q_win, const void* k, const float* lse_win,
                                  float* scores, float* page_scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx("kvsel_score_from_lse");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (q_win == nullptr || k == nullptr || scores == nullptr || lse_win == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (!aligned16(q_win) || !aligned16(k) || !aligned16(scores)) return KVSEL_ERR_INVALID_ARG;
  if (d.page_size > 1 && page_scores == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (d.score_mode != KVSEL_SCORE_SOFTMAX) return KVSEL_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != KVSEL_OK) return st;
  const WsLayout w = ws_layout(d);
  ScoreShape sh = make_shape(d);
  sh.lse_given = 1;
  const SeqTable base = make_table(d, d.n_layers);
  return launch_score(sh, base, q_win, k, scores, page_scores, const_cast<float*>(lse_win),
                      reinterpret_cast<float2*>(static_cast<char*>(ws) + w.part_off), reinterpret_cast<DeviceError*>(ws),
                      stream);
}

kvsel_status kvsel_prefill_attention(const kvsel_desc* desc, const void* q, const void* k, const void* v, void* o,
                                     float* lse, float* lse_win, void* q_win, void* ws, cudaStream_t stream) {
  NvtxRange nvtx("kvsel_prefill_attention");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (d.head_dim != 128) return KVSEL_ERR_UNSUPPORTED;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse_win == nullptr || q_win == nullptr)
    return KVSEL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(q_win)) return KVSEL_ERR_INVALID_ARG;
  if (ws != nullptr && ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0) return KVSEL_ERR_WORKSPACE;
  const SeqTable t = make_table(d, d.n_layers);
  return launch_prefill(d, t, q, k, v, o, lse, lse_win, q_win, reinterpret_cast<DeviceError*>(ws), stream);
}

kvsel_status kvsel_combine_layers(const kvsel_desc* desc, const float* scores, int32_t layer_lo,
                                  int32_t layer_hi, float* combined, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  NvtxRange nvtx("kvsel_combine_layers");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (scores == nullptr || combined == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (layer_lo < 0 || layer_hi < layer_lo || layer_hi >= d.n_layers) return KVSEL_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != KVSEL_OK) return st;
  SeqTable t = make_table(d, d.n_layers);
  const WsLayout w = ws_layout(d);
  return launch_aggregate(d, t, scores, layer_lo, layer_hi, KVSEL_LAYERS_L1_MEAN, KVSEL_HEADS_EACH,
                          reinterpret_cast<float*>(static_cast<char*>(ws) + w.norm_off), combined, stream);
}

kvsel_status kvsel_aggregate(const kvsel_desc* desc, const float* scores, int32_t layer_lo, int32_t layer_hi,
                             int32_t layer_op, int32_t head_op, float* out, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  NvtxRange nvtx("kvsel_aggregate");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (scores == nullptr || out == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (layer_lo < 0 || layer_hi < layer_lo || layer_hi >= d.n_layers) return KVSEL_ERR_INVALID_ARG;
  if (layer_op != KVSEL_LAYERS_EACH && layer_op != KVSEL_LAYERS_L1_MEAN && layer_op != KVSEL_LAYERS_MAX)
    return KVSEL_ERR_INVALID_ARG;
  if (head_op != KVSEL_HEADS_EACH && head_op != KVSEL_HEADS_SUM) return KVSEL_ERR_INVALID_ARG;
  if ((st = check_ws(d, ws, ws_bytes)) != KVSEL_OK) return st;
  SeqTable t = make_table(d, d.n_layers);
  const WsLayout w = ws_layout(d);
  return launch_aggregate(d, t, scores, layer_lo, layer_hi, layer_op, head_op,
                          reinterpret_cast<float*>(static_cast<char*>(ws) + w.norm_off), out, stream);
}

kvsel_status kvsel_select(const kvsel_desc* desc, const float* scores, int32_t rows, int32_t k, int32_t n_recent,
                          int32_t append_window, int32_t* idx_out, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
  NvtxRange nvtx("kvsel_select");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (scores == nullptr || idx_out == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (rows < 1 || (int64_t)rows * d.batch >= (int64_t(1) << 31)) return KVSEL_ERR_INVALID_ARG;
  if ((st = check_topk(d, k, n_recent)) != KVSEL_OK) return st;
  if ((st = check_ws(d, ws, ws_bytes)) != KVSEL_OK) return st;
  SeqTable t = make_table_rows(d, rows);
  return launch_topk(d, t, rows, k, n_recent, append_window != 0, scores, idx_out, stream);
}

kvsel_status kvsel_topk(const kvsel_desc* desc, const float* scores, int32_t layers, int32_t k,
                        int32_t n_recent, int32_t* idx_out, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  NvtxRange nvtx("kvsel_topk");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (scores == nullptr || idx_out == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (layers != 1 && layers != d.n_layers) return KVSEL_ERR_INVALID_ARG;
  if ((st = check_topk(d, k, n_recent)) != KVSEL_OK) return st;
  if ((st = check_ws(d, ws, ws_bytes)) != KVSEL_OK) return st;
  const int32_t rows = layers * d.h_kv;
  SeqTable t = make_table_rows(d, rows);
  return launch_topk(d, t, rows, k, n_recent, true, scores, idx_out, stream);
}

kvsel_status kvsel_compact(const kvsel_desc* desc, const void* k, const void* v, const int32_t* idx,
                           int32_t idx_layers, int32_t n_sel, void* k_out, void* v_out, void* ws,
                           cudaStream_t stream) {
  NvtxRange nvtx("kvsel_compact");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (k == nullptr || v == nullptr || idx == nullptr || k_out == nullptr || v_out == nullptr)
    return KVSEL_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out)) return KVSEL_ERR_INVALID_ARG;
  if (idx_layers != 1 && idx_layers != d.n_layers) return KVSEL_ERR_INVALID_ARG;
  if (n_sel < 0) return KVSEL_ERR_INVALID_ARG;
  if ((int64_t)n_sel * d.page_size >= (int64_t(1) << 31)) return KVSEL_ERR_INVALID_ARG;
  if (ws != nullptr && ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0) return KVSEL_ERR_WORKSPACE;
  if (n_sel == 0) return KVSEL_OK;
  SeqTable t = make_table(d, d.n_layers);
  return launch_compact(d, t, k, v, idx, idx_layers, d.h_kv, 0, d.n_layers, n_sel, k_out, v_out,
                        reinterpret_cast<DeviceError*>(ws), stream);
}

kvsel_status kvsel_compact_layers(const kvsel_desc* desc, const void* k, const void* v, const int32_t* idx,
                                  int32_t idx_layers, int32_t idx_heads, int32_t layer_lo, int32_t n_layers_out,
                                  int32_t n_sel, void* k_out, void* v_out, void* ws, cudaStream_t stream) {
  NvtxRange nvtx("kvsel_compact_layers");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (k == nullptr || v == nullptr || idx == nullptr || k_out == nullptr || v_out == nullptr)
    return KVSEL_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out)) return KVSEL_ERR_INVALID_ARG;
  if (layer_lo < 0 || n_layers_out < 1 || layer_lo + n_layers_out > d.n_layers) return KVSEL_ERR_INVALID_ARG;
  if (idx_layers != 1 && idx_layers != n_layers_out) return KVSEL_ERR_INVALID_ARG;
  if (idx_heads != 1 && idx_heads != d.h_kv) return KVSEL_ERR_INVALID_ARG;
  if (n_sel < 0) return KVSEL_ERR_INVALID_ARG;
  if ((int64_t)n_sel * d.page_size >= (int64_t(1) << 31)) return KVSEL_ERR_INVALID_ARG;
  if (ws != nullptr && ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0) return KVSEL_ERR_WORKSPACE;
  if (n_sel == 0) return KVSEL_OK;
  SeqTable t = make_table(d, d.n_layers);
  return launch_compact(d, t, k, v, idx, idx_layers, idx_heads, layer_lo, n_layers_out, n_sel, k_out, v_out,
                        reinterpret_cast<DeviceError*>(ws), stream);
}

static kvsel_status attend_plan(const kvsel_desc& d, int32_t n_q, int32_t block, int32_t max_blocks,
                                int64_t* S, size_t* bytes) {
  if (n_q < 1 || (int64_t)(d.h_q / d.h_kv) * n_q > 32) return KVSEL_ERR_UNSUPPORTED;
  if (block < 1 || block > KVSEL_MAX_PAGE || max_blocks < 0) return KVSEL_ERR_INVALID_ARG;
  const int64_t rows = total_units(d);
  const int64_t R = (int64_t)(d.h_q / d.h_kv) * n_q;
  *S = attend_splits(rows, std::max<int64_t>(1, (int64_t)max_blocks * block), (int)R, d.head_dim);
  if (rows * *S >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  // error word, partials of the splits
  *bytes = align_up(sizeof(DeviceError) + (size_t)(rows * *S * R * (d.head_dim + 2)) * sizeof(float), KVSEL_WS_ALIGN);
  return KVSEL_OK;
}

kvsel_status kvsel_attend_workspace_size(const kvsel_desc* desc, int32_t n_q, int32_t block, int32_t max_blocks,
                                         size_t* bytes) {
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  if (bytes == nullptr) return KVSEL_ERR_INVALID_ARG;
  int64_t S = 0;
  return attend_plan(*desc, n_q, block, max_blocks, &S, bytes);
}

kvsel_status kvsel_attend(const kvsel_desc* desc, const void* q, int32_t n_q, const void* k, const void* v,
                          const int32_t* kv_indptr, const int32_t* kv_indices, int32_t n_per_row, int32_t block,
                          int32_t max_blocks, float* o, void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx("kvsel_attend");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return KVSEL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return KVSEL_ERR_INVALID_ARG;
  if (kv_indices == nullptr && kv_indptr != nullptr) return KVSEL_ERR_INVALID_ARG;
  if (kv_indices != nullptr && kv_indptr == nullptr && (n_per_row < 0 || n_per_row > max_blocks))
    return KVSEL_ERR_INVALID_ARG;
  int64_t S = 0;
  size_t need = 0;
  if ((st = attend_plan(d, n_q, block, max_blocks, &S, &need)) != KVSEL_OK) return st;
  if (ws == nullptr || ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0 || ws_bytes < need) return KVSEL_ERR_WORKSPACE;
  if (kv_indices == nullptr)
    for (int b = 0; b < d.batch; ++b)
      if (cdiv(d.prefix_lens[b] + d.window, block) > max_blocks) return KVSEL_ERR_INVALID_ARG;
  SeqTable t = make_table(d, d.n_layers);
  return launch_attend(d, t, q, n_q, k, v, kv_indptr, kv_indices, n_per_row, block, S,
                       reinterpret_cast<float*>(static_cast<char*>(ws) + sizeof(DeviceError)), o,
                       reinterpret_cast<DeviceError*>(ws), stream);
}

kvsel_status kvsel_pagetable(const kvsel_desc* desc, const uint8_t* mask, int32_t n_qblk,
                             int32_t n_kvblk_max, const int32_t* n_kvblk, int32_t* kv_indptr,
                             int32_t* kv_indices, void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx("kvsel_pagetable");
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (mask == nullptr || n_kvblk == nullptr || kv_indptr == nullptr || kv_indices == nullptr)
    return KVSEL_ERR_INVALID_ARG;
  if (n_qblk < 1 || n_kvblk_max < 1) return KVSEL_ERR_INVALID_ARG;
  if (total_units(d) * n_kvblk_max >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  if ((st = check_ws(d, ws, ws_bytes)) != KVSEL_OK) return st;
  SeqTable t = make_table(d, d.n_layers);
  for (int b = 0; b < d.batch; ++b) {
    if (n_kvblk[b] < 0 || n_kvblk[b] > n_kvblk_max) return KVSEL_ERR_INVALID_ARG;
    t.s[b].aux = n_kvblk[b];
  }
  const WsLayout w = ws_layout(d);
  return launch_pagetable(d, t, mask, n_qblk, n_kvblk_max,
                          reinterpret_cast<int32_t*>(static_cast<char*>(ws) + w.cnt_off), kv_indptr,
                          kv_indices, stream);
}

kvsel_status kvsel_read_device_error(void* ws, cudaStream_t stream) {
  if (ws == nullptr || ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0) return KVSEL_ERR_WORKSPACE;
  uint32_t h[2] = {0, 0};
  if (cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return KVSEL_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KVSEL_ERR_CUDA;
  if (h[0] != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(h), stream) != cudaSuccess) return KVSEL_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KVSEL_ERR_CUDA;
    return (kvsel_status)h[0];
  }
  return KVSEL_OK;
}

void kvsel_trace_enable(int32_t on) {
  TraceState& t = trace();
  std::lock_guard<std::mutex> lk(t.mu);
  t.on = on != 0;
}

kvsel_status kvsel_trace_read(kvsel_trace_entry* out, int32_t capacity, int32_t* n_out) {
  TraceState& t = trace();
  std::lock_guard<std::mutex> lk(t.mu);
  std::vector<kvsel_trace_entry> acc;
  kvsel_status st = KVSEL_OK;
  for (Pending& p : t.pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess)
      st = KVSEL_ERR_CUDA;
    kvsel_trace_entry* e = nullptr;
    for (auto& x : acc)
      if (p.name == x.name) e = &x;
    if (e == nullptr) {
      acc.push_back(kvsel_trace_entry{});
      e = &acc.back();
      strncpy(e->name, p.name.c_str(), sizeof(e->name) - 1);
    }
    e->launches += 1;
    e->ms += ms;
    t.pool.push_back(p.a);
    t.pool.push_back(p.b);
  }
  t.pending.clear();
  int32_t n = 0;
  for (auto& x : acc) {
    if (out != nullptr && n < capacity) out[n] = x;
    ++n;
  }
  if (n_out) *n_out = n;
  return st;
}

int64_t kvsel_launch_count(void) { return g_launches.load(); }

}  // extern "C"
