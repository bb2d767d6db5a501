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
static bool lens_on_device(const kvsel_desc& d) { return d.prefix_lens_dev != nullptr; }
// L_b as the host sees it: the real length, or with device lengths the bound (which sizes everything).
static int64_t len_at(const kvsel_desc& d, int b) { return lens_on_device(d) ? d.prefix_len_max : d.prefix_lens[b]; }
static int64_t nseg1(const kvsel_desc& d, int b) { return cdiv(len_at(d, b) + d.window, kScoreSeg1); }

struct WsLayout {
  size_t lse_off, part_off, norm_off, cnt_off, total;
};

static WsLayout ws_layout(const kvsel_desc& d) {
  WsLayout w{};
  const int64_t R = (int64_t)(d.h_q / d.h_kv) * d.window;
  const int64_t units = total_units(d);
  size_t off = kTableOff + kTableArea;           // error word, then the device-built tables
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
  if (d == nullptr) return KVSEL_ERR_INVALID_ARG;
  if ((d->prefix_lens == nullptr) == (d->prefix_lens_dev == nullptr)) return KVSEL_ERR_INVALID_ARG;  // exactly one
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
  for (int b = 0; b < d->batch; ++b) {     // with device lengths: the bound here, each L_b on the device
    const int64_t L = len_at(*d, b);
    if (L < 1 || L + d->window >= (int64_t(1) << 31)) return KVSEL_ERR_INVALID_ARG;
  }
  if (total_units(*d) > (int64_t(1) << 24)) return KVSEL_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return KVSEL_ERR_UNSUPPORTED;
  if ((int64_t)(d->h_q / d->h_kv) * d->window > KVSEL_MAX_ROWS) return KVSEL_ERR_UNSUPPORTED;
  return KVSEL_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// A source the gather kernel may read: memory of the current device (or managed), or pinned host
// memory mapped at the same address (on a Grace-Blackwell node the kernel then reads only the kept
// rows over the host link).  Anything else — pageable or foreign memory, another device's — is
// refused on the host instead of being dereferenced by a kernel.
// The queries are host-side and not stream-ordered: while a stream capture is under way they run
// with this thread's capture mode relaxed, so that they neither fail nor invalidate the capture.
static bool device_readable(const void* p) {
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  const bool swapped = cudaThreadExchangeStreamCaptureMode(&mode) == cudaSuccess;
  cudaPointerAttributes at;
  int dev = -1;
  bool ok = false;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
  } else if (cudaGetDevice(&dev) == cudaSuccess) {
    if (at.type == cudaMemoryTypeDevice) ok = at.device == dev;
    else if (at.type == cudaMemoryTypeManaged) ok = true;
    else if (at.type == cudaMemoryTypeHost) ok = at.devicePointer == p;
  }
  if (swapped) (void)cudaThreadExchangeStreamCaptureMode(&mode);
  return ok;
}

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
  sh.Wp = d.window;         // padded by the tensor-core launcher where it needs it
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

// ----------------------------------------------------------------------------- sequence tables
// Per-sequence checks a device-built table makes (the host makes them itself with host lengths).
struct SeqChecks {
  int32_t topk = 0, k = 0, n_recent = 0;   // kvsel_topk / kvsel_select rules on each L_b
  const int32_t* aux = nullptr;           // per-sequence aux values ([host] or [device] like the lengths)
  int32_t aux_max = 0;
};

struct PlanLaunch {
  TablePlan p;
  SeqTable* out;
  int32_t batch, with_items, include_window;
  int64_t units, seg;
};

// Builds one call's sequence table from the device-resident prefix lengths (one thread: a batch is at
// most KVSEL_MAX_BATCH sequences).  A length outside [1, prefix_len_max], or one that breaks the
// call's selection rules, records KVSEL_ERR_INVALID_ARG with the sequence as detail and leaves a
// table of empty sequences (L = 0), which every kernel skips.
__global__ void __launch_bounds__(32) seq_table_kernel(const __grid_constant__ PlanLaunch a) {
  if (threadIdx.x != 0) return;
  const TablePlan& p = a.p;
  SeqTable& t = *a.out;
  int bad = -1;
  for (int b = 0; b < a.batch && bad < 0; ++b) {
    const int64_t L = p.lens_dev[b];
    bool ok = L >= 1 && L <= p.lmax;
    if (ok && p.chk_topk) {
      if (p.P == 1) {
        ok = p.topk_k <= L;
      } else {
        const int64_t n_pages = (L + p.P - 1) / p.P;
        ok = p.n_recent <= n_pages && p.topk_k <= n_pages - p.n_recent && (L % p.P == 0 || p.n_recent >= 1);
      }
    }
    if (ok && p.aux_dev != nullptr) ok = p.aux_dev[b] >= 0 && p.aux_dev[b] <= p.aux_max;
    if (!ok) bad = b;
  }
  if (bad >= 0) {
    set_device_error(p.err, KVSEL_ERR_INVALID_ARG, (uint32_t)bad);
    t.batch = a.batch;
    t.n_items = 0;
    t.dev = nullptr;
    for (int b = 0; b < a.batch; ++b) t.s[b] = SeqInfo{};
    return;
  }
  fill_table(t, a.batch, p.lens_dev, p.aux_dev, p.n_layers, p.h_kv, p.d, p.W, p.P, p.score_rows);
  t.dev = nullptr;
  if (a.with_items) fill_items(t, a.units, a.seg, a.include_window != 0, p.W);
}

static kvsel_status launch_table(const SeqTable& host, bool with_items_, int64_t units, int64_t seg,
                                 bool include_window, int slot, cudaStream_t s) {
  PlanLaunch a;
  a.p = host.plan;
  a.out = host.plan.slots + slot;
  a.batch = host.batch;
  a.with_items = with_items_ ? 1 : 0;
  a.include_window = include_window ? 1 : 0;
  a.units = units;
  a.seg = seg;
  TraceScope ts("seq_table", s);
  seq_table_kernel<<<1, 32, 0, s>>>(a);
  return launch_status();
}

// The call's sequence table for score arrays of `score_rows` rows per sequence.  With host lengths it
// is exact.  With device lengths the host copy holds the bound for every sequence (grids and tensor
// maps are sized from it) and the real table is built on the device into workspace slot 0, on the
// call's stream; the copy's `dev` points at it.
static kvsel_status make_table(const kvsel_desc& d, int64_t score_rows, void* ws, cudaStream_t s, SeqTable* t,
                               const SeqChecks& chk = SeqChecks{}, bool build = true) {
  memset(t, 0, sizeof(*t));
  std::vector<int64_t> lens(d.batch);
  for (int b = 0; b < d.batch; ++b) lens[b] = len_at(d, b);
  const bool dev = lens_on_device(d);
  fill_table(*t, d.batch, lens.data(), dev ? nullptr : chk.aux, d.n_layers, d.h_kv, d.head_dim, d.window,
             d.page_size, score_rows);
  if (!dev) return KVSEL_OK;
  if (ws == nullptr || ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0) return KVSEL_ERR_WORKSPACE;
  if (chk.aux != nullptr)
    for (int b = 0; b < d.batch; ++b) t->s[b].aux = chk.aux_max;   // bound for sizing; real values on the device
  TablePlan& p = t->plan;
  p.lens_dev = d.prefix_lens_dev;
  p.aux_dev = chk.aux;
  p.slots = reinterpret_cast<SeqTable*>(static_cast<char*>(ws) + kTableOff);
  p.err = reinterpret_cast<DeviceError*>(ws);
  p.lmax = d.prefix_len_max;
  p.score_rows = score_rows;
  p.n_layers = d.n_layers;
  p.h_kv = d.h_kv;
  p.d = d.head_dim;
  p.W = d.window;
  p.P = d.page_size;
  p.aux_max = chk.aux_max;
  p.chk_topk = chk.topk;
  p.topk_k = chk.k;
  p.n_recent = chk.n_recent;
  t->dev = p.slots;
  return build ? launch_table(*t, false, 0, 0, false, 0, s) : KVSEL_OK;
}

kvsel_status with_items(const SeqTable& base, int64_t units_per_seq, int64_t seg, bool include_window,
                        int32_t window, int slot, cudaStream_t s, SeqTable* out) {
  *out = base;
  fill_items(*out, units_per_seq, seg, include_window, window);
  if (base.plan.lens_dev == nullptr) {
    out->dev = nullptr;
    return KVSEL_OK;
  }
  out->dev = base.plan.slots + slot;
  return launch_table(*out, true, units_per_seq, seg, include_window, slot, s);
}

// Shared checks of a top-k request (token or page mode).
static kvsel_status check_topk(const kvsel_desc& d, int32_t k, int32_t n_recent) {
  if (k < 0 || n_recent < 0) return KVSEL_ERR_INVALID_ARG;
  const int P = d.page_size;
  if (P == 1) {
    if (n_recent != 0) return KVSEL_ERR_INVALID_ARG;
    for (int b = 0; b < d.batch; ++b)
      if (k > len_at(d, b)) return KVSEL_ERR_INVALID_ARG;
  } else {
    if (d.window % P != 0) return KVSEL_ERR_UNSUPPORTED;
    for (int b = 0; b < d.batch; ++b) {
      const int64_t L = len_at(d, b);
      const int64_t n_pages = cdiv(L, P);
      if (n_recent > n_pages || k > n_pages - n_recent) return KVSEL_ERR_INVALID_ARG;
      if (!lens_on_device(d) && L % P != 0 && n_recent < 1) return KVSEL_ERR_INVALID_ARG;
    }
  }
  return KVSEL_OK;   // with device lengths these held for the bound; the device checks each L_b
}

static SeqChecks topk_checks(int32_t k, int32_t n_recent) {
  SeqChecks c;
  c.topk = 1;
  c.k = k;
  c.n_recent = n_recent;
  return c;
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
  SeqTable base;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &base, SeqChecks{}, false)) != KVSEL_OK) return st;
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
  SeqTable base;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &base, SeqChecks{}, false)) != KVSEL_OK) return st;
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
  // The prefill's last K / V tile may reach past the real rows, which must then be finite: with host
  // lengths the tensor maps end there and fill zeros; bound-sized maps could read unwritten memory.
  if (lens_on_device(d)) return KVSEL_ERR_UNSUPPORTED;
  SeqTable t;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &t)) != KVSEL_OK) return st;
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
  SeqTable t;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &t)) != KVSEL_OK) return st;
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
  SeqTable t;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &t)) != KVSEL_OK) return st;
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
  SeqTable t;
  if ((st = make_table(d, rows, ws, stream, &t, topk_checks(k, n_recent))) != KVSEL_OK) return st;
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
  SeqTable t;
  if ((st = make_table(d, rows, ws, stream, &t, topk_checks(k, n_recent))) != KVSEL_OK) return st;
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
  if (lens_on_device(d) && ws == nullptr) return KVSEL_ERR_WORKSPACE;
  if (n_sel == 0) return KVSEL_OK;
  if (!device_readable(k) || !device_readable(v)) return KVSEL_ERR_INVALID_ARG;
  SeqTable t;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &t)) != KVSEL_OK) return st;
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
  if (lens_on_device(d) && ws == nullptr) return KVSEL_ERR_WORKSPACE;
  if (n_sel == 0) return KVSEL_OK;
  if (!device_readable(k) || !device_readable(v)) return KVSEL_ERR_INVALID_ARG;
  SeqTable t;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &t)) != KVSEL_OK) return st;
  return launch_compact(d, t, k, v, idx, idx_layers, idx_heads, layer_lo, n_layers_out, n_sel, k_out, v_out,
                        reinterpret_cast<DeviceError*>(ws), stream);
}

static kvsel_status attend_plan(const kvsel_desc& d, int32_t n_q, int32_t block, int32_t max_blocks,
                                int64_t* S, size_t* bytes) {
  if (n_q < 1 || (int64_t)(d.h_q / d.h_kv) * n_q > 32) return KVSEL_ERR_UNSUPPORTED;
  if (block < 1 || block > KVSEL_MAX_PAGE || max_blocks < 0) return KVSEL_ERR_INVALID_ARG;
  const int64_t rows = total_units(d);
  const int64_t R = (int64_t)(d.h_q / d.h_kv) * n_q;
  *S = attend_splits(rows, std::max<int64_t>(1, (int64_t)max_blocks * block), (int)R, d.head_dim, block);
  if (rows * *S >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  // error word, device-built tables, partials of the splits
  *bytes = align_up(kTableOff + kTableArea + (size_t)(rows * *S * R * (d.head_dim + 2)) * sizeof(float),
                    KVSEL_WS_ALIGN);
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
  if (kv_indices == nullptr)   // whole caches: with device lengths the bound must fit
    for (int b = 0; b < d.batch; ++b)
      if (cdiv(len_at(d, b) + d.window, block) > max_blocks) return KVSEL_ERR_INVALID_ARG;
  SeqTable t;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &t)) != KVSEL_OK) return st;
  return launch_attend(d, t, q, n_q, k, v, kv_indptr, kv_indices, n_per_row, block, S,
                       reinterpret_cast<float*>(static_cast<char*>(ws) + kTableOff + kTableArea), o,
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
  if (!lens_on_device(d))
    for (int b = 0; b < d.batch; ++b)
      if (n_kvblk[b] < 0 || n_kvblk[b] > n_kvblk_max) return KVSEL_ERR_INVALID_ARG;
  SeqChecks chk;
  chk.aux = n_kvblk;            // [host], or [device] with device lengths (checked there)
  chk.aux_max = n_kvblk_max;
  SeqTable t;
  if ((st = make_table(d, (int64_t)d.n_layers * d.h_kv, ws, stream, &t, chk)) != KVSEL_OK) return st;
  const WsLayout w = ws_layout(d);
  return launch_pagetable(d, t, mask, n_qblk, n_kvblk_max,
                          reinterpret_cast<int32_t*>(static_cast<char*>(ws) + w.cnt_off), kv_indptr,
                          kv_indices, stream);
}

// ----------------------------------------------------------------------------- CLAA schedule
static kvsel_status claa_check(const kvsel_desc* desc, const kvsel_claa_params* p) {
  kvsel_status st = check_desc(desc);
  if (st != KVSEL_OK) return st;
  if (p == nullptr) return KVSEL_ERR_INVALID_ARG;
  const kvsel_desc& d = *desc;
  if (d.batch != 1 || lens_on_device(d) || d.page_size != 1) return KVSEL_ERR_UNSUPPORTED;
  if (d.group_reduce != KVSEL_REDUCE_SUM || d.score_mode != KVSEL_SCORE_SOFTMAX) return KVSEL_ERR_INVALID_ARG;
  if (p->defer < 0 || p->prune_layer < p->defer || p->prune_layer >= d.n_layers || p->n_buffer < 1)
    return KVSEL_ERR_INVALID_ARG;
  if (!(p->keep_rate >= 0.0 && p->keep_rate <= 1.0)) return KVSEL_ERR_INVALID_ARG;
  return KVSEL_OK;
}

// The scored layers' descriptor: layers m .. l_p of the prompt, pooled or (pool_k = 1) raw.
static kvsel_desc claa_sub(const kvsel_desc& d, const kvsel_claa_params& p, bool raw) {
  kvsel_desc s = d;
  s.n_layers = p.prune_layer - p.defer + 1;
  if (raw) s.pool_k = 1;
  return s;
}

kvsel_status kvsel_claa_shape(const kvsel_desc* desc, const kvsel_claa_params* p, kvsel_claa_shape_t* out) {
  kvsel_status st = claa_check(desc, p);
  if (st != KVSEL_OK) return st;
  if (out == nullptr) return KVSEL_ERR_INVALID_ARG;
  const int64_t L = desc->prefix_lens[0];
  out->n_scored = p->prune_layer - p->defer + 1;
  out->buffer_lo = std::max(p->defer, p->prune_layer - p->n_buffer + 1);
  // keep_rate -> k: floor(r L + 1/2), clipped to [0, L]
  const double kk = std::floor(p->keep_rate * (double)L + 0.5);
  out->k = (int32_t)std::min<double>((double)L, std::max(0.0, kk));
  out->n_sel = out->k + desc->window;
  const kvsel_desc sub = claa_sub(*desc, *p, false);
  out->ws_bytes = std::max(ws_layout(sub).total, ws_layout(*desc).total);
  return KVSEL_OK;
}

kvsel_status kvsel_claa_select(const kvsel_desc* desc, const kvsel_claa_params* p, const void* q, const void* k,
                               const void* v, float* scores, float* layer_scores, float* prune_scores, int32_t* idx,
                               int32_t* prune_idx, void* k_out, void* v_out, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  NvtxRange nvtx("kvsel_claa_select");
  kvsel_claa_shape_t sh;
  kvsel_status st = kvsel_claa_shape(desc, p, &sh);
  if (st != KVSEL_OK) return st;
  const kvsel_desc& d = *desc;
  if (q == nullptr || k == nullptr || v == nullptr || scores == nullptr || layer_scores == nullptr ||
      prune_scores == nullptr || idx == nullptr || prune_idx == nullptr || k_out == nullptr || v_out == nullptr)
    return KVSEL_ERR_INVALID_ARG;
  if (ws == nullptr || ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0 || ws_bytes < sh.ws_bytes) return KVSEL_ERR_WORKSPACE;
  if (sh.n_sel > 0 && (!device_readable(k) || !device_readable(v))) return KVSEL_ERR_INVALID_ARG;  // before any launch
  const int64_t L = d.prefix_lens[0];
  const kvsel_desc raw = claa_sub(d, *p, true);
  const kvsel_desc pooled = claa_sub(d, *p, false);
  // the scored layers are a contiguous slice of the prompt's q and K
  const auto* qb = static_cast<const uint16_t*>(q) + (int64_t)p->defer * d.h_q * d.window * d.head_dim;
  const auto* kb = static_cast<const uint16_t*>(k) + (int64_t)p->defer * d.h_kv * (L + d.window) * d.head_dim;
  // decision 2: every scored layer's window score, summed over the window rows and all heads, pooled
  if ((st = kvsel_score(&raw, qb, kb, scores, nullptr, ws, ws_bytes, stream)) != KVSEL_OK) return st;
  if ((st = kvsel_aggregate(&pooled, scores, 0, sh.n_scored - 1, KVSEL_LAYERS_EACH, KVSEL_HEADS_SUM, layer_scores,
                            ws, ws_bytes, stream)) != KVSEL_OK)
    return st;
  // each scored layer keeps topk(score, keep_rate) plus the window, and its cache is gathered to them
  if ((st = kvsel_select(&pooled, layer_scores, sh.n_scored, sh.k, 0, 1, idx, ws, ws_bytes, stream)) != KVSEL_OK)
    return st;
  if ((st = kvsel_compact_layers(&d, k, v, idx, sh.n_scored, 1, p->defer, sh.n_scored, sh.n_sel, k_out, v_out, ws,
                                 stream)) != KVSEL_OK)
    return st;
  // decision 3 (Eq. 6): the token-wise max over the buffer, pooled, picks the prune index at l_p
  if ((st = kvsel_aggregate(&pooled, scores, sh.buffer_lo - p->defer, sh.n_scored - 1, KVSEL_LAYERS_MAX,
                            KVSEL_HEADS_SUM, prune_scores, ws, ws_bytes, stream)) != KVSEL_OK)
    return st;
  return kvsel_select(&pooled, prune_scores, 1, sh.k, 0, 1, prune_idx, ws, ws_bytes, stream);
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
