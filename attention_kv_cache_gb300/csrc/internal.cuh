// Internal declarations shared by the translation units of libkvsel.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "kvsel.h"

namespace kvsel {

// A named range on a profiler's host timeline spanning one entry-point call (NVTX, header-only);
// a no-op unless a tool that records NVTX ranges is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Error word at the start of every workspace (device side).
struct DeviceError {
  uint32_t code;       // 0 = none, else a kvsel_status value
  uint32_t where;      // kernel-specific detail (first failure wins)
  uint32_t pad[62];
};
static_assert(sizeof(DeviceError) == 256, "error header is one 256-byte line");

__device__ __forceinline__ void set_device_error(DeviceError* e, uint32_t code, uint32_t where) {
  if (e == nullptr) return;
  if (atomicCAS(&e->code, 0u, code) == 0u) atomicExch(&e->where, where);
}

// Per-sequence geometry of one call (lives in kernel parameters, or in the workspace when the
// prefix lengths live on the device).
struct SeqInfo {
  int32_t L;            // prefix length L_b (0 in a table whose device lengths failed the checks)
  int32_t n_keys;       // L_b + W
  int64_t k_off;        // element offset of the sequence's K / V block
  int64_t s_off;        // element offset of its token scores ([layers][h_kv][L_b])
  int64_t p_off;        // element offset of its page scores ([layers][h_kv][ceil(L_b/P)])
  int32_t item0;        // first work item of this sequence in the current launch
  int32_t n_seg;        // segments per (layer, KV head) unit in the current launch
  int64_t part_off;     // index of its first (unit, segment) partial record
  int32_t unit0;        // global index of its first (layer, KV head) unit
  int32_t aux;          // launch-specific (KV blocks for the page table)
};

struct SeqTable;

// How a call whose prefix lengths live on the device rebuilds its tables there (host side only;
// the kernels never read it).  The host copy of such a table is built from the bound prefix_len_max
// for every sequence, so the grids and tensor maps sized from it cover every real length.
struct TablePlan {
  const int64_t* lens_dev;   // [device] L_b, or nullptr: host lengths, the host table is the real one
  const int32_t* aux_dev;    // [device] per-sequence aux values (page-table KV blocks), or nullptr
  SeqTable* slots;           // [device] kTableSlots tables in the workspace
  DeviceError* err;
  int64_t lmax;              // every L_b must lie in [1, lmax]
  int64_t score_rows;        // score rows per sequence (the s_off / p_off strides)
  int32_t n_layers, h_kv, d, W, P;
  int32_t aux_max;           // aux_dev entries must lie in [0, aux_max]
  int32_t chk_topk, topk_k, n_recent;   // per-sequence selection checks (kvsel_topk / kvsel_select)
};

struct SeqTable {
  int32_t batch;
  int32_t n_items;
  const SeqTable* dev;       // [device] the real table (built from device lengths), or nullptr
  TablePlan plan;
  SeqInfo s[KVSEL_MAX_BATCH];
};

// Tables a call may keep in its workspace, right after the error word.
constexpr int kTableSlots = 2;
constexpr size_t kTableArea = (kTableSlots * sizeof(SeqTable) + KVSEL_WS_ALIGN - 1) / KVSEL_WS_ALIGN * KVSEL_WS_ALIGN;
constexpr size_t kTableOff = sizeof(DeviceError);

// The table a kernel reads: its parameter, or the device-built table the parameter points to.
__device__ __forceinline__ const SeqTable& real_table(const SeqTable& param) {
  return param.dev != nullptr ? *param.dev : param;
}

__device__ __forceinline__ int find_seq(const SeqTable& t, int item) {
  int b = 0;
  while (b + 1 < t.batch && t.s[b + 1].item0 <= item) ++b;
  return b;
}

// Per-sequence geometry from the prefix lengths (host lengths, bounds, or on the device, the real
// ones): offsets of each sequence in the packed K / V, score and page-score layouts.  Work items
// are left empty (with_items fills them).
__host__ __device__ inline void fill_table(SeqTable& t, int batch, const int64_t* lens, const int32_t* aux,
                                           int n_layers, int h_kv, int d, int W, int P, int64_t score_rows) {
  t.batch = batch;
  t.n_items = 0;
  int64_t k_off = 0, s_off = 0, p_off = 0;
  for (int b = 0; b < batch; ++b) {
    SeqInfo& s = t.s[b];
    s.L = (int32_t)lens[b];
    s.n_keys = s.L + W;
    s.k_off = k_off;
    s.s_off = s_off;
    s.p_off = p_off;
    s.item0 = 0;
    s.n_seg = 0;
    s.part_off = 0;
    s.unit0 = b * n_layers * h_kv;
    s.aux = aux != nullptr ? aux[b] : 0;
    k_off += (int64_t)n_layers * h_kv * s.n_keys * d;
    s_off += score_rows * s.L;
    p_off += score_rows * ((s.L + P - 1) / P);
  }
}

// Work items: n_seg = ceil(len_b / seg) segments for each (layer, KV head) unit of sequence b,
// where len_b is L_b + W (pass 1) or L_b (pass 2).
__host__ __device__ inline void fill_items(SeqTable& t, int64_t units_per_seq, int64_t seg, bool include_window,
                                           int32_t window) {
  int64_t item = 0;
  for (int b = 0; b < t.batch; ++b) {
    const int64_t len = (int64_t)t.s[b].L + (include_window && t.s[b].L > 0 ? window : 0);
    const int64_t ns = (len + seg - 1) / seg;
    t.s[b].item0 = (int32_t)item;
    t.s[b].n_seg = (int32_t)ns;
    t.s[b].part_off = item;
    item += units_per_seq * ns;
  }
  t.n_items = (int32_t)item;
}

// Keys per pass-1 segment (fixes the size of the per-segment partials in the workspace).
constexpr int64_t kScoreSeg1 = 2048;

// Problem description handed to every scoring kernel.
struct ScoreShape {
  int32_t n_layers, h_q, h_kv, d, W, G, R;   // R = G * W rows per unit
  int32_t Wp;                                // tensor-core tile rows per head (a power of two >= W for the
                                             // group max, so every head fills whole register groups; else W)
  int32_t group_reduce, pool_k, page_size, page_reduce;
  int32_t pool_type;                         // KVSEL_POOL_MAX / KVSEL_POOL_AVG
  int32_t logits;                            // 1: pre-softmax scaled logits (one pass, no lse)
  int32_t lse_given;                         // 1: the rows' lse is an input (the prefill's); pass 2 only
  int32_t seg1, seg2;                        // keys per pass-1 / pass-2 segment
  float scale_log2;                          // log2(e) / sqrt(d)
  float scale_nat;                           // 1 / sqrt(d)
  float gscale;                              // factor on the group score: 1, or 1 / (G * W) for the mean
};

// Score shape of a checked descriptor (kvsel_api.cu).
ScoreShape make_shape(const kvsel_desc& d);

// The checks kvsel_score makes of its descriptor and pointers, workspace aside (kvsel_api.cu).
kvsel_status check_score_args(const kvsel_desc* desc, const void* q, const void* k, const float* scores,
                              const float* page_scores);

// ---- launch plumbing (kvsel_api.cu) ------------------------------------------------
struct TraceScope {
  TraceScope(const char* name, cudaStream_t s);
  ~TraceScope();
  const char* name;
  cudaStream_t stream;
  cudaEvent_t start;
  bool on;
};
void count_launch();
cudaError_t set_smem(const void* func, size_t bytes);

inline kvsel_status launch_status() {
  count_launch();
  return cudaGetLastError() == cudaSuccess ? KVSEL_OK : KVSEL_ERR_CUDA;
}

// ---- kernel launchers ---------------------------------------------------------------
// Scoring: launch_score (score_tc.cu) picks the tensor-core kernels for the shapes they
// cover and the CUDA-core kernels otherwise.  `base` carries the per-sequence geometry;
// the launchers add their own work-item tables.
kvsel_status launch_score(const ScoreShape& sh, const SeqTable& base, const void* q, const void* k,
                          float* scores, float* page_scores, float* lse, float2* part, DeviceError* err,
                          cudaStream_t s);
kvsel_status launch_score_simt(const ScoreShape& sh, const SeqTable& t1, const SeqTable& t2,
                               const void* q, const void* k, float* scores, float* page_scores,
                               float* lse, float2* part, DeviceError* err, cudaStream_t s);
kvsel_status launch_lse_combine(const ScoreShape& sh, const SeqTable& t1, float2* part, float* lse,
                                cudaStream_t s);

// A copy of `base` with work items (fill_items).  With device lengths the same table is also built on
// the device, into workspace slot `slot`, and the copy points at it (kvsel_api.cu).
kvsel_status with_items(const SeqTable& base, int64_t units_per_seq, int64_t seg, bool include_window,
                        int32_t window, int slot, cudaStream_t s, SeqTable* out);

// Top-k over `rows` score rows per sequence; sequence b's rows start at element
// rows * (sum of n over earlier sequences), n = L_b or ceil(L_b / P).
kvsel_status launch_topk(const kvsel_desc& desc, const SeqTable& t, int rows, int k, int n_recent,
                         bool append_window, const float* scores, int32_t* idx, cudaStream_t s);

kvsel_status launch_aggregate(const kvsel_desc& desc, const SeqTable& t, const float* scores, int lo, int hi,
                              int layer_op, int head_op, float* norms, float* out, cudaStream_t s);

kvsel_status launch_compact(const kvsel_desc& desc, const SeqTable& t, const void* k, const void* v,
                            const int32_t* idx, int idx_layers, int idx_heads, int layer_lo, int n_layers_out,
                            int n_sel, void* k_out, void* v_out, DeviceError* err, cudaStream_t s);

// Causal prefill attention with the window rows' lse and queries (prefill.cu).
kvsel_status launch_prefill(const kvsel_desc& d, const SeqTable& t, const void* q, const void* k, const void* v,
                            void* o, float* lse, float* lse_win, void* q_win, DeviceError* err, cudaStream_t s);

// Attention over a page / block table (attend.cu).
// R = query rows per table row; block = rows per listed block
int64_t attend_splits(int64_t rows, int64_t max_rows_per_list, int R, int d, int block);
kvsel_status launch_attend(const kvsel_desc& d, const SeqTable& t, const void* q, int n_q, const void* k,
                           const void* v, const int32_t* indptr, const int32_t* indices, int n_per_row, int P,
                           int64_t S, float* part, float* o, DeviceError* err, cudaStream_t s);

kvsel_status launch_pagetable(const kvsel_desc& desc, const SeqTable& t, const uint8_t* mask,
                              int n_qblk, int n_kvblk_max, int32_t* counts, int32_t* kv_indptr,
                              int32_t* kv_indices, cudaStream_t s);

}  // namespace kvsel
