// KV compaction (16-byte vector gather) and the block-union page table.
#include "internal.cuh"

namespace kvsel {
namespace {

// ------------------------------------------------------------------------ compaction
struct CompactArgs {
  const uint4* k;
  const uint4* v;
  const int32_t* idx;
  uint4* k_out;
  uint4* v_out;
  DeviceError* err;
  int32_t n_layers, h_kv, vpr, n_sel, P, idx_layers;
  int64_t rows_per_seq;   // n_layers * h_kv * n_sel * P
  int64_t total_vecs;     // batch * rows_per_seq * vpr
};

// One thread moves one 16-byte vector of K and of V.  Consecutive threads cover
// consecutive vectors of a row, so every row is read and written as whole
// 128-byte lines.
__global__ void __launch_bounds__(256) compact_kernel(const __grid_constant__ CompactArgs a,
                                                      const __grid_constant__ SeqTable t) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t per_sel = (int64_t)a.n_sel * a.P;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < a.total_vecs; v += stride) {
    const int64_t row = v / a.vpr;
    const int c = (int)(v % a.vpr);
    const int b = (int)(row / a.rows_per_seq);
    const int64_t rr = row % a.rows_per_seq;
    const int lg = (int)(rr / per_sel);
    const int within = (int)(rr % per_sel);
    const int layer = lg / a.h_kv, g = lg % a.h_kv;
    const int il = a.idx_layers == 1 ? 0 : layer;
    const SeqInfo& si = t.s[b];
    const int32_t id = a.idx[(((int64_t)b * a.idx_layers + il) * a.h_kv + g) * a.n_sel + within / a.P];
    const int64_t src_row = (int64_t)id * a.P + within % a.P;
    const int64_t lim = a.P == 1 ? si.n_keys : ((int64_t)si.n_keys + a.P - 1) / a.P;
    uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (id < 0 || id >= lim) {
      if (c == 0) set_device_error(a.err, KVSEL_ERR_DEVICE, (uint32_t)row);
    } else if (src_row < si.n_keys) {
      const int64_t off = (si.k_off / 8) + (((int64_t)layer * a.h_kv + g) * si.n_keys + src_row) * a.vpr + c;
      kv = a.k[off];
      vv = a.v[off];
    }
    a.k_out[v] = kv;
    a.v_out[v] = vv;
  }
}

// ------------------------------------------------------------------------ page table
constexpr int kPtThreads = 256;

struct PtArgs {
  const uint8_t* mask;
  int32_t* counts;
  int32_t* indptr;
  int32_t* indices;
  int32_t n_layers, h_q, h_kv, n_qblk, nmax, rows;
};

// OR over the Q blocks and the query heads of group g for KV block j.
__device__ __forceinline__ bool union_hit(const PtArgs& a, int b, int layer, int g, int j) {
  const int G = a.h_q / a.h_kv;
  for (int h = g * G; h < (g + 1) * G; ++h) {
    const uint8_t* m = a.mask + ((((int64_t)b * a.n_layers + layer) * a.h_q + h) * a.n_qblk) * a.nmax + j;
    for (int i = 0; i < a.n_qblk; ++i)
      if (m[(int64_t)i * a.nmax]) return true;
  }
  return false;
}

__global__ void __launch_bounds__(kPtThreads) pt_count(const __grid_constant__ PtArgs a,
                                                       const __grid_constant__ SeqTable t) {
  const int row = blockIdx.x;
  const int per_seq = a.n_layers * a.h_kv;
  const int b = row / per_seq, lg = row % per_seq;
  const int layer = lg / a.h_kv, g = lg % a.h_kv;
  const int nkv = t.s[b].aux;
  int total = 0;
  for (int j0 = 0; j0 < nkv; j0 += kPtThreads) {
    const int j = j0 + threadIdx.x;
    const bool hit = j < nkv && union_hit(a, b, layer, g, j);
    total += __syncthreads_count(hit);
  }
  if (threadIdx.x == 0) a.counts[row] = total;
}

// Exclusive scan of the per-row counts into kv_indptr (one CTA).
__global__ void __launch_bounds__(1024) pt_scan(const __grid_constant__ PtArgs a) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int base = 0; base < a.rows; base += 1024) {
    const int i = base + threadIdx.x;
    const int v = i < a.rows ? a.counts[i] : 0;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int w = warp_tot[lane];
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_tot[lane] = w;
    }
    __syncthreads();
    const int excl = carry + (wid > 0 ? warp_tot[wid - 1] : 0) + x - v;
    if (i < a.rows) a.indptr[i] = excl;
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_tot[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) a.indptr[a.rows] = carry;
}

__global__ void __launch_bounds__(kPtThreads) pt_write(const __grid_constant__ PtArgs a,
                                                       const __grid_constant__ SeqTable t) {
  __shared__ int warp_cnt[kPtThreads / 32];
  const int row = blockIdx.x;
  const int per_seq = a.n_layers * a.h_kv;
  const int b = row / per_seq, lg = row % per_seq;
  const int layer = lg / a.h_kv, g = lg % a.h_kv;
  const int nkv = t.s[b].aux;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int written = a.indptr[row];
  for (int j0 = 0; j0 < nkv; j0 += kPtThreads) {
    const int j = j0 + threadIdx.x;
    const bool hit = j < nkv && union_hit(a, b, layer, g, j);
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) warp_cnt[wid] = __popc(bal);
    __syncthreads();
    int before = 0, chunk_total = 0;
    for (int w = 0; w < kPtThreads / 32; ++w) {
      if (w < wid) before += warp_cnt[w];
      chunk_total += warp_cnt[w];
    }
    if (hit) a.indices[written + before + __popc(bal & ((1u << lane) - 1u))] = j;
    written += chunk_total;
    __syncthreads();
  }
}

}  // namespace

kvsel_status launch_compact(const kvsel_desc& d, const SeqTable& t, const void* k, const void* v,
                            const int32_t* idx, int idx_layers, int n_sel, void* k_out, void* v_out,
                            DeviceError* err, cudaStream_t s) {
  CompactArgs a;
  a.k = static_cast<const uint4*>(k);
  a.v = static_cast<const uint4*>(v);
  a.idx = idx;
  a.k_out = static_cast<uint4*>(k_out);
  a.v_out = static_cast<uint4*>(v_out);
  a.err = err;
  a.n_layers = d.n_layers;
  a.h_kv = d.h_kv;
  a.vpr = d.head_dim / 8;
  a.n_sel = n_sel;
  a.P = d.page_size;
  a.idx_layers = idx_layers;
  a.rows_per_seq = (int64_t)d.n_layers * d.h_kv * n_sel * d.page_size;
  a.total_vecs = (int64_t)d.batch * a.rows_per_seq * a.vpr;
  const int64_t blocks = (a.total_vecs + 255) / 256;
  const unsigned grid = (unsigned)(blocks < 152 * 32 ? blocks : 152 * 32);
  TraceScope ts("kv_compact", s);
  compact_kernel<<<grid, 256, 0, s>>>(a, t);
  return launch_status();
}

kvsel_status launch_pagetable(const kvsel_desc& d, const SeqTable& t, const uint8_t* mask, int n_qblk,
                              int n_kvblk_max, int32_t* counts, int32_t* kv_indptr, int32_t* kv_indices,
                              cudaStream_t s) {
  PtArgs a;
  a.mask = mask;
  a.counts = counts;
  a.indptr = kv_indptr;
  a.indices = kv_indices;
  a.n_layers = d.n_layers;
  a.h_q = d.h_q;
  a.h_kv = d.h_kv;
  a.n_qblk = n_qblk;
  a.nmax = n_kvblk_max;
  a.rows = d.batch * d.n_layers * d.h_kv;
  kvsel_status st;
  {
    TraceScope ts("pagetable_count", s);
    pt_count<<<a.rows, kPtThreads, 0, s>>>(a, t);
    if ((st = launch_status()) != KVSEL_OK) return st;
  }
  {
    TraceScope ts("pagetable_scan", s);
    pt_scan<<<1, 1024, 0, s>>>(a);
    if ((st = launch_status()) != KVSEL_OK) return st;
  }
  TraceScope ts("pagetable_write", s);
  pt_write<<<a.rows, kPtThreads, 0, s>>>(a, t);
  return launch_status();
}

}  // namespace kvsel
