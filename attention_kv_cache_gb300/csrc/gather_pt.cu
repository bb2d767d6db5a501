// KV compaction (16-byte vector gather) and the block-union page table.
#include "internal.cuh"

namespace kvsel {
namespace {

// ------------------------------------------------------------------------ compaction
constexpr int kCompactThreads = 256;
constexpr int kCompactRows = 128;     // output rows per CTA

struct CompactArgs {
  const uint4* k;
  const uint4* v;
  const int32_t* idx;
  uint4* k_out;
  uint4* v_out;
  DeviceError* err;
  int32_t n_layers, h_kv, vpr, vpr_shift, n_sel, P, idx_layers, idx_heads, layer_lo, n_out;
  int32_t rows_per_unit;   // n_sel * P
  int32_t chunks;          // CTAs per (sequence, output layer, KV head) unit
};

// One CTA copies up to kCompactRows consecutive output rows of one unit.  A row of d bf16 is
// vpr 16-byte vectors; consecutive threads take consecutive vectors, so every row is read and
// written as whole 128-byte lines, and the unit's geometry is decoded once per CTA.
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const __grid_constant__ CompactArgs a,
                                                                  const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  const int unit = blockIdx.x / a.chunks;
  const int chunk = blockIdx.x % a.chunks;
  const int per_seq = a.n_out * a.h_kv;
  const int b = unit / per_seq;
  const int rem = unit % per_seq;
  const int lo = rem / a.h_kv, g = rem % a.h_kv;
  const int layer = a.layer_lo + lo;
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  if (si.n_keys == 0) return;            // a table whose device lengths failed the checks
  const int il = a.idx_layers == 1 ? 0 : lo;
  const int ih = a.idx_heads == 1 ? 0 : g;
  const int32_t* idx = a.idx + (((int64_t)b * a.idx_layers + il) * a.idx_heads + ih) * a.n_sel;
  const int64_t lim = a.P == 1 ? si.n_keys : ((int64_t)si.n_keys + a.P - 1) / a.P;
  const uint4* ksrc = a.k + si.k_off / 8 + ((int64_t)layer * a.h_kv + g) * si.n_keys * a.vpr;
  const uint4* vsrc = a.v + si.k_off / 8 + ((int64_t)layer * a.h_kv + g) * si.n_keys * a.vpr;
  const int64_t out0 = (int64_t)unit * a.rows_per_unit * a.vpr;
  const int r0 = chunk * kCompactRows;
  const int r1 = min(a.rows_per_unit, r0 + kCompactRows);
  const int n_vec = (r1 - r0) * a.vpr;
  constexpr int kUnroll = 4;
  for (int base = 0; base < n_vec; base += kCompactThreads * kUnroll) {
    uint4 kv[kUnroll], vv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int vi = base + u * kCompactThreads + threadIdx.x;
      kv[u] = make_uint4(0, 0, 0, 0);
      vv[u] = make_uint4(0, 0, 0, 0);
      if (vi < n_vec) {
        const int row = r0 + (vi >> a.vpr_shift);
        const int c = vi & (a.vpr - 1);
        const int sel = row / a.P;
        const int32_t id = idx[sel];
        const int64_t src_row = (int64_t)id * a.P + (row - sel * a.P);
        if (id < 0 || id >= lim) {
          if (c == 0) set_device_error(a.err, KVSEL_ERR_DEVICE, (uint32_t)((int64_t)unit * a.rows_per_unit + row));
        } else if (src_row < si.n_keys) {
          kv[u] = ksrc[src_row * a.vpr + c];
          vv[u] = vsrc[src_row * a.vpr + c];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int vi = base + u * kCompactThreads + threadIdx.x;
      if (vi < n_vec) {
        a.k_out[out0 + (int64_t)r0 * a.vpr + vi] = kv[u];
        a.v_out[out0 + (int64_t)r0 * a.vpr + vi] = vv[u];
      }
    }
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

// OR over the Q blocks and the query heads of group g for KV block j.  Every entry is read (no
// early exit), so the loads are independent and many are in flight at once instead of forming a
// chain of dependent loads for a block that no head selects.
__device__ __forceinline__ bool union_hit(const PtArgs& a, int b, int layer, int g, int j) {
  const int G = a.h_q / a.h_kv;
  const int n = G * a.n_qblk;                       // (head, Q block) rows of the group, consecutive
  const uint8_t* m = a.mask + ((((int64_t)b * a.n_layers + layer) * a.h_q + (int64_t)g * G) * a.n_qblk) * a.nmax + j;
  uint32_t acc = 0;
#pragma unroll 8
  for (int r = 0; r < n; ++r) acc |= m[(int64_t)r * a.nmax];
  return acc != 0;
}

__global__ void __launch_bounds__(kPtThreads) pt_count(const __grid_constant__ PtArgs a,
                                                       const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
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
                                                       const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
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
                            const int32_t* idx, int idx_layers, int idx_heads, int layer_lo, int n_layers_out,
                            int n_sel, void* k_out, void* v_out, DeviceError* err, cudaStream_t s) {
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
  a.vpr_shift = a.vpr == 16 ? 4 : 3;
  a.n_sel = n_sel;
  a.P = d.page_size;
  a.idx_layers = idx_layers;
  a.idx_heads = idx_heads;
  a.layer_lo = layer_lo;
  a.n_out = n_layers_out;
  a.rows_per_unit = n_sel * d.page_size;
  a.chunks = (a.rows_per_unit + kCompactRows - 1) / kCompactRows;
  const int64_t units = (int64_t)d.batch * n_layers_out * d.h_kv;
  if (units * a.chunks >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  TraceScope ts("kv_compact", s);
  compact_kernel<<<(unsigned)(units * a.chunks), kCompactThreads, 0, s>>>(a, t);
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
